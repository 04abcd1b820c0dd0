"""The native base-3 format on the GPU against the oracle.

tern_f3_pack is compared byte for byte with the oracle's packer (invalid
entries counted the same way), and tern_f3_gemv element by element with the
oracle's product on the oracle's bytes, within |y - y_ref| <= 1e-3 * sum_k
|x w| + 1e-6: ragged N, K not a multiple of the kernel's 1024-wide chunk,
every M the product takes, and the decode shape 5120 -> 17408 in full.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import assert_fp32_close, dev_bf16, dev_scales, dev_trits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tern():
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


@pytest.mark.parametrize("N,K", [(1, 128), (37, 640), (300, 5120), (5, 17408)])
def test_f3_pack_matches_oracle(tern, orc, N, K):
    t = synth.trits(80, f"f3p{N}x{K}", (N, K))
    t[0, 0] = 3          # invalid: packed as -1 and counted
    if K > 200:
        t[-1, 133] = -2
    want, bad = orc.f3_pack(t)
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = tern.f3_pack(dev_trits(t), bad_count=cnt)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)
    assert int(cnt.item()) == bad == (2 if K > 200 else 1)


@pytest.mark.parametrize("M,N,K", [(1, 300, 640), (1, 1000, 5120), (2, 129, 2048), (5, 77, 1152),
                                   (8, 50, 3072), (16, 33, 1024), (3, 17, 17408)])
def test_f3_gemv_matches_oracle(tern, orc, M, N, K):
    p = synth.problem(81 + M, M, N, K, tag=f"f3g{N}x{K}")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.f3_gemv(dev_bf16(p.x), torch.from_numpy(packed).cuda(), dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"f3 M={M} N={N} K={K}")


def test_f3_gemv_decode_shape_full(tern, orc):
    """The gate shape of the decode sweep, every output, on the GPU packer's
    bytes (checked equal to the oracle's first)."""
    M, N, K = 1, 17408, 5120
    p = synth.problem(90, M, N, K, tag="f3full")
    packed, _ = orc.f3_pack(p.t)
    dp = tern.f3_pack(dev_trits(p.t))
    torch.cuda.synchronize()
    assert np.array_equal(dp.cpu().numpy(), packed)
    y = tern.f3_gemv(dev_bf16(p.x), dp, dev_scales(p.s))
    torch.cuda.synchronize()
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what="f3 decode shape")


def test_f3_zero_rows_and_scale_edges(tern, orc):
    """Rows of zero weights give exactly 0; zero, negative and subnormal
    scales are products like any other."""
    M, N, K = 2, 64, 1024
    p = synth.problem(91, M, N, K, tag="f3edge")
    t = p.t.copy()
    t[5] = 0
    t[40] = 0
    s = p.s.copy()
    s[7, :] = np.float16(0.0)
    s[8, :] = -s[8, :]
    s[9, 3] = np.float16(2.0 ** -20)      # subnormal fp16
    packed, _ = orc.f3_pack(t)
    y = tern.f3_gemv(dev_bf16(p.x), torch.from_numpy(packed).cuda(), dev_scales(s))
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    assert (yh[:, 5] == 0).all() and (yh[:, 40] == 0).all() and (yh[:, 7] == 0).all()
    y_ref, a_ref = orc.f3_matmul(p.x, packed, s)
    assert_fp32_close(yh, y_ref, a_ref, what="f3 edges")
