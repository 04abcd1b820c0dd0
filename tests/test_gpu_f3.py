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


@pytest.mark.parametrize("N,K", [(1, 512), (37, 512), (300, 1536), (1000, 3072), (129, 17408), (5, 65536)])
def test_f3_gemv_one_token_tensor_pipe(tern, orc, N, K):
    """One token with K a multiple of 512 runs the tensor-pipe product (the
    five codes of a byte from a table, assembled into 2-bit words): ragged
    N, one K-slice and many, every output against the oracle."""
    p = synth.problem(95, 1, N, K, tag=f"f3m{N}x{K}")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.f3_gemv(dev_bf16(p.x), torch.from_numpy(packed).cuda(), dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"f3 one token N={N} K={K}")


def test_f3_one_token_exact_cases(tern, orc):
    """Exact answers on the tensor-pipe product: zero trits give exactly 0;
    trits +-1 with x = 2 at one position give 2 s exactly, at every position
    of a 512-wide row (every byte, digit and lane of the assembly, the
    three-trit last byte included)."""
    N, K = 16, 512
    s = synth.scales(96, "f3e", (N, K // 128), synth.SCALE_UNIFORM)
    z, _ = orc.f3_pack(np.zeros((N, 1536), dtype=np.int8))
    y = tern.f3_gemv(dev_bf16(synth.activations(96, "f3x", (1, 1536))), torch.from_numpy(z).cuda(),
                     dev_scales(synth.scales(96, "f3z", (N, 12))))
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    t = np.ones((N, K), dtype=np.int8)
    t[1::2] = -1
    t[:, 120:128] *= -1
    packed, _ = orc.f3_pack(t)
    dp = torch.from_numpy(packed).cuda()
    ds = dev_scales(s)
    for k in range(K):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x4000                                    # bf16 2.0
        y = tern.f3_gemv(dev_bf16(x), dp, ds).cpu().numpy()
        want = 2.0 * t[:, k].astype(np.float64) * s[:, k // 128].astype(np.float64)
        assert np.array_equal(y[0].astype(np.float64), want), k


def test_f3_one_token_bytes_outside_the_pack(tern, orc):
    """Bytes above 242 are not a pack's (their weights are undefined), but a
    call on them stays within its buffers and reports no device error."""
    N, K = 40, 1024
    rs = np.random.default_rng(97)
    packed = rs.integers(0, 256, size=(N, 26 * (K // 128)), dtype=np.uint8)
    y = tern.f3_gemv(dev_bf16(synth.activations(97, "f3o", (1, K))), torch.from_numpy(packed).cuda(),
                     dev_scales(synth.scales(97, "f3os", (N, K // 128))))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("M", [2, 5, 9, 16])
@pytest.mark.parametrize("N,K", [(37, 512), (300, 1536), (129, 17408)])
def test_f3_gemv_tokens_tensor_pipe(tern, orc, M, N, K):
    """Several tokens with K a multiple of 512 (one token tile up to eight
    tokens, two up to sixteen): every output against the oracle."""
    p = synth.problem(98 + M, M, N, K, tag=f"f3t{N}x{K}")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.f3_gemv(dev_bf16(p.x), torch.from_numpy(packed).cuda(), dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"f3 M={M} N={N} K={K}")


def test_f3_tokens_exact_cases(tern, orc):
    """Sixteen tokens, x = 2 at a different position for each: 2 s exactly,
    over every position of a 512-wide row."""
    N, K, M = 16, 512, 16
    s = synth.scales(99, "f3te", (N, K // 128), synth.SCALE_UNIFORM)
    t = np.ones((N, K), dtype=np.int8)
    t[1::2] = -1
    t[:, 60:70] *= -1
    packed, _ = orc.f3_pack(t)
    dp = torch.from_numpy(packed).cuda()
    ds = dev_scales(s)
    for k0 in range(0, K, M):
        x = np.zeros((M, K), dtype=np.uint16)
        for i in range(M):
            x[i, k0 + i] = 0x4000                           # bf16 2.0
        y = tern.f3_gemv(dev_bf16(x), dp, ds).cpu().numpy()
        for i in range(M):
            k = k0 + i
            want = 2.0 * t[:, k].astype(np.float64) * s[:, k // 128].astype(np.float64)
            assert np.array_equal(y[i].astype(np.float64), want), k
