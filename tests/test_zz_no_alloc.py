"""The decode product for callers that cannot allocate device memory.

tern_gemv_noalloc takes no workspace: its scratch (one flag word per 16-row
tile, ordering the clearing of y before the K-chunks' additions) is a fixed
array inside the library.  It exists for code that must not call cudaMalloc --
for instance code running inside an allocator's own callback, or under a
runtime that owns all device memory -- and so cannot provide the workspace
tern_gemv asks for.

These checks call it through the C ABI and compare it with the oracle's
product on the same inputs, twice in a row (the second call starts from
whatever the first left in the shared array), within the decode tolerance
|y - y_ref| <= 1e-3 * sum_k |x w| + 1e-6.  The largest accepted shape (its
flags fill the array exactly) must be accepted and correct, and the second
call must leave the device's free memory unchanged.  This file sorts last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests._util import assert_fp32_close, dev_bf16, dev_codes, dev_scales

TERN_ERR_NULL, TERN_ERR_SHAPE, TERN_ERR_ALIGN, TERN_ERR_WORKSPACE = 1, 2, 3, 4
NOALLOC_BYTES = 256 << 10


@pytest.fixture(scope="module")
def tern():
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def _call_noalloc(tern, x, codes, s, y):
    M, K = x.shape
    N = codes.shape[0]
    st = tern.lib().tern_gemv_noalloc(x.data_ptr(), codes.data_ptr(), s.data_ptr(), y.data_ptr(), M, N, K,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"tern_gemv_noalloc status {st}"


def test_noalloc_validates_before_any_device_use(tern):
    """Bad shapes, NULL and misaligned pointers are refused up front."""
    P = 4096   # a fake aligned address: the checks come before any device use
    lib = tern.lib()
    assert lib.tern_gemv_noalloc(P, P, P, P, 17, 64, 128, None) == TERN_ERR_SHAPE
    assert lib.tern_gemv_noalloc(P, P, P, P, 1, 64, 100, None) == TERN_ERR_SHAPE
    assert lib.tern_gemv_noalloc(None, P, P, P, 1, 64, 128, None) == TERN_ERR_NULL
    assert lib.tern_gemv_noalloc(P, P + 4, P, P, 1, 64, 128, None) == TERN_ERR_ALIGN


def test_noalloc_rejects_oversized_shapes_without_launching(tern):
    """A shape whose scratch exceeds the fixed array is refused up front."""
    M, N, K = 1, 1100000, 2048
    assert tern.gemv_workspace_bytes(M, N, K) > NOALLOC_BYTES
    P = 4096   # a fake aligned address: the size check comes before any device use
    assert tern.lib().tern_gemv_noalloc(P, P, P, P, M, N, K, None) == TERN_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(1, 17408, 5120), (1, 5120, 17408), (3, 1000, 5120), (16, 600, 2048),
                                   (5, 200, 512), (2, 300, 1152)])
def test_noalloc_matches_oracle_twice(tern, orc, M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = synth.problem(500 + M, M, N, K, tag=f"na{N}x{K}")
    ocodes, bad = orc.pack(p.t)
    assert bad == 0
    x, codes, s = dev_bf16(p.x), dev_codes(ocodes), dev_scales(p.s)
    y_ref, a_ref = orc.matmul(p.x, ocodes, p.s)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        _call_noalloc(tern, x, codes, s, y)
        torch.cuda.synchronize()
        assert tern.device_error() == 0
        assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"noalloc call {call} M={M} N={N} K={K}")


@pytest.mark.gpu
def test_noalloc_largest_shape_allocates_nothing(tern, orc):
    """N = 1,048,576 rows: one flag word per 16-row tile fills the array
    exactly.  The call is accepted, matches the oracle on sampled outputs
    (the last rows included) twice in a row, and the second call leaves the
    device's free memory as it was."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 1, 1 << 20, 2048
    assert (N // 16) * 4 == NOALLOC_BYTES
    # 4096 distinct rows of trits repeated down the matrix, with a distinct
    # scale per row and group, so every output differs
    base = synth.problem(510, M, 4096, K, tag="nabig")
    ocodes_small, bad = orc.pack(base.t)
    assert bad == 0
    ocodes = np.tile(ocodes_small, (N // 4096, 1))
    s = synth.scales(511, "nabig_s", (N, K // 128))
    x, codes, sd = dev_bf16(base.x), dev_codes(ocodes), dev_scales(s)
    rs = np.random.default_rng(512)
    ns = np.concatenate([rs.integers(0, N, 3000), np.arange(N - 40, N), np.arange(0, 40)]).astype(np.int32)
    ms = np.zeros_like(ns)
    y_ref, a_ref = orc.matmul_sampled(base.x, ocodes, s, ms, ns)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    _call_noalloc(tern, x, codes, sd, y)          # the first call loads and plans
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    assert_fp32_close(y.cpu().numpy()[ms, ns], y_ref, a_ref, what="noalloc largest, call 0")
    y.fill_(float("nan"))
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    _call_noalloc(tern, x, codes, sd, y)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"the call changed free device memory by {free_before - free_after} bytes"
    assert tern.device_error() == 0
    assert_fp32_close(y.cpu().numpy()[ms, ns], y_ref, a_ref, what="noalloc largest, call 1")
    # one row more is refused, without launching
    P = 4096
    assert tern.lib().tern_gemv_noalloc(P, P, P, P, M, N + 16, K, None) == TERN_ERR_WORKSPACE
