"""GPU parity of the 1-bit sibling format (binary g128, w = (2b - 1) s_g).

The device packer must agree with the oracle's packing bit for bit.  The
product is held to the decode tolerance |y - y_ref| <= 1e-3 * sum_k |x w| + 1e-6
against the oracle's double-precision product; a one-hot activation picks
+-s_g of a column, which the kernel computes exactly.  Shapes span full and
short K-slices (a slice is 8 groups of 128; K = 640, 1152 and 2176 leave
warps with no group), ragged N, and the token counts 1..16.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import (ACC_REL, assert_bf16_close, assert_fp32_close, assert_within, dev_bf16, dev_scales,
                         dev_trits, f16_to_bf16_f16, l2_xw, scale_rounding_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def words_host(words: torch.Tensor) -> np.ndarray:
    return words.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("N,K", [(37, 128), (1000, 2048), (3, 17408)])
def test_bin_pack_matches_oracle(tern, orc, N, K):
    t = synth.binary(50, f"p{N}", (N, K))
    t[0, 5] = 0                      # invalid: counted, stored as -1
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    words = tern.bin_pack(dev_trits(t), bad_count=bad)
    want, wbad = orc.bin_pack(t)
    assert int(bad.item()) == wbad == 1
    assert np.array_equal(words_host(words), want)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (1, 1000, 5120), (3, 777, 17408), (6, 129, 2176),
                                   (5, 200, 640), (16, 300, 1152), (2, 48, 128), (8, 129, 1024),
                                   (1, 16, 128)])
def test_bin_gemv_matches_oracle(tern, orc, M, N, K):
    p = synth.binary_problem(60 + M, M, N, K, tag=f"g{N}x{K}")
    words = tern.bin_pack(dev_trits(p.t))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.bin_gemv(dev_bf16(p.x), words, dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.bin_matmul(p.x, orc.bin_pack(p.t)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"binary M={M} N={N} K={K}")


def test_bin_gemv_one_hot_exact(tern):
    """x = e_k picks (2b[n][k] - 1) s[n][k / 128] exactly, at every slot position."""
    N, K = 64, 256
    t = synth.binary(70, "oh", (N, K))
    s = synth.scales(70, "s", (N, K // 128))
    words = tern.bin_pack(dev_trits(t))
    W = t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
    ks = [0, 9, 10, 11, 12, 15, 16, 27, 28, 31, 32, 100, 127, 128, 200, 255]
    for i in range(0, len(ks), 8):
        chunk = ks[i:i + 8]
        x = np.zeros((len(chunk), K), dtype=np.uint16)
        for j, k in enumerate(chunk):
            x[j, k] = 0x3F80
        y = tern.bin_gemv(dev_bf16(x), words, dev_scales(s)).cpu().numpy()
        for j, k in enumerate(chunk):
            assert np.array_equal(y[j].astype(np.float64), W[:, k]), k


@pytest.mark.parametrize("M,K,N", [(1, 5120, 17408), (1, 17408, 5120), (5, 5120, 6144), (16, 5120, 17408)])
def test_bin_gemv_full_size_sampled(tern, orc, M, K, N):
    p = synth.binary_problem(80 + M, M, N, K, tag=f"f{K}")
    words = tern.bin_pack(dev_trits(p.t))
    y = tern.bin_gemv(dev_bf16(p.x), words, dev_scales(p.s))
    torch.cuda.synchronize()
    rs = np.random.default_rng(K + N + M)
    ms, ns = rs.integers(0, M, 3000), rs.integers(0, N, 3000)
    ms[:4], ns[:4] = M - 1, [0, N - 1, N - 2, N // 2]
    y_ref, a_ref = orc.bin_matmul_sampled(p.x, orc.bin_pack(p.t)[0], p.s, ms, ns)
    assert_fp32_close(y.cpu().numpy()[ms, ns], y_ref, a_ref, what=f"binary full M={M} {K}->{N}")


def test_bin_and_ternary_agree_on_pm1(tern, orc):
    """The same +-1 weights through both layouts and both kernel variants."""
    M, N, K = 3, 500, 5120
    p = synth.binary_problem(90, M, N, K, tag="both")
    x, s = dev_bf16(p.x), dev_scales(p.s)
    yb = tern.bin_gemv(x, tern.bin_pack(dev_trits(p.t)), s)
    yt = tern.gemv(x, tern.pack(dev_trits(p.t)), s)
    torch.cuda.synchronize()
    y_ref, a_ref = orc.bin_matmul(p.x, orc.bin_pack(p.t)[0], p.s)
    assert_fp32_close(yb.cpu().numpy(), y_ref, a_ref, what="binary kernel")
    assert_fp32_close(yt.cpu().numpy(), y_ref, a_ref, what="ternary kernel on +-1")


# --------------------------------------------------------------------------
# the prefill product on the 1-bit layout (tcgen05).  Each weight is exactly
# (2b - 1) * bf16(s_g), so the oracle is given the bf16-rounded scales: fp32
# output within 1e-3 * sum_k |x w| + 1e-6, bf16 output within
# 8e-3 * max(|y_ref|, ||x (.) w||_2); against the exact-scale oracle the
# difference stays within sum_g |bf16(s_g) - s_g| |sum_{k in g} x_k w_k / s_g|
# plus 2^-12 * A for the accumulation.
# --------------------------------------------------------------------------

FP32_REL = 1e-3
BF16_REL = 8e-3


def bin_check_fp32(orc, y, p, words, ms=None, ns=None, what=""):
    got = y.cpu().numpy()
    sb = f16_to_bf16_f16(p.s)
    if ms is None:
        y_b, a_b = orc.bin_matmul(p.x, words, sb)
        y_ref, a_ref = orc.bin_matmul(p.x, words, p.s)
    else:
        got = got[ms, ns]
        y_b, a_b = orc.bin_matmul_sampled(p.x, words, sb, ms, ns)
        y_ref, a_ref = orc.bin_matmul_sampled(p.x, words, p.s, ms, ns)
    assert_fp32_close(got, y_b, a_b, rel=FP32_REL, what=what)
    assert_within(got, y_ref, scale_rounding_bound(p.x, p.t, p.s, ms, ns) + ACC_REL * a_ref + 1e-6,
                  what=what + " (exact s)")


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 200, 256), (200, 256, 1024), (300, 130, 640),
                                   (512, 512, 2048), (17, 1000, 128), (256, 256, 8192), (40, 128, 2048)])
def test_bin_gemm_matches_oracle(tern, orc, M, N, K):
    p = synth.binary_problem(100 + M, M, N, K, tag=f"m{N}x{K}")
    y = tern.bin_gemm(dev_bf16(p.x), tern.bin_pack(dev_trits(p.t)), dev_scales(p.s))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    words, bad = orc.bin_pack(p.t)
    assert bad == 0
    bin_check_fp32(orc, y, p, words, what=f"binary gemm M={M} N={N} K={K}")


def test_bin_gemm_bf16_and_one_hot(tern, orc):
    M, N, K = 256, 384, 512
    p = synth.binary_problem(110, M, N, K, tag="b16")
    words = tern.bin_pack(dev_trits(p.t))
    y = tern.bin_gemm(dev_bf16(p.x), words, dev_scales(p.s), out_dtype=torch.bfloat16)
    owords, _ = orc.bin_pack(p.t)
    sb = f16_to_bf16_f16(p.s)
    y_b, _ = orc.bin_matmul(p.x, owords, sb)
    assert_bf16_close(y.to(torch.float64).cpu().numpy(), y_b, l2_xw(p.x, p.t, sb), rel=BF16_REL,
                      what="binary gemm bf16")
    # one-hot rows of x pick (2b - 1) * bf16(s) exactly
    x = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        x[m, (37 * m) % K] = 0x3F80
    y = tern.bin_gemm(dev_bf16(x), words, dev_scales(p.s)).cpu().numpy()
    W = p.t.astype(np.float64) * np.repeat(sb.astype(np.float64), 128, axis=1)
    for m in range(M):
        assert np.array_equal(y[m].astype(np.float64), W[:, (37 * m) % K]), m


@pytest.mark.parametrize("name,K,N", [(n, k, nn) for (n, k, nn) in synth.PREFILL_LAYER])
def test_bin_gemm_prefill_layer_sampled(tern, orc, name, K, N):
    M = synth.PREFILL_M
    p = synth.binary_problem(120, M, N, K, tag=f"bp{name}")
    words = tern.bin_pack(dev_trits(p.t))
    y = tern.bin_gemm(dev_bf16(p.x), words, dev_scales(p.s), out_dtype=torch.bfloat16)
    y32 = tern.bin_gemm(dev_bf16(p.x), words, dev_scales(p.s))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    rs = np.random.default_rng(K + N + 1)
    ms, ns = rs.integers(0, M, 3000), rs.integers(0, N, 3000)
    ms[:4], ns[:4] = M - 1, [0, N - 1, N - 2, N // 2]
    owords, _ = orc.bin_pack(p.t)
    sb = f16_to_bf16_f16(p.s)
    y_b, _ = orc.bin_matmul_sampled(p.x, owords, sb, ms, ns)
    assert_bf16_close(y.to(torch.float64).cpu().numpy()[ms, ns], y_b, l2_xw(p.x, p.t, sb, ms, ns), rel=BF16_REL,
                      what=f"binary pp512 {name}")
    bin_check_fp32(orc, y32, p, owords, ms, ns, what=f"binary pp512 {name} fp32")
