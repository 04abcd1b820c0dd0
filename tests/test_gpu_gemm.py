"""GPU parity of the tcgen05 prefill product against the CPU oracle.

Tolerances.  The prefill kernel folds each group scale into the bf16 weight
operand ("unpacked to bf16 with the group scale folded in"): every weight is
exactly t * bf16(s_g), the fp16 scale rounded to nearest even.  The oracle is
given those rounded scales, and the outputs are held to the stated bounds:
fp32 within 1e-3 * sum_k |x w| + 1e-6, bf16 within
8e-3 * max(|y_ref|, ||x (.) w||_2).  Against the oracle on the exact fp16
scales, the difference is bounded by what the rounding of each scale explains,
sum_g |bf16(s_g) - s_g| |sum_{k in g} x_k t_k|, plus 2^-12 * A for the fp32
accumulation (A = sum_k |x w|).
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import (ACC_REL, assert_bf16_close, assert_fp32_close, assert_within, dev_bf16, dev_scales,
                         dev_trits, f16_to_bf16_f16, l2_xw, scale_rounding_bound)

pytestmark = pytest.mark.gpu

FP32_REL = 1e-3
BF16_REL = 8e-3


@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def run(tern, orc, p, out_dtype=torch.float32, s=None):
    """The product on the device-packed codes; returns (y, the oracle's codes)."""
    s = p.s if s is None else s
    ocodes, bad = orc.pack(p.t)
    assert bad == 0
    y = tern.gemm(dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(s), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    return y, ocodes


def check_fp32(orc, y, p, ocodes, s=None, what=""):
    """fp32 output: the stated bound against the oracle on the bf16-rounded
    scales, and the scale-rounding bound against the exact-scale oracle."""
    s = p.s if s is None else s
    y = y.cpu().numpy()
    y_b, a_b = orc.matmul(p.x, ocodes, f16_to_bf16_f16(s))
    assert_fp32_close(y, y_b, a_b, rel=FP32_REL, what=what)
    y_ref, a_ref = orc.matmul(p.x, ocodes, s)
    assert_within(y, y_ref, scale_rounding_bound(p.x, p.t, s) + ACC_REL * a_ref + 1e-6, what=what + " (exact s)")


def check_bf16(orc, y, p, ocodes, ms=None, ns=None, what=""):
    got = y.to(torch.float64).cpu().numpy()
    sb = f16_to_bf16_f16(p.s)
    if ms is None:
        y_b, _ = orc.matmul(p.x, ocodes, sb)
    else:
        got = got[ms, ns]
        y_b, _ = orc.matmul_sampled(p.x, ocodes, sb, ms, ns)
    assert_bf16_close(got, y_b, l2_xw(p.x, p.t, sb, ms, ns), rel=BF16_REL, what=what)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 200, 256), (200, 256, 1024), (256, 384, 512),
                                   (300, 130, 640), (512, 512, 2048), (17, 1000, 128)])
def test_gemm_fp32_matches_oracle(tern, orc, M, N, K):
    p = synth.problem(200 + M, M, N, K, tag=f"g{N}x{K}")
    y, ocodes = run(tern, orc, p)
    check_fp32(orc, y, p, ocodes, what=f"gemm M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(64, 256, 512), (512, 384, 1024)])
def test_gemm_bf16_matches_oracle(tern, orc, M, N, K):
    p = synth.problem(300 + M, M, N, K, tag="b")
    y, ocodes = run(tern, orc, p, torch.bfloat16)
    check_bf16(orc, y, p, ocodes, what="gemm bf16")


def test_gemm_exact_cases(tern):
    """Zero weights give exactly 0; one-hot x picks t * bf16(s) exactly."""
    M, N, K = 256, 128, 256
    t = np.zeros((N, K), dtype=np.int8)
    s = synth.scales(7, "s", (N, K // 128))
    x = synth.activations(7, "x", (M, K))
    y = tern.gemm(dev_bf16(x), tern.pack(dev_trits(t)), dev_scales(s))
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    t = synth.trits(8, "t", (N, K), synth.UNIFORM)
    x = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        x[m, m % K] = 0x3F80
    y = tern.gemm(dev_bf16(x), tern.pack(dev_trits(t)), dev_scales(s)).cpu().numpy()
    sb = torch.from_numpy(s.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    W = t.astype(np.float64) * np.repeat(sb, 128, axis=1)
    for m in range(M):
        assert np.array_equal(y[m].astype(np.float64), W[:, m % K]), m


def test_gemm_exact_cases_ragged_tokens(tern):
    """Three token tiles, the last one ragged (M = 700): zero weights give
    exactly 0, and one-hot x picks t * bf16(s) exactly at every (token, k)."""
    M, N, K = 700, 136, 256
    t = np.zeros((N, K), dtype=np.int8)
    s = synth.scales(9, "ws", (N, K // 128))
    x = synth.activations(9, "wx", (M, K))
    y = tern.gemm(dev_bf16(x), tern.pack(dev_trits(t)), dev_scales(s))
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    t = synth.trits(10, "wt", (N, K), synth.UNIFORM)
    x = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        x[m, (7 * m) % K] = 0x3F80
    y = tern.gemm(dev_bf16(x), tern.pack(dev_trits(t)), dev_scales(s)).cpu().numpy()
    assert tern.device_error() == 0
    sb = torch.from_numpy(s.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    W = t.astype(np.float64) * np.repeat(sb, 128, axis=1)
    for m in range(M):
        assert np.array_equal(y[m].astype(np.float64), W[:, (7 * m) % K]), m


@pytest.mark.parametrize("name,K,N", [(n, k, nn) for (n, k, nn) in synth.PREFILL_LAYER])
def test_gemm_prefill_layer_sampled(tern, orc, name, K, N):
    """One pp512 layer's projection at full size (M=512), sampled outputs."""
    M = synth.PREFILL_M
    p = synth.problem(5, M, N, K, tag=f"pp{name}")
    y, ocodes = run(tern, orc, p, torch.bfloat16)
    rs = np.random.default_rng(K + N)
    ms = rs.integers(0, M, 3000)
    ns = rs.integers(0, N, 3000)
    ms[:8], ns[:8] = M - 1, N - 1 - np.arange(8)
    check_bf16(orc, y, p, ocodes, ms, ns, what=f"pp512 {name}")
    # and with fp32 output, against the exact-scale oracle as well
    y32, _ = run(tern, orc, p)
    got = y32.cpu().numpy()[ms, ns]
    y_b, a_b = orc.matmul_sampled(p.x, ocodes, f16_to_bf16_f16(p.s), ms, ns)
    assert_fp32_close(got, y_b, a_b, rel=FP32_REL, what=f"pp512 {name} fp32")
    y_ref, a_ref = orc.matmul_sampled(p.x, ocodes, p.s, ms, ns)
    assert_within(got, y_ref, scale_rounding_bound(p.x, p.t, p.s, ms, ns) + ACC_REL * a_ref + 1e-6,
                  what=f"pp512 {name} fp32 (exact s)")


def test_gemm_back_to_back(tern, orc):
    """Several products back to back on one stream (programmatic dependent
    launch between them) stay correct."""
    ps = [synth.problem(400 + i, 100 + 50 * i, 256, 512, tag=f"bb{i}") for i in range(4)]
    ins = [(dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(p.s)) for p in ps]
    outs = [tern.gemm(*a) for a in ins for _ in range(2)]
    torch.cuda.synchronize()
    for i, p in enumerate(ps):
        ocodes, _ = orc.pack(p.t)
        for j in range(2):
            check_fp32(orc, outs[2 * i + j], p, ocodes, what=f"bb {i}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 8192), (300, 130, 4096), (512, 384, 17408), (40, 128, 2048)])
def test_gemm_stream_k_split_tiles(tern, orc, M, N, K):
    """Shapes with few tiles and deep K run on the stream-K schedule: each tile's
    K stages are spread over many CTAs (dozens for the smallest) whose fp32
    parts meet in the workspace sums; ragged M and N included."""
    p = synth.problem(600 + M, M, N, K, tag=f"sk{N}x{K}")
    y, ocodes = run(tern, orc, p)
    check_fp32(orc, y, p, ocodes, what=f"stream-K M={M} N={N} K={K}")
    # the counters and sums are back at zero: a second call on the same workspace agrees
    codes = tern.pack(dev_trits(p.t))
    ws = tern.workspace(tern.gemm_workspace_bytes(M, N, K))
    y1 = tern.gemm(dev_bf16(p.x), codes, dev_scales(p.s), ws=ws)
    y2 = tern.gemm(dev_bf16(p.x), codes, dev_scales(p.s), ws=ws)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_b, a_b = orc.matmul(p.x, ocodes, f16_to_bf16_f16(p.s))
    assert_fp32_close(y2.cpu().numpy(), y_b, a_b, rel=FP32_REL, what=f"stream-K second call M={M}")
    assert_fp32_close(y1.cpu().numpy(), y_b, a_b, rel=FP32_REL, what=f"stream-K first call M={M}")


@pytest.mark.parametrize("M,N,K", [(3, 64, 65536), (1100, 48, 1024), (8, 4096, 128)])
def test_gemm_extreme_shapes(tern, orc, M, N, K):
    """Very deep K on few tiles (stream-K over hundreds of stages), many
    token tiles on one row tile, and the shortest K."""
    p = synth.problem(1700 + M, M, N, K, tag=f"xe{N}x{K}")
    y, ocodes = run(tern, orc, p)
    rs = np.random.default_rng(M + N + K)
    ms, ns = rs.integers(0, M, 2000), rs.integers(0, N, 2000)
    ms[0], ns[0] = M - 1, N - 1
    got = y.cpu().numpy()[ms, ns]
    y_b, a_b = orc.matmul_sampled(p.x, ocodes, f16_to_bf16_f16(p.s), ms, ns)
    assert_fp32_close(got, y_b, a_b, rel=FP32_REL, what=f"extreme gemm M={M} N={N} K={K}")
    y_ref, a_ref = orc.matmul_sampled(p.x, ocodes, p.s, ms, ns)
    assert_within(got, y_ref, scale_rounding_bound(p.x, p.t, p.s, ms, ns) + ACC_REL * a_ref + 1e-6,
                  what=f"extreme gemm M={M} N={N} K={K} (exact s)")


def test_gemm_large_and_mixed_scales(tern, orc):
    """Scales up to a few hundred, mixed with small ones per group and row
    (the unpack's q * 2^-126 trick and the bf16 scale must hold over the whole
    fp16 scale range, not only the small scales of the synthetic workloads)."""
    M, N, K = 300, 256, 1024
    p = synth.problem(1800, M, N, K, tag="bigs")
    rs = np.random.default_rng(1800)
    big = rs.random((N, K // 128)) < 0.3
    s = np.where(big, rs.uniform(4.0, 300.0, (N, K // 128)), rs.uniform(0.01, 3.9, (N, K // 128))).astype(np.float16)
    s[:32, :] = np.float16(3.99)
    s[32:64, 0] = np.float16(60000.0)    # near the fp16 maximum
    y, ocodes = run(tern, orc, p, s=s)
    check_fp32(orc, y, p, ocodes, s=s, what="mixed scales")


@pytest.mark.parametrize("kind", ["zero", "negative", "subnormal", "mixed"])
def test_gemm_scale_edge_cases(tern, orc, kind):
    """Zero, negative and fp16-subnormal group scales (the synthetic workloads
    draw only positive normal ones)."""
    M, N, K = 130, 200, 512
    p = synth.problem(1900, M, N, K, tag=f"se{kind}")
    s = p.s.copy()
    rs = np.random.default_rng(1900)
    if kind == "zero":
        s[rs.random(s.shape) < 0.5] = np.float16(0.0)
    elif kind == "negative":
        s = (-s.astype(np.float32)).astype(np.float16)
    elif kind == "subnormal":
        s = (rs.integers(1, 1024, s.shape) * 2.0 ** -24).astype(np.float16)   # every fp16 subnormal magnitude
    else:
        sign = np.where(rs.random(s.shape) < 0.5, -1.0, 1.0)
        sub = rs.random(s.shape) < 0.3
        s = np.where(sub, sign * rs.integers(1, 1024, s.shape) * 2.0 ** -24, sign * s.astype(np.float64))
        s[rs.random(s.shape) < 0.1] = 0.0
        s = s.astype(np.float16)
    y, ocodes = run(tern, orc, p, s=s)
    check_fp32(orc, y, p, ocodes, s=s, what=f"scales {kind}")
