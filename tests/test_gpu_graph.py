"""The products replayed from CUDA graphs, the way the benchmark runs them.

A sequence of calls (programmatic dependent launch between consecutive
kernels, one workspace shared by all of them) is captured once and replayed;
the outputs are filled with NaN before the checked replay, so every element
must be written by that replay.  Each product is compared with the oracle on
sampled outputs at full size, within the tolerance of its kind:
|y - y_ref| <= 1e-3 * sum_k |x w| + 1e-6 for the decode products, and, for
the prefill products (bf16 out, weights t * bf16(s_g)), the bf16-output bound
8e-3 * max(|y_ref|, ||x (.) w||_2) against the oracle on the bf16-rounded
scales.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import assert_bf16_close, assert_fp32_close, dev_bf16, dev_scales, dev_trits, f16_to_bf16_f16, l2_xw

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def capture(fn):
    """Warm up on a side stream, then capture fn into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def sample(M, N, seed, n=1500):
    rs = np.random.default_rng(seed)
    ms, ns = rs.integers(0, M, n), rs.integers(0, N, n)
    ms[:4], ns[:4] = M - 1, [0, N - 1, N - 2, N // 2]
    return ms, ns


def replay_and_check(tern, orc, g, probs, ys, prefill=False, what=""):
    for _ in range(2):
        g.replay()
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    for i, ((p, codes), y) in enumerate(zip(probs, ys)):
        ms, ns = sample(p.M, p.N, 77 + i)
        got = y.to(torch.float64).cpu().numpy()[ms, ns]
        ocodes = orc.pack(p.t)[0]
        if prefill:
            sb = f16_to_bf16_f16(p.s)
            y_b, _ = orc.matmul_sampled(p.x, ocodes, sb, ms, ns)
            assert_bf16_close(got, y_b, l2_xw(p.x, p.t, sb, ms, ns), what=f"{what} product {i} ({p.M}x{p.N}x{p.K})")
        else:
            y_ref, a_ref = orc.matmul_sampled(p.x, ocodes, p.s, ms, ns)
            assert_fp32_close(got, y_ref, a_ref, what=f"{what} product {i} ({p.M}x{p.N}x{p.K})")


def test_verify_step_graph(tern, orc):
    """Speculative verify: k + 1 = 5 tokens through two layers' qkv, gate,
    up and down products, one graph."""
    M = synth.VERIFY_STEP_M
    shapes = [(5120, 6144), (5120, 17408), (5120, 17408), (17408, 5120)] * 2
    probs = []
    for i, (K, N) in enumerate(shapes):
        p = synth.problem(1100 + i, M, N, K, tag=f"vs{i}")
        probs.append((p, tern.pack(dev_trits(p.t))))
    xs = [dev_bf16(p.x) for p, _ in probs]
    ss = [dev_scales(p.s) for p, _ in probs]
    ys = [torch.empty((M, p.N), dtype=torch.float32, device="cuda") for p, _ in probs]
    ws = tern.workspace(max(tern.gemv_workspace_bytes(M, N, K) for K, N in shapes))

    def run():
        for i, (p, codes) in enumerate(probs):
            tern.gemv(xs[i], codes, ss[i], y=ys[i], ws=ws)

    replay_and_check(tern, orc, capture(run), probs, ys, what="verify step")


def test_decode_sweep_graph(tern, orc):
    """Single-token decode: two layers' gate, up and down products, one graph."""
    shapes = [(5120, 17408), (5120, 17408), (17408, 5120)] * 2
    probs = []
    for i, (K, N) in enumerate(shapes):
        p = synth.problem(1200 + i, 1, N, K, tag=f"ds{i}")
        probs.append((p, tern.pack(dev_trits(p.t))))
    xs = [dev_bf16(p.x) for p, _ in probs]
    ss = [dev_scales(p.s) for p, _ in probs]
    ys = [torch.empty((1, p.N), dtype=torch.float32, device="cuda") for p, _ in probs]
    ws = tern.workspace(max(tern.gemv_workspace_bytes(1, N, K) for K, N in shapes))

    def run():
        for i, (p, codes) in enumerate(probs):
            tern.gemv(xs[i], codes, ss[i], y=ys[i], ws=ws)

    replay_and_check(tern, orc, capture(run), probs, ys, what="decode")


def test_prefill_layer_graph(tern, orc):
    """pp512: one layer's gate, up, qkv and down products (bf16 out), one graph;
    the down product runs the stream-K schedule."""
    M = synth.PREFILL_M
    probs = []
    for i, (name, K, N) in enumerate(synth.PREFILL_LAYER):
        p = synth.problem(1300 + i, M, N, K, tag=f"pl{name}")
        probs.append((p, tern.pack(dev_trits(p.t))))
    xs = [dev_bf16(p.x) for p, _ in probs]
    ss = [dev_scales(p.s) for p, _ in probs]
    ys = [torch.empty((M, p.N), dtype=torch.bfloat16, device="cuda") for p, _ in probs]
    ws = tern.workspace(max(tern.gemm_workspace_bytes(M, N, K) for _, K, N in synth.PREFILL_LAYER))

    def run():
        for i, (p, codes) in enumerate(probs):
            tern.gemm(xs[i], codes, ss[i], y=ys[i], ws=ws)

    replay_and_check(tern, orc, capture(run), probs, ys, prefill=True, what="prefill")


@pytest.mark.parametrize("M", [1, 16])
def test_fused_rotation_graph(tern, orc, M):
    """The rotated workload, two fused calls with different activations and
    weights, one graph."""
    K, N = synth.ROTATED["K"], synth.ROTATED["N"]
    ps = [synth.problem(1400 + M + c, M, N, K, with_signs=True, tag=f"fr{c}") for c in range(2)]
    codes = [tern.pack(dev_trits(p.t)) for p in ps]
    xs = [dev_bf16(p.x) for p in ps]
    ss = [dev_scales(p.s) for p in ps]
    sg = [torch.from_numpy(p.signs).cuda() for p in ps]
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in ps]
    ws = tern.workspace(tern.gemv_workspace_bytes(M, N, K))

    def run():
        for c in range(2):
            tern.fwht_gemm(xs[c], sg[c], codes[c], ss[c], y=ys[c], ws=ws)

    g = capture(run)
    for _ in range(2):
        g.replay()
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    rs = np.random.default_rng(M)
    rows = np.unique(rs.integers(0, N, 384))
    for c, p in enumerate(ps):
        y_ref, a_ref = orc.rotate_matmul(p.x, p.signs, orc.pack(p.t)[0][rows], p.s[rows])
        assert_fp32_close(ys[c].cpu().numpy()[:, rows], y_ref, a_ref, what=f"rotated graph M={M} call {c}")


def test_binary_decode_graph(tern, orc):
    """The 1-bit product: two layers' gate, up and down at M = 1, one graph."""
    shapes = [(5120, 17408), (5120, 17408), (17408, 5120)] * 2
    probs = [synth.binary_problem(1500 + i, 1, N, K, tag=f"bg{i}") for i, (K, N) in enumerate(shapes)]
    words = [tern.bin_pack(dev_trits(p.t)) for p in probs]
    xs = [dev_bf16(p.x) for p in probs]
    ss = [dev_scales(p.s) for p in probs]
    ys = [torch.empty((1, p.N), dtype=torch.float32, device="cuda") for p in probs]
    ws = tern.workspace(max(tern.gemv_workspace_bytes(1, N, K) for K, N in shapes))

    def run():
        for i in range(len(probs)):
            tern.bin_gemv(xs[i], words[i], ss[i], y=ys[i], ws=ws)

    g = capture(run)
    for _ in range(2):
        g.replay()
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    for i, p in enumerate(probs):
        ms, ns = sample(1, p.N, 88 + i)
        y_ref, a_ref = orc.bin_matmul_sampled(p.x, orc.bin_pack(p.t)[0], p.s, ms, ns)
        assert_fp32_close(ys[i].cpu().numpy()[ms, ns], y_ref, a_ref, what=f"binary graph product {i}")


def test_pair_decode_graph(tern, orc):
    """The decode step as the benchmark runs it: per layer, gate and up in one
    pair call on their shared activation, then down; two layers, one graph."""
    probs, xs = [], []
    for l in range(2):
        pg = synth.problem(1600 + 3 * l, 1, 17408, 5120, tag=f"pg{l}")
        pu = synth.problem(1601 + 3 * l, 1, 17408, 5120, tag=f"pu{l}")
        pd = synth.problem(1602 + 3 * l, 1, 5120, 17408, tag=f"pd{l}")
        for p in (pg, pu, pd):
            probs.append((p, tern.pack(dev_trits(p.t))))
        xs += [dev_bf16(pg.x), dev_bf16(pd.x)]
    ss = [dev_scales(p.s) for p, _ in probs]
    ys = [torch.empty((1, p.N), dtype=torch.float32, device="cuda") for p, _ in probs]
    ws = tern.workspace(max(int(tern.lib().tern_gemv_pair_workspace_bytes(1, 17408, 17408, 5120)),
                            tern.gemv_workspace_bytes(1, 5120, 17408)))

    def run():
        for l in range(2):
            g, u, d = 3 * l, 3 * l + 1, 3 * l + 2
            tern.gemv_pair(xs[2 * l], probs[g][1], ss[g], probs[u][1], ss[u], y_a=ys[g], y_b=ys[u], ws=ws)
            tern.gemv(xs[2 * l + 1], probs[d][1], ss[d], y=ys[d], ws=ws)

    g = capture(run)
    for _ in range(2):
        g.replay()
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    for i, (p, codes) in enumerate(probs):
        x_bits = probs[i - 1][0].x if i % 3 == 1 else p.x          # up reads gate's activation
        ms, ns = sample(1, p.N, 99 + i)
        y_ref, a_ref = orc.matmul_sampled(x_bits, orc.pack(p.t)[0], p.s, ms, ns)
        assert_fp32_close(ys[i].cpu().numpy()[ms, ns], y_ref, a_ref, what=f"pair graph product {i}")
