"""GPU parity: device packer, decode/small-batch product, rotation and the
rotation-fused product against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from tests._util import (assert_fp32_close, bf16_to_f64, dev_bf16, dev_codes, dev_scales, dev_trits,
                         host_codes)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def run_gemv(tern, p, codes_dev=None):
    x = dev_bf16(p.x)
    if codes_dev is None:
        codes_dev = tern.pack(dev_trits(p.t))
    s = dev_scales(p.s)
    y = tern.gemv(x, codes_dev, s)
    torch.cuda.synchronize()
    return y.cpu().numpy(), codes_dev


# ---------------------------------------------------------------------------
# packing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (256, 512), (1000, 1024)])
def test_pack_bit_exact(tern, orc, N, K):
    t = synth.trits(N, "t", (N, K), synth.UNIFORM)
    codes = tern.pack(dev_trits(t))
    torch.cuda.synchronize()
    want, bad = orc.pack(t)
    assert bad == 0
    assert np.array_equal(host_codes(codes), want)


def test_pack_counts_invalid(tern, orc):
    t = synth.trits(1, "t", (64, 256), synth.UNIFORM)
    t[0, 0] = 2
    t[10, 100] = -3
    t[63, 255] = 77
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes = tern.pack(dev_trits(t), bad_count=bad)
    torch.cuda.synchronize()
    want, nbad = orc.pack(t)
    assert int(bad.item()) == nbad == 3
    assert np.array_equal(host_codes(codes), want)


def test_pack_full_decode_shape(tern, orc):
    t = synth.trits(2, "t", (17408, 5120))
    codes = tern.pack(dev_trits(t))
    torch.cuda.synchronize()
    want, _ = orc.pack(t)
    assert np.array_equal(host_codes(codes), want)


# ---------------------------------------------------------------------------
# decode / small-batch product
# ---------------------------------------------------------------------------

def test_gemv_tiny_workload(tern, orc):
    """M=1, K=512, N=256; uniform trits, U[0.005, 0.05] scales; seed 0."""
    c = synth.TINY
    p = synth.problem(c["seed"], c["M"], c["N"], c["K"], trit_dist=c["trit_dist"],
                      scale_dist=c["scale_dist"])
    y, codes = run_gemv(tern, p)
    want_codes, _ = orc.pack(p.t)
    assert np.array_equal(host_codes(codes), want_codes)
    y_ref, a_ref = orc.matmul(p.x, want_codes, p.s)
    assert_fp32_close(y, y_ref, a_ref, what="tiny")


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("N,K", [(200, 1152), (16, 128), (37, 256), (512, 4096)])
def test_gemv_ragged_shapes(tern, orc, M, N, K):
    p = synth.problem(100 + M, M, N, K, tag=f"{N}x{K}")
    y, codes = run_gemv(tern, p)
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y, y_ref, a_ref, what=f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [2, 3, 5, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(37, 512), (300, 1536), (77, 2304), (1000, 3072), (129, 17408)])
def test_gemv_tile_major_shapes(tern, orc, M, N, K):
    """Five tokens and more, or two and more on at most 8192 rows, with K a
    multiple of 256 (the tile-major loop):
    ragged N (an odd tile count leaves a pair's second tile past the matrix),
    one K-slice and several, every output against the oracle."""
    p = synth.problem(120 + M, M, N, K, tag=f"tm{N}x{K}")
    y, _ = run_gemv(tern, p)
    assert tern.device_error() == 0
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y, y_ref, a_ref, what=f"tile-major M={M} N={N} K={K}")


def test_gemv_tile_major_exact(tern, orc):
    """The tile-major loop on inputs with exact answers: zero trits give 0
    (the all-ones correction cancels bit for bit), and x = 2 at one position
    with trits +-1 gives 2 s exactly, for every position of a 512-wide row."""
    N, K, M = 16, 512, 16
    s = synth.scales(6, "tme", (N, K // 128), synth.SCALE_UNIFORM)
    x = synth.activations(6, "tmx", (M, 1536))
    z = tern.gemv(dev_bf16(x), tern.pack(dev_trits(np.zeros((N, 1536), dtype=np.int8))),
                  dev_scales(synth.scales(6, "tmz", (N, 12))))
    torch.cuda.synchronize()
    assert (z.cpu().numpy() == 0).all()
    t = np.ones((N, K), dtype=np.int8)
    t[1::2] = -1
    t[:, 300:310] *= -1
    codes = tern.pack(dev_trits(t))
    for k0 in range(0, K, M):
        xe = np.zeros((M, K), dtype=np.uint16)
        for i in range(M):
            xe[i, k0 + i] = 0x4000                          # bf16 2.0
        y = tern.gemv(dev_bf16(xe), codes, dev_scales(s)).cpu().numpy()
        for i in range(M):
            k = k0 + i
            want = 2.0 * t[:, k].astype(np.float64) * s[:, k // 128].astype(np.float64)
            assert np.array_equal(y[i].astype(np.float64), want), k


def test_gemv_exact_cases(tern, orc):
    """Cases with an exact answer: all-zero trits give 0; one-hot x gives the
    column of W exactly (one nonzero product per output)."""
    N, K = 48, 512
    t = np.zeros((N, K), dtype=np.int8)
    s = synth.scales(3, "s", (N, K // 128))
    x = synth.activations(3, "x", (4, K))
    codes = tern.pack(dev_trits(t))
    y = tern.gemv(dev_bf16(x), codes, dev_scales(s))
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    t = synth.trits(4, "t", (N, K), synth.UNIFORM)
    codes = tern.pack(dev_trits(t))
    ks = [0, 5, 8, 13, 16, 100, 127, 128 + 77, 511]
    for k0 in range(0, len(ks), 8):
        kk = ks[k0:k0 + 8]
        x = np.zeros((len(kk), K), dtype=np.uint16)
        for i, k in enumerate(kk):
            x[i, k] = 0x3F80
        y = tern.gemv(dev_bf16(x), codes, dev_scales(s)).cpu().numpy()
        W = t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
        for i, k in enumerate(kk):
            assert np.array_equal(y[i].astype(np.float64), W[:, k].astype(np.float32).astype(np.float64)), k


def test_gemv_every_slot_position(tern, orc):
    """x = 1 at one position k and trits all +1: y = s exactly, for every k in
    a word and every word of a group (exercises each unpack mask and shift)."""
    N, K = 16, 128
    t = np.ones((N, K), dtype=np.int8)
    t[::2] = -1
    s = synth.scales(5, "s", (N, 1), synth.SCALE_UNIFORM)
    codes = tern.pack(dev_trits(t))
    for k0 in range(0, 128, 16):
        x = np.zeros((16, K), dtype=np.uint16)
        for i in range(16):
            x[i, k0 + i] = 0x4000                           # bf16 2.0
        y = tern.gemv(dev_bf16(x), codes, dev_scales(s)).cpu().numpy()
        want = 2.0 * t[:, 0].astype(np.float64) * s[:, 0].astype(np.float64)
        for i in range(16):
            assert np.array_equal(y[i].astype(np.float64), want), (k0 + i)


def test_gemv_wide_dynamic_range(tern, orc):
    """Activations spanning many binades (scaled per group to fp16 internally)."""
    M, N, K = 3, 64, 1024
    p = synth.problem(21, M, N, K)
    xf = np.frombuffer(p.x.tobytes(), dtype=np.uint16).copy().reshape(M, K)
    rs = np.random.default_rng(3)
    # multiply by 2^e, e in [-60, 60], by editing the bf16 exponent field
    exp = ((xf >> 7) & 0xFF).astype(np.int64)
    e = rs.integers(-60, 61, size=xf.shape)
    e[:, :128] = 40                                        # a whole group of large values
    e[:, 128:256] = -50                                    # and one of tiny values
    newexp = np.clip(exp + e, 1, 254)
    keep = exp > 0
    xf = np.where(keep, (xf & 0x807F) | (newexp.astype(np.uint16) << 7), xf).astype(np.uint16)
    y = tern.gemv(dev_bf16(xf), tern.pack(dev_trits(p.t)), dev_scales(p.s)).cpu().numpy()
    codes, _ = orc.pack(p.t)
    y_ref, a_ref = orc.matmul(xf, codes, p.s)
    assert_fp32_close(y, y_ref, a_ref, what="wide range")


def test_gemv_repeat_and_workspace_reuse(tern, orc):
    """Back-to-back calls sharing one workspace, on one stream, stay exact."""
    p1 = synth.problem(31, 5, 300, 640, tag="a")
    p2 = synth.problem(32, 16, 100, 640, tag="b")
    ws = tern.workspace(max(tern.gemv_workspace_bytes(5, 300, 640), tern.gemv_workspace_bytes(16, 100, 640)))
    c1 = tern.pack(dev_trits(p1.t))
    c2 = tern.pack(dev_trits(p2.t))
    outs = []
    for _ in range(3):
        outs.append(tern.gemv(dev_bf16(p1.x), c1, dev_scales(p1.s), ws=ws))
        outs.append(tern.gemv(dev_bf16(p2.x), c2, dev_scales(p2.s), ws=ws))
    torch.cuda.synchronize()
    r1 = orc.matmul(p1.x, orc.pack(p1.t)[0], p1.s)
    r2 = orc.matmul(p2.x, orc.pack(p2.t)[0], p2.s)
    for i, y in enumerate(outs):
        ref = r1 if i % 2 == 0 else r2
        assert_fp32_close(y.cpu().numpy(), ref[0], ref[1], what=f"call {i}")


@pytest.mark.parametrize("K,N", synth.DECODE_SHAPES)
def test_gemv_decode_full_size(tern, orc, K, N):
    """The decode shapes at M=1, every output checked (gate/up 5120->17408, down 17408->5120)."""
    p = synth.problem(2, 1, N, K, tag=f"dec{K}")
    y, codes = run_gemv(tern, p)
    want_codes, _ = orc.pack(p.t)
    assert np.array_equal(host_codes(codes), want_codes)
    y_ref, a_ref = orc.matmul(p.x, want_codes, p.s)
    assert_fp32_close(y, y_ref, a_ref, what=f"decode K={K} N={N}")


@pytest.mark.parametrize("M", synth.VERIFY_M)
@pytest.mark.parametrize("K,N", synth.VERIFY_SHAPES)
def test_gemv_verify_full_size_sampled(tern, orc, M, K, N):
    """Small-batch / speculative-verify shapes, 2048 sampled outputs each."""
    p = synth.problem(3, M, N, K, tag=f"ver{N}")
    y, codes = run_gemv(tern, p)
    rs = np.random.default_rng(M * 1000 + N)
    ms = rs.integers(0, M, 2048)
    ns = rs.integers(0, N, 2048)
    ns[:16] = N - 1 - np.arange(16)                      # the last tile
    y_ref, a_ref = orc.matmul_sampled(p.x, orc.pack(p.t)[0], p.s, ms, ns)
    assert_fp32_close(y[ms, ns], y_ref, a_ref, what=f"verify M={M} N={N}")


# ---------------------------------------------------------------------------
# rotation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (3, 8192), (2, 12288), (200, 4096)])
def test_fwht_matches_oracle(tern, orc, M, K):
    """Small calls run one CTA per 1024-wide slice, calls with at least as
    many 4096-blocks as SMs (200 tokens) one CTA per block."""
    x = synth.activations(40 + M, "x", (M, K))
    s = synth.signs(40 + M, "signs", K)
    y = tern.fwht(dev_bf16(x), torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    got = bf16_to_f64(y)
    want = orc.rotate(x, s)
    # fp32 evaluation (12 add/sub levels) then one bf16 rounding
    bound = 2.0 ** -8 * np.abs(want) + 1e-5 * np.sqrt((want ** 2).mean())
    assert (np.abs(got - want) <= bound).all(), np.max(np.abs(got - want) / bound)


def test_fwht_closed_forms(tern):
    K = 4096
    ones = torch.ones(K, dtype=torch.int8, device="cuda")
    x = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    x[0, 0] = 1.0
    x[1, :] = 3.0
    y = tern.fwht(x, ones).to(torch.float64).cpu().numpy()
    assert (y[0] == 1.0 / 64).all()
    assert y[1, 0] == 192.0 and (y[1, 1:] == 0).all()


def test_fwht_roundtrip_and_norm(tern, orc):
    K = 4096
    x = synth.activations(50, "x", (4, K))
    s = synth.signs(50, "signs", K)
    sd = torch.from_numpy(s).cuda()
    y = tern.fwht(dev_bf16(x), sd)
    xf = bf16_to_f64(dev_bf16(x))
    yn = np.linalg.norm(bf16_to_f64(y), axis=1)
    assert np.allclose(yn, np.linalg.norm(xf, axis=1), rtol=4e-3)


@pytest.mark.parametrize("M,K", [(1, 4096), (2, 4096), (5, 4096), (16, 4096), (1, 8192), (2, 12288), (3, 8192)])
def test_fwht_gemm_fused_matches_oracle(tern, orc, M, K):
    """Fused rotation + product, rotated activation kept in fp32 on chip,
    against the oracle with the rotation kept in double: the in-product
    rotation (M <= 2) and the prologue kernel (M > 2), one and several
    4096-blocks."""
    N = 1000
    p = synth.problem(60 + M, M, N, K, with_signs=True, tag=f"fz{K}")
    codes = tern.pack(dev_trits(p.t))
    y = tern.fwht_gemm(dev_bf16(p.x), torch.from_numpy(p.signs).cuda(), codes, dev_scales(p.s))
    torch.cuda.synchronize()
    y_ref, a_ref = orc.rotate_matmul(p.x, p.signs, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"fused M={M}")


def test_fwht_gemm_fused_large_n(tern, orc):
    """Three tokens on more than 8192 rows: the prologue's staged fragments
    read by the per-group product (smaller matrices take the tile-major one)."""
    M, N, K = 3, 9000, 4096
    p = synth.problem(64, M, N, K, with_signs=True, tag="fzl")
    codes = tern.pack(dev_trits(p.t))
    y = tern.fwht_gemm(dev_bf16(p.x), torch.from_numpy(p.signs).cuda(), codes, dev_scales(p.s))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.rotate_matmul(p.x, p.signs, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what="fused M=3 N=9000")


@pytest.mark.parametrize("M", [1, 16])
def test_fwht_then_gemv_separate(tern, orc, M):
    """The unfused path: tern_fwht (bf16 out), then tern_gemv on that bf16 x',
    checked against the oracle fed the same bf16 x'."""
    K, N = 4096, 12288
    p = synth.problem(70 + M, M, N, K, with_signs=True)
    codes = tern.pack(dev_trits(p.t))
    xr = tern.fwht(dev_bf16(p.x), torch.from_numpy(p.signs).cuda())
    y = tern.gemv(xr, codes, dev_scales(p.s))
    torch.cuda.synchronize()
    xr_bits = xr.view(torch.int16).cpu().numpy().view(np.uint16)
    rs = np.random.default_rng(M)
    ms = rs.integers(0, M, 4096)
    ns = rs.integers(0, N, 4096)
    y_ref, a_ref = orc.matmul_sampled(xr_bits, orc.pack(p.t)[0], p.s, ms, ns)
    assert_fp32_close(y.cpu().numpy()[ms, ns], y_ref, a_ref, what="separate")


@pytest.mark.parametrize("M", [1, 16])
def test_fwht_gemm_full_size_sampled(tern, orc, M):
    """The rotated workload: K=4096, N=12288, M in {1, 16}, sampled outputs."""
    K, N = synth.ROTATED["K"], synth.ROTATED["N"]
    p = synth.problem(4, M, N, K, with_signs=True, tag="rot")
    codes = tern.pack(dev_trits(p.t))
    y = tern.fwht_gemm(dev_bf16(p.x), torch.from_numpy(p.signs).cuda(), codes, dev_scales(p.s))
    torch.cuda.synchronize()
    # oracle on a row subset (the rotation is per token; the product per row)
    rs = np.random.default_rng(7 + M)
    rows = np.unique(rs.integers(0, N, 512))
    y_ref, a_ref = orc.rotate_matmul(p.x, p.signs, orc.pack(p.t)[0][rows], p.s[rows])
    assert_fp32_close(y.cpu().numpy()[:, rows], y_ref, a_ref, what=f"rot full M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (1, 1000, 5120), (3, 777, 17408), (6, 129, 2176), (9, 129, 2560)])
def test_gemv_overwrites_prefilled_y(tern, orc, M, N, K):
    """y holding NaN before the call is fully overwritten, for one K-slice and
    for several (whose sums are added into a y the kernel clears first)."""
    p = synth.problem(900 + M, M, N, K, tag=f"nan{N}x{K}")
    codes = tern.pack(dev_trits(p.t))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.gemv(dev_bf16(p.x), codes, dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"prefilled y M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(1, 64, 131072), (16, 40, 65536), (1, 262144, 1024), (3, 131091, 2048),
                                   (1, 1, 128), (16, 1, 17408)])
def test_gemv_extreme_shapes(tern, orc, M, N, K):
    """Very deep K (128 to 1024 groups: up to 128 K-slices per row range),
    very tall N (16,384 tiles: several CTAs per SM of ranges), and single
    rows; sampled outputs against the oracle."""
    p = synth.problem(1600 + M, M, N, K, tag=f"x{N}x{K}")
    codes = tern.pack(dev_trits(p.t))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.gemv(dev_bf16(p.x), codes, dev_scales(p.s), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    rs = np.random.default_rng(N + K)
    n = min(2000, M * N)
    ms, ns = rs.integers(0, M, n), rs.integers(0, N, n)
    ms[0], ns[0] = M - 1, N - 1
    y_ref, a_ref = orc.matmul_sampled(p.x, orc.pack(p.t)[0], p.s, ms, ns)
    assert_fp32_close(y.cpu().numpy()[ms, ns], y_ref, a_ref, what=f"extreme M={M} N={N} K={K}")
    assert torch.isfinite(y).all()


def test_scales_from_g64_device(tern, orc):
    """The group-size-64 pack's scales on the device: bit-exact against the
    oracle, differing halves counted, and the product on the converted scales
    equal to the product on the g128 scales."""
    N, K = 1000, 5120
    s128 = synth.scales(62, "g64d", (N, K // 128))
    s64 = np.repeat(s128, 2, axis=1)
    s64[10, 3] = np.float16(0.25)
    s64[999, 79] = np.float16(-1.0)
    mism = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tern.scales_from_g64(torch.from_numpy(s64).cuda(), K, mismatch=mism)
    want, wbad = orc.scales_from_g64(s64)
    assert int(mism.item()) == wbad == 2
    assert np.array_equal(out.cpu().numpy().view(np.uint16), want.view(np.uint16))
    s64 = np.repeat(s128, 2, axis=1)
    p = synth.problem(63, 1, N, K, tag="g64p")
    codes = tern.pack(dev_trits(p.t))
    x = dev_bf16(p.x)
    y64 = tern.gemv(x, codes, tern.scales_from_g64(torch.from_numpy(s64).cuda(), K))
    y128 = tern.gemv(x, codes, dev_scales(s128))
    torch.cuda.synchronize()
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], s128)
    assert_fp32_close(y64.cpu().numpy(), y_ref, a_ref, what="g64 scales")
    assert_fp32_close(y128.cpu().numpy(), y_ref, a_ref, what="g128 scales")


@pytest.mark.parametrize("M,Na,Nb,K", [(1, 17408, 17408, 5120), (1, 300, 5000, 2048), (3, 777, 129, 17408),
                                       (16, 64, 48, 1024), (5, 1000, 1000, 640), (1, 16, 16, 128),
                                       (8, 777, 300, 5120), (13, 33, 1000, 2560)])
def test_gemv_pair_matches_two_products(tern, orc, M, Na, Nb, K):
    """Two matrices read with one activation in one launch: each output against
    the oracle, ragged row counts, one and several K-slices, twice on the same
    workspace."""
    pa = synth.problem(1900 + M, M, Na, K, tag=f"pa{Na}x{K}")
    pb = synth.problem(1950 + M, M, Nb, K, tag=f"pb{Nb}x{K}")
    x = dev_bf16(pa.x)
    ca, cb = tern.pack(dev_trits(pa.t)), tern.pack(dev_trits(pb.t))
    sa, sb = dev_scales(pa.s), dev_scales(pb.s)
    ws = tern.workspace(int(tern.lib().tern_gemv_pair_workspace_bytes(M, Na, Nb, K)))
    ya_ref, aa_ref = orc.matmul(pa.x, orc.pack(pa.t)[0], pa.s)
    yb_ref, ab_ref = orc.matmul(pa.x, orc.pack(pb.t)[0], pb.s)
    for call in range(2):
        ya = torch.full((M, Na), float("nan"), dtype=torch.float32, device="cuda")
        yb = torch.full((M, Nb), float("nan"), dtype=torch.float32, device="cuda")
        tern.gemv_pair(x, ca, sa, cb, sb, y_a=ya, y_b=yb, ws=ws)
        torch.cuda.synchronize()
        assert tern.device_error() == 0
        assert_fp32_close(ya.cpu().numpy(), ya_ref, aa_ref, what=f"pair a call {call} M={M} {Na}/{Nb} K={K}")
        assert_fp32_close(yb.cpu().numpy(), yb_ref, ab_ref, what=f"pair b call {call} M={M} {Na}/{Nb} K={K}")
