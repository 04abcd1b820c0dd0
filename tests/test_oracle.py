"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: library number-format
conversions, hand-worked packing words, brute-force dense matmul from an
explicitly expanded W (built from the trits, not from the oracle's unpack),
closed forms of the Sylvester Hadamard matrix, Parseval, and the bit-rate
figures printed on the "prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Library route (torch) from bf16 bit patterns to float64."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def dense_w(t: np.ndarray, s: np.ndarray) -> np.ndarray:
    """W[n, k] = t[n, k] * s[n, k // 128], expanded from the trits themselves."""
    return t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_f16_decoder_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def test_bf16_decoder_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_bits_to_f64(bits)
    got = np.array([orc.bf16_to_f64(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# --------------------------------------------------------------------------
# packing
# --------------------------------------------------------------------------

def _golden_pack_rows():
    rows = []
    with open(os.path.join(GOLDEN, "pack_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append(([int(v) for v in parts[:16]], int(parts[16], 16)))
    return rows


def test_pack_golden_words(orc):
    rows = _golden_pack_rows()
    assert len(rows) >= 7
    t = np.array([r[0] for r in rows], dtype=np.int8)
    codes, bad = orc.pack(t)
    assert bad == 0
    assert [int(w) for w in codes[:, 0]] == [r[1] for r in rows]


def test_pack_every_slot_every_pattern(orc):
    """All 3^4 patterns of 4 consecutive trits at every slot offset 0..12 of a
    word, surrounded by random trits; the round trip must be exact."""
    rs = np.random.default_rng(7)
    pats = np.array(np.meshgrid(*[[-1, 0, 1]] * 4, indexing="ij")).reshape(4, -1).T
    rows = []
    for off in range(13):
        for p in pats:
            row = rs.integers(-1, 2, size=32).astype(np.int8)
            row[off:off + 4] = p
            row[16 + off:16 + off + 4] = p[::-1]
            rows.append(row)
    t = np.stack(rows)
    codes, bad = orc.pack(t)
    assert bad == 0 and codes.shape == (t.shape[0], 2)
    back, bad2 = orc.unpack(codes, 32)
    assert bad2 == 0
    assert np.array_equal(back, t)
    # each code individually, read from the word by the layout definition
    for i in range(0, t.shape[0], 37):
        for k in range(32):
            q = (int(codes[i, k // 16]) >> (2 * (k % 16))) & 3
            assert q == t[i, k] + 1


def test_pack_invalid_values_counted(orc):
    t = np.zeros((3, 32), dtype=np.int8)
    t[0, 5] = 2
    t[1, 31] = -2
    t[2, 0] = 127
    codes, bad = orc.pack(t)
    assert bad == 3
    assert (int(codes[0, 0]) >> 10) & 3 == 3
    assert (int(codes[1, 1]) >> 30) & 3 == 3
    back, bad2 = orc.unpack(codes, 32)
    assert bad2 == 3
    assert back[0, 5] == 0 and back[1, 31] == 0 and back[2, 0] == 0


def test_code3_rejected_by_matmul(orc):
    K = 128
    codes = np.full((1, K // 16), 0x55555555, dtype=np.uint32)
    codes[0, 3] |= 3 << 6
    s = np.ones((1, 1), dtype=np.float16)
    x = synth.activations(1, "x", (1, K))
    with pytest.raises(ValueError):
        orc.matmul(x, codes, s)


def test_pack_random_roundtrip_large(orc):
    t = synth.trits(3, "t", (64, 4096), synth.SPARSE40)
    codes, bad = orc.pack(t)
    assert bad == 0
    back, bad2 = orc.unpack(codes, 4096)
    assert bad2 == 0 and np.array_equal(back, t)


# --------------------------------------------------------------------------
# packed size and the card's bit-rate figures
# --------------------------------------------------------------------------

def test_packed_size_and_bitrates(orc):
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    N, K = 48, 1024
    t = synth.trits(4, "t", (N, K))
    s = synth.scales(4, "s", (N, K // g["group_size"]["value"]))
    codes, _ = orc.pack(t)
    nbytes = codes.nbytes + s.nbytes
    assert nbytes == N * K // 4 + N * K // 64
    bpw = 8.0 * nbytes / (N * K)
    assert bpw == g["deployed_bpw"]["value"]              # 2 + 16/128, exact
    # theoretical: log2(3) + 16/128
    theo = math.log2(3) + 16 / 128
    assert round(math.log2(3), 3) == g["log2_3_bits_per_trit"]["value"]
    assert round(theo, 2) == g["theoretical_bpw"]["value"]
    assert round(16 / g["theoretical_bpw"]["value"], 1) == g["shrink_vs_fp16"]["value"]
    # MLX: scale and bias per group -> 2 + 2*16/128
    assert 2 + 2 * 16 / 128 == g["mlx_bpw"]["value"]
    # binary sibling: 1 + 16/128
    assert 1 + 16 / 128 == g["binary_bpw"]["value"]
    # sizes, from the parameter count (the card's rounding, within 2 %)
    P = g["params_total"]["value"]
    for bpw_, key in ((bpw, "deployed_size_gb"), (theo, "theoretical_size_gb"),
                      (16.0, "fp16_size_gb"), (1.125, "binary_size_gb")):
        gb = P * bpw_ / 8 / 1e9
        assert abs(gb - g[key]["value"]) / g[key]["value"] < 0.02, (key, gb)
    # group-size-64 pack = same codes with each scale repeated per 64 values:
    # its size over the g128 pack is (2 + 16/64) / (2 + 16/128)
    ratio = g["lm_pack_g64_gb"]["value"] / g["lm_pack_g128_gb"]["value"]
    assert abs(ratio - (2 + 16 / 64) / (2 + 16 / 128)) < 1e-3


# --------------------------------------------------------------------------
# the product
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,dist", [(1, 1, 128, synth.UNIFORM), (1, 8, 128, synth.SPARSE40),
                                        (4, 8, 256, synth.UNIFORM), (3, 5, 256, synth.SPARSE40),
                                        (2, 40, 1024, synth.SPARSE40)])
def test_matmul_matches_dense_bruteforce(orc, M, N, K, dist):
    p = synth.problem(11 + M + N, M, N, K, trit_dist=dist)
    codes, bad = orc.pack(p.t)
    assert bad == 0
    y, a = orc.matmul(p.x, codes, p.s)
    xf = bf16_bits_to_f64(p.x)
    W = dense_w(p.t, p.s)
    ref = xf @ W.T
    ref_a = np.abs(xf)[:, None, :] * np.abs(W)[None, :, :]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, ref_a.sum(-1), rtol=1e-12, atol=1e-12)
    assert (a >= np.abs(y) - 1e-12).all()


def test_matmul_zero_codes_give_zero(orc):
    M, N, K = 2, 6, 384
    t = np.zeros((N, K), dtype=np.int8)
    codes, _ = orc.pack(t)
    assert (codes == 0x55555555).all()
    s = synth.scales(5, "s", (N, K // 128))
    x = synth.activations(5, "x", (M, K))
    y, a = orc.matmul(x, codes, s)
    assert (y == 0).all() and (a == 0).all()


def test_matmul_linear_in_scales(orc):
    p = synth.problem(6, 2, 7, 256)
    codes, _ = orc.pack(p.t)
    y1, _ = orc.matmul(p.x, codes, p.s)
    for alpha in (2.0, 0.5, 8.0):
        s2 = (p.s.astype(np.float32) * alpha).astype(np.float16)
        assert np.array_equal(s2.astype(np.float64), p.s.astype(np.float64) * alpha)
        y2, _ = orc.matmul(p.x, codes, s2)
        assert np.array_equal(y2, y1 * alpha)


def test_matmul_one_hot_picks_column(orc):
    N, K = 9, 256
    t = synth.trits(8, "t", (N, K), synth.UNIFORM)
    s = synth.scales(8, "s", (N, K // 128), synth.SCALE_UNIFORM)
    codes, _ = orc.pack(t)
    ks = [0, 1, 15, 16, 127, 128, 200, 255]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80                                   # bf16 1.0
    y, _ = orc.matmul(x, codes, s)
    W = dense_w(t, s)
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], W[:, k])


def test_matmul_sampled_equals_full(orc):
    p = synth.problem(9, 3, 33, 512)
    codes, _ = orc.pack(p.t)
    y, a = orc.matmul(p.x, codes, p.s)
    rs = np.random.default_rng(0)
    ms = rs.integers(0, 3, 50)
    ns = rs.integers(0, 33, 50)
    ys, as_ = orc.matmul_sampled(p.x, codes, p.s, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


def test_matmul_threads_agree(orc):
    p = synth.problem(10, 2, 64, 512)
    codes, _ = orc.pack(p.t)
    y1, _ = orc.matmul(p.x, codes, p.s, nthreads=1)
    y4, _ = orc.matmul(p.x, codes, p.s, nthreads=4)
    assert np.array_equal(y1, y4)


# --------------------------------------------------------------------------
# the MLX affine form ("MLX packaging" on the model card)
# --------------------------------------------------------------------------

def _all_positive_f16():
    bits = np.arange(1, 0x7C00, dtype=np.uint16)           # +subnormals .. max finite
    return bits.view(np.float16).astype(np.float32)


def test_mlx_affine_ternary_reading_is_exact(orc):
    """With q = t + 1, the affine map (scale s_g, bias -s_g) gives (q-1) s_g
    exactly in float32, for every positive finite fp16 scale."""
    svals = _all_positive_f16()
    for q in (0, 1, 2):
        got = np.array([orc.mlx_affine(q, float(s), float(-s)) for s in svals[::97]],
                       dtype=np.float32)
        want = ((q - 1) * svals[::97]).astype(np.float32)
        assert np.array_equal(got, want)


def test_mlx_affine_pages_literal_map(orc):
    """The card's literal map s_mlx = 2 s_g, bias = -s_g reproduces +-s_g on
    codes {0, 1} (the binary alphabet) but not the ternary code: q = 1 gives
    +s_g instead of 0 and q = 2 gives 3 s_g.  Recorded, not papered over."""
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    a, b = g["mlx_scale_factor"]["value"], g["mlx_bias_factor"]["value"]
    for s in _all_positive_f16()[::211]:
        s = float(s)
        v0 = orc.mlx_affine(0, a * s, b * s)
        v1 = orc.mlx_affine(1, a * s, b * s)
        v2 = orc.mlx_affine(2, a * s, b * s)
        assert v0 == np.float32(-s) and v1 == np.float32(s)
        assert v1 != 0.0                      # ternary q = 1 must decode to 0
        assert v2 == np.float32(3 * s) or abs(v2 - 3 * s) <= 4 * np.spacing(np.float32(3 * s))


# --------------------------------------------------------------------------
# the Walsh-Hadamard rotation
# --------------------------------------------------------------------------

def test_hadamard_explicit_matches_golden_h8(orc):
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "hadamard_h8.txt"))
            if l.strip() and not l.startswith("#")]
    assert np.array_equal(orc.hadamard_explicit(8), np.array(rows, dtype=np.float64))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
def test_hadamard_closed_form_and_orthogonality(orc, n):
    H = orc.hadamard_explicit(n)
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    assert np.array_equal(H, (-1.0) ** pc)
    assert np.array_equal(H @ H, n * np.eye(n))
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
def test_fast_transform_equals_explicit(orc, n):
    rs = np.random.default_rng(n)
    for _ in range(5):
        v = rs.standard_normal(n)
        assert np.allclose(orc.fwht(v), orc.hadamard_explicit(n) @ v, rtol=1e-13, atol=1e-13)
    # unit vectors give the columns exactly
    for j in range(n):
        e = np.zeros(n)
        e[j] = 1.0
        assert np.array_equal(orc.fwht(e), orc.hadamard_explicit(n)[:, j])


def test_rotate_closed_forms(orc):
    K = 4096
    ones = np.ones(K, dtype=np.int8)
    # e_0 -> constant 1/64
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, 0] = 0x3F80
    assert np.array_equal(orc.rotate(x, ones)[0], np.full(K, 1.0 / 64))
    # constant c -> 64 c e_0
    c = np.full((1, K), 0x4040, dtype=np.uint16)            # bf16 3.0
    r = orc.rotate(c, ones)[0]
    assert r[0] == 64 * 3.0 and (r[1:] == 0).all()
    # twice the transform is the identity (sign vector all +1)
    xf = synth.activations(12, "x", (2, K))
    r1 = orc.rotate(xf, ones)
    back = orc.unrotate(r1, ones)
    assert np.allclose(back, bf16_bits_to_f64(xf), rtol=0, atol=1e-12)


def test_rotate_parseval_signs_and_inverse(orc):
    K = 8192                                                # two blocks of 4096
    x = synth.activations(13, "x", (3, K))
    s = synth.signs(13, "signs", K)
    r = orc.rotate(x, s)
    xf = bf16_bits_to_f64(x)
    for b in (0, 4096):
        assert np.allclose(np.linalg.norm(r[:, b:b + 4096], axis=1),
                           np.linalg.norm(xf[:, b:b + 4096], axis=1), rtol=1e-13)
    # the signs multiply the input before the transform
    H = orc.hadamard_explicit(64)
    x64 = synth.activations(14, "x", (1, 64))
    s64 = synth.signs(14, "signs", 64)
    want = H @ (s64 * bf16_bits_to_f64(x64)[0]) / 8.0
    assert np.allclose(orc.rotate(x64, s64, block=64)[0], want, rtol=1e-13, atol=1e-14)
    # inverse
    back = orc.unrotate(r, s)
    assert np.allclose(back, xf, rtol=0, atol=1e-12)
    # blocks are independent: a change in block 1 leaves block 0 alone
    x2 = x.copy()
    x2[:, 5000] ^= 0x0001
    r2 = orc.rotate(x2, s)
    assert np.array_equal(r2[:, :4096], r[:, :4096])
    assert not np.array_equal(r2[:, 4096:], r[:, 4096:])


def test_rotate_matmul_bruteforce(orc):
    M, N, K = 2, 24, 4096
    p = synth.problem(15, M, N, K, with_signs=True)
    codes, _ = orc.pack(p.t)
    y, a = orc.rotate_matmul(p.x, p.signs, codes, p.s)
    H = orc.hadamard_explicit(64)
    # rotation by the Kronecker structure H_4096 = H_64 (x) H_64, written out
    xf = bf16_bits_to_f64(p.x) * p.signs
    xr = np.einsum("ab,cd,mbd->mac", H, H, xf.reshape(M, 64, 64)).reshape(M, K) / 64.0
    W = dense_w(p.t, p.s)
    assert np.allclose(y, xr @ W.T, rtol=1e-10, atol=1e-10)
    assert np.allclose(a, np.abs(xr) @ np.abs(W).T, rtol=1e-10)


# --------------------------------------------------------------------------
# the 1-bit sibling (binary g128): w = (2b - 1) s_g, bit k%32 of word k/32
# --------------------------------------------------------------------------

def binary_trits(seed: int, name: str, shape) -> np.ndarray:
    return np.where(synth.trits(seed, name, shape, synth.UNIFORM) >= 0, 1, -1).astype(np.int8)


def test_bin_pack_golden_words(orc):
    rows = []
    with open(os.path.join(GOLDEN, "bin_pack_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            rows.append(([int(v) for v in parts[:32]], int(parts[32], 16)))
    assert len(rows) >= 8
    t = np.array([r[0] for r in rows], dtype=np.int8)
    words, bad = orc.bin_pack(t)
    assert bad == 0
    assert [int(w) for w in words[:, 0]] == [r[1] for r in rows]
    assert np.array_equal(orc.bin_unpack(words, 32), t)


def test_bin_pack_every_position_and_roundtrip(orc):
    """A single +1 at any position k of a row sets bit k % 32 of word k / 32
    only; random rows survive the round trip."""
    K = 128
    for k in range(K):
        t = -np.ones((1, K), dtype=np.int8)
        t[0, k] = 1
        words, bad = orc.bin_pack(t)
        want = np.zeros(K // 32, dtype=np.uint32)
        want[k // 32] = np.uint32(1) << np.uint32(k % 32)
        assert bad == 0 and np.array_equal(words[0], want), k
    t = binary_trits(21, "rt", (37, 2048))
    words, bad = orc.bin_pack(t)
    assert bad == 0
    assert np.array_equal(orc.bin_unpack(words, 2048), t)


def test_bin_pack_invalid_values_counted(orc):
    t = np.array([[1, -1, 0, 2] + [1] * 28], dtype=np.int8)
    words, bad = orc.bin_pack(t)
    assert bad == 2
    # invalid entries are stored as -1 (bit 0)
    assert int(words[0, 0]) == (0xFFFFFFFF & ~0b1110)


def test_bin_packed_size_and_bitrate(orc):
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    N, K = 48, 1024
    words, _ = orc.bin_pack(binary_trits(22, "sz", (N, K)))
    s = synth.scales(22, "s", (N, K // 128))
    nbytes = words.nbytes + s.nbytes
    assert nbytes == N * K // 8 + N * K // 64
    assert 8.0 * nbytes / (N * K) == g["binary_bpw"]["value"]   # 1 + 16/128, exact


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (1, 8, 128), (4, 8, 256), (3, 5, 384), (2, 40, 1024)])
def test_bin_matmul_matches_dense_bruteforce(orc, M, N, K):
    t = binary_trits(30 + N, "bf", (N, K))
    s = synth.scales(30 + N, "s", (N, K // 128))
    x = synth.activations(30 + N, "x", (M, K))
    words, _ = orc.bin_pack(t)
    y, a = orc.bin_matmul(x, words, s)
    xf = bf16_bits_to_f64(x)
    W = dense_w(t, s)
    assert np.allclose(y, xf @ W.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf) @ np.abs(W).T, rtol=1e-12, atol=1e-12)


def test_bin_matmul_equals_ternary_oracle_on_pm1(orc):
    """On weights in {-1, +1} the binary product is the ternary product of the
    same trits, through the ternary packing and the ternary dot product."""
    M, N, K = 3, 17, 640
    t = binary_trits(31, "tt", (N, K))
    s = synth.scales(31, "s", (N, K // 128))
    x = synth.activations(31, "x", (M, K))
    yb, ab = orc.bin_matmul(x, orc.bin_pack(t)[0], s)
    yt, at = orc.matmul(x, orc.pack(t)[0], s)
    assert np.array_equal(yb, yt) and np.array_equal(ab, at)


def test_bin_matmul_closed_forms(orc):
    """All weights +1: y = sum_g s_g sum_{k in g} x_k; flipping every sign
    negates y; a one-hot x picks +-s of one column; powers of two scale y
    exactly."""
    M, N, K = 2, 6, 384
    s = synth.scales(32, "s", (N, K // 128))
    x = synth.activations(32, "x", (M, K))
    ones = np.ones((N, K), dtype=np.int8)
    y, _ = orc.bin_matmul(x, orc.bin_pack(ones)[0], s)
    xf = bf16_bits_to_f64(x).reshape(M, K // 128, 128).sum(-1)      # exact sums of bf16 values
    assert np.array_equal(y, xf @ s.astype(np.float64).T)
    ym, _ = orc.bin_matmul(x, orc.bin_pack(-ones)[0], s)
    assert np.array_equal(ym, -y)
    t = binary_trits(33, "oh", (N, K))
    words = orc.bin_pack(t)[0]
    ks = [0, 31, 32, 127, 128, 383]
    xo = np.zeros((len(ks), K), dtype=np.uint16)
    for i, k in enumerate(ks):
        xo[i, k] = 0x3F80
    yo, _ = orc.bin_matmul(xo, words, s)
    W = dense_w(t, s)
    for i, k in enumerate(ks):
        assert np.array_equal(yo[i], W[:, k])
    y1, _ = orc.bin_matmul(x, words, s)
    y2, _ = orc.bin_matmul(x, words, (s.astype(np.float32) * 4).astype(np.float16))
    assert np.array_equal(y2, 4 * y1)


def test_bin_matmul_sampled_equals_full(orc):
    M, N, K = 3, 29, 512
    t = binary_trits(34, "sm", (N, K))
    s = synth.scales(34, "s", (N, K // 128))
    x = synth.activations(34, "x", (M, K))
    words = orc.bin_pack(t)[0]
    y, a = orc.bin_matmul(x, words, s)
    ms = np.repeat(np.arange(M), N)
    ns = np.tile(np.arange(N), M)
    ys, as_ = orc.bin_matmul_sampled(x, words, s, ms, ns)
    assert np.array_equal(ys, y.reshape(-1)) and np.array_equal(as_, a.reshape(-1))


# --------------------------------------------------------------------------
# the group-size-64 pack's scales: each g128 scale repeated in both halves
# --------------------------------------------------------------------------

def test_scales_from_g64(orc):
    s128 = synth.scales(60, "g64", (7, 5))
    s64 = np.repeat(s128, 2, axis=1)                  # the repeated layout, built independently
    out, bad = orc.scales_from_g64(s64)
    assert bad == 0 and np.array_equal(out.view(np.uint16), s128.view(np.uint16))
    s64[2, 3] = np.float16(0.5)                       # second half of group 1 differs
    s64[6, 8] = np.float16(-0.0)                      # first half of group 4 differs (bitwise)
    out, bad = orc.scales_from_g64(s64)
    assert bad == 2
    assert out[2, 1] == s128[2, 1] and out[6, 4].view(np.uint16) == np.float16(-0.0).view(np.uint16)
    # the card's pack sizes agree with one fp16 per 64 weights instead of per 128
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    assert abs(g["lm_pack_g64_gb"]["value"] / g["lm_pack_g128_gb"]["value"] - (2 + 16 / 64) / (2 + 16 / 128)) < 1e-3


# --------------------------------------------------------------------------
# the affine pack ("MLX packaging": a scale and a bias per group of 128),
# w = s q + b with every 2-bit code 0..3 valid
# --------------------------------------------------------------------------

def pack_codes_np(q: np.ndarray) -> np.ndarray:
    """uint32 words from codes q [N, K] in 0..3: code k at bits 2 (k % 16) of
    word k / 16 (the slot order the packing golden words fix), built with
    numpy independently of the oracle."""
    N, K = q.shape
    w = q.astype(np.uint64).reshape(N, K // 16, 16) << (2 * np.arange(16, dtype=np.uint64))
    return w.sum(-1).astype(np.uint32)


def dense_affine_w(q: np.ndarray, s: np.ndarray, b: np.ndarray) -> np.ndarray:
    return q.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1) + \
        np.repeat(b.astype(np.float64), 128, axis=1)


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (1, 8, 128), (4, 8, 256), (3, 5, 384), (2, 40, 1024)])
def test_affine_matmul_matches_dense_bruteforce(orc, M, N, K):
    q = synth.rng(40 + N, "q").integers(0, 4, size=(N, K))
    s = synth.scales(40 + N, "s", (N, K // 128))
    b = synth.biases(40 + N, "b", s)
    x = synth.activations(40 + N, "x", (M, K))
    y, a = orc.affine_matmul(x, pack_codes_np(q), s, b)
    xf = bf16_bits_to_f64(x)
    W = dense_affine_w(q, s, b)
    assert np.allclose(y, xf @ W.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf) @ np.abs(W).T, rtol=1e-12, atol=1e-12)


def test_affine_packer_agrees_with_ternary_golden_layout(orc):
    """The test's own packer and the oracle's ternary packer lay codes 0..2 out
    identically (so the affine pins use the layout the golden words fix)."""
    t = synth.trits(41, "t", (6, 256), synth.UNIFORM)
    assert np.array_equal(pack_codes_np(t.astype(np.int64) + 1), orc.pack(t)[0])


def test_affine_matmul_ternary_case_is_the_ternary_product(orc):
    """b = -s on codes q = t + 1 is the ternary product, bit for bit."""
    p = synth.problem(42, 3, 21, 640)
    codes, _ = orc.pack(p.t)
    ya, aa = orc.affine_matmul(p.x, codes, p.s, -p.s)
    yt, at = orc.matmul(p.x, codes, p.s)
    assert np.array_equal(ya, yt) and np.array_equal(aa, at)


def test_affine_matmul_cards_literal_pair_is_the_binary_product(orc):
    """The card's MLX pair (2 s_g, -s_g) on codes {0, 1} is the 1-bit product
    of b = q, bit for bit ("exactly reproduces +-s_g" holds there)."""
    M, N, K = 2, 13, 512
    q = (synth.binary(43, "q", (N, K)) > 0).astype(np.int8)          # 0 or 1
    s = synth.scales(43, "s", (N, K // 128))
    x = synth.activations(43, "x", (M, K))
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    fa, fb = g["mlx_scale_factor"]["value"], g["mlx_bias_factor"]["value"]
    s_mlx = (s.astype(np.float64) * fa).astype(np.float16)
    b_mlx = (s.astype(np.float64) * fb).astype(np.float16)
    assert np.array_equal(s_mlx.astype(np.float64), 2 * s.astype(np.float64))
    ya, aa = orc.affine_matmul(x, orc.pack(q - 1)[0], s_mlx, b_mlx)
    yb, ab = orc.bin_matmul(x, orc.bin_pack(2 * q - 1)[0], s)
    assert np.array_equal(ya, yb) and np.array_equal(aa, ab)


def test_affine_matmul_closed_forms(orc):
    """All codes 3: y = sum_g (3 s_g + b_g) X_g with X_g the group sums of x;
    zero scales: y = sum_g b_g X_g; zero scales and biases: y = 0; a one-hot x
    picks s q + b of one column exactly."""
    M, N, K = 2, 6, 384
    s = synth.scales(44, "s", (N, K // 128))
    b = synth.biases(44, "b", s)
    x = synth.activations(44, "x", (M, K))
    X = bf16_bits_to_f64(x).reshape(M, K // 128, 128).sum(-1)     # exact sums of bf16 values
    threes = np.full((N, K // 16), 0xFFFFFFFF, dtype=np.uint32)
    y, _ = orc.affine_matmul(x, threes, s, b)
    assert np.allclose(y, X @ (3 * s.astype(np.float64) + b.astype(np.float64)).T, rtol=1e-13, atol=1e-13)
    z = np.zeros_like(s)
    words = synth.code_words(44, "c", (N, K // 16))
    y, _ = orc.affine_matmul(x, words, z, b)
    assert np.allclose(y, X @ b.astype(np.float64).T, rtol=1e-13, atol=1e-13)
    y, a = orc.affine_matmul(x, words, z, z)
    assert (y == 0).all() and (a == 0).all()
    q = synth.rng(44, "q").integers(0, 4, size=(N, K))
    ks = [0, 15, 16, 127, 128, 383]
    xo = np.zeros((len(ks), K), dtype=np.uint16)
    for i, k in enumerate(ks):
        xo[i, k] = 0x3F80
    yo, _ = orc.affine_matmul(xo, pack_codes_np(q), s, b)
    W = dense_affine_w(q, s, b)
    for i, k in enumerate(ks):
        assert np.array_equal(yo[i], W[:, k])


def test_affine_matmul_sampled_equals_full(orc):
    p = synth.affine_problem(45, 3, 29, 512)
    y, a = orc.affine_matmul(p.x, p.codes, p.s, p.b)
    ms = np.repeat(np.arange(3), 29)
    ns = np.tile(np.arange(29), 3)
    ys, as_ = orc.affine_matmul_sampled(p.x, p.codes, p.s, p.b, ms, ns)
    assert np.array_equal(ys, y.reshape(-1)) and np.array_equal(as_, a.reshape(-1))


# --------------------------------------------------------------------------
# the rotation at its real block size against a library routine
# --------------------------------------------------------------------------

def test_rotation_at_4096_matches_scipy_sylvester_matrix(orc):
    """scipy.linalg.hadamard builds Sylvester's construction (natural order)
    independently; the oracle's 4096-point rotation is H_4096 (s x) / 64
    against it, for two blocks of two tokens, and the explicit matrix agrees
    with it entry for entry up to n = 1024."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    for n in (1, 2, 16, 256, 1024):
        assert np.array_equal(orc.hadamard_explicit(n), scipy_linalg.hadamard(n).astype(np.float64))
    K = 8192
    H = scipy_linalg.hadamard(4096, dtype=np.int8).astype(np.float64)
    x = synth.activations(16, "x4096", (2, K))
    s = synth.signs(16, "s4096", K)
    got = orc.rotate(x, s)
    xs = bf16_bits_to_f64(x) * s
    want = np.concatenate([xs[:, :4096] @ H.T, xs[:, 4096:] @ H.T], axis=1) / 64.0
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    v = synth.activations(17, "v", (1, 4096)).astype(np.float64)
    assert np.allclose(orc.fwht(v[0]), H @ v[0], rtol=0, atol=1e-9)
