"""GPU parity of the affine pack (a scale and a bias per group of 128,
w = s q + b, every 2-bit code 0..3 valid).

The decode product is held to |y - y_ref| <= 1e-3 * sum_k |x w| + 2^-23 *
sum_k |x_k b_g(k)| + 1e-6 against the oracle's double-precision product: the
kernel sums s * sum q x and b * sum x in fp32 and the two parts may cancel, so
the rounding of the bias part is bounded by its own magnitude.

The prefill product forms each of a group's four weights s q + b in fp32 and
rounds it once to bf16, so a weight differs from the exact one by
d_q = bf16(fp32(s q + b)) - (s q + b), which the test computes exactly.  The
difference from the oracle is then bounded by what those roundings explain,
sum_g sum_q |d_q| |sum_{k in g, q_k = q} x_k|, plus 2^-12 * sum_k |x w| for the
fp32 accumulation and 1e-6; a bf16 output adds its own rounding, 2^-8 of the
result.  A one-hot activation picks s q + b of one column: exactly its fp32
value from the decode product and exactly its bf16 value from the prefill
product, at every slot position (codes 5-7 and 13-15 are the ones the ternary
unpack cannot read as 3).  Shapes span full and short K-slices, ragged N,
M = 1..16, and the lean and general loops.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import ACC_REL, assert_fp32_close, assert_within, dev_bf16, dev_codes, dev_scales, dev_trits, x_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def bias_scale(x_bits: np.ndarray, b: np.ndarray) -> np.ndarray:
    """sum_k |x[m, k]| |b[n, k / 128]| for every (m, n)."""
    xa = np.abs(x_f64(x_bits))
    M, K = xa.shape
    return xa.reshape(M, K // 128, 128).sum(-1) @ np.abs(b.astype(np.float64)).T


def check_decode(y, p, y_ref, a_ref, ms=None, ns=None, what=""):
    B = bias_scale(p.x, p.b)
    if ms is not None:
        B = B[ms, ns]
    assert_fp32_close(y, y_ref, a_ref, abs_=2.0 ** -23 * B + 1e-6, what=what)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (1, 1000, 5120), (3, 777, 17408), (6, 129, 2176),
                                   (5, 200, 640), (16, 300, 1152), (2, 48, 128), (8, 129, 1024),
                                   (1, 16, 128), (9, 100, 3072), (1, 333, 2176)])
def test_affine_gemv_matches_oracle(tern, orc, M, N, K):
    p = synth.affine_problem(200 + M, M, N, K, tag=f"a{N}x{K}")
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    tern.affine_gemv(dev_bf16(p.x), dev_codes(p.codes), dev_scales(p.s), dev_scales(p.b), y=y)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.affine_matmul(p.x, p.codes, p.s, p.b)
    check_decode(y.cpu().numpy(), p, y_ref, a_ref, what=f"affine M={M} N={N} K={K}")


def one_hot_rows(ks, K):
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80
    return x


ONE_HOT_KS = [0, 4, 5, 6, 7, 8, 12, 13, 14, 15, 21, 29, 100, 127, 128, 133, 255]


def test_affine_gemv_one_hot_exact(tern):
    """x = e_k picks fp32(s q + b) of column k, every slot position and code."""
    N, K = 64, 256
    p = synth.affine_problem(210, 1, N, K, tag="oh")
    codes = p.codes.copy()
    codes[:4] = 0xFFFFFFFF                     # code 3 at every slot of four rows
    q = ((codes[:, :, None] >> (2 * np.arange(16, dtype=np.uint32))) & 3).reshape(N, K)
    W = (np.repeat(p.s.astype(np.float32), 128, axis=1) * q.astype(np.float32) +
         np.repeat(p.b.astype(np.float32), 128, axis=1))
    c, s, b = dev_codes(codes), dev_scales(p.s), dev_scales(p.b)
    for i in range(0, len(ONE_HOT_KS), 8):
        chunk = ONE_HOT_KS[i:i + 8]
        y = tern.affine_gemv(dev_bf16(one_hot_rows(chunk, K)), c, s, b).cpu().numpy()
        for j, k in enumerate(chunk):
            assert np.array_equal(y[j], W[:, k]), k


@pytest.mark.parametrize("M,K,N", [(1, 5120, 17408), (1, 17408, 5120), (5, 5120, 6144), (16, 5120, 17408)])
def test_affine_gemv_full_size_sampled(tern, orc, M, K, N):
    p = synth.affine_problem(220 + M, M, N, K, tag=f"f{K}")
    y = tern.affine_gemv(dev_bf16(p.x), dev_codes(p.codes), dev_scales(p.s), dev_scales(p.b))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    rs = np.random.default_rng(K + N + M)
    ms, ns = rs.integers(0, M, 3000), rs.integers(0, N, 3000)
    ms[:4], ns[:4] = M - 1, [0, N - 1, N - 2, N // 2]
    y_ref, a_ref = orc.affine_matmul_sampled(p.x, p.codes, p.s, p.b, ms, ns)
    check_decode(y.cpu().numpy()[ms, ns], p, y_ref, a_ref, ms, ns, what=f"affine full M={M} {K}->{N}")


def test_affine_special_cases(tern, orc):
    """b = -s on ternary codes is the ternary product; the card's MLX pair
    (2 s, -s) on codes {0, 1} is the 1-bit product."""
    M, N, K = 3, 500, 5120
    p = synth.problem(230, M, N, K, tag="tern")
    codes = tern.pack(dev_trits(p.t))
    x, s = dev_bf16(p.x), dev_scales(p.s)
    y = tern.affine_gemv(x, codes, s, -s)
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, abs_=2.0 ** -23 * bias_scale(p.x, p.s) + 1e-6,
                      what="affine as ternary")
    qb = (synth.binary(231, "q", (N, K)) > 0).astype(np.int8)
    codes01 = tern.pack(dev_trits(qb - 1))                         # codes q in {0, 1}
    s2 = (p.s.astype(np.float64) * 2).astype(np.float16)
    y = tern.affine_gemv(x, codes01, dev_scales(s2), -s)
    y_ref, a_ref = orc.bin_matmul(p.x, orc.bin_pack(2 * qb - 1)[0], p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, abs_=2.0 ** -23 * bias_scale(p.x, p.s) + 1e-6,
                      what="affine as the card's MLX pair")


# --------------------------------------------------------------------------
# the prefill product (tcgen05)
# --------------------------------------------------------------------------

def codes_q(codes: np.ndarray) -> np.ndarray:
    """The 2-bit codes [N, K] of a packed matrix."""
    N = codes.shape[0]
    return ((codes[:, :, None] >> (2 * np.arange(16, dtype=np.uint32))) & 3).reshape(N, -1).astype(np.uint8)


def weight_rounding(s: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|bf16(fp32(s q + b)) - (s q + b)| for q = 0..3: [N, G, 4]."""
    q = np.arange(4, dtype=np.float32)
    w32 = s.astype(np.float32)[:, :, None] * q + b.astype(np.float32)[:, :, None]
    wb = torch.from_numpy(w32).to(torch.bfloat16).to(torch.float64).numpy()
    exact = s.astype(np.float64)[:, :, None] * q.astype(np.float64) + b.astype(np.float64)[:, :, None]
    return np.abs(wb - exact)


def affine_rounding_bound(p, ms=None, ns=None) -> np.ndarray:
    """sum_g sum_q |d_q| |sum_{k in g, q_k = q} x_k| per output."""
    x = x_f64(p.x)
    qa = codes_q(p.codes)
    d = weight_rounding(p.s, p.b)
    M, K = x.shape
    G = K // 128
    if ms is None:
        out = np.zeros((M, qa.shape[0]))
        for g in range(G):
            sl = slice(128 * g, 128 * g + 128)
            for q in range(4):
                out += np.abs(x[:, sl] @ (qa[:, sl] == q).T.astype(np.float64)) * d[:, g, q][None, :]
        return out
    xs = x[ms].reshape(len(ms), G, 128)
    qs = qa[ns].reshape(len(ns), G, 128)
    out = np.zeros(len(ms))
    for q in range(4):
        out += (np.abs((xs * (qs == q)).sum(axis=2)) * d[ns, :, q]).sum(axis=1)
    return out


def check_prefill(y, p, y_ref, a_ref, bf16_out, ms=None, ns=None, what=""):
    bound = affine_rounding_bound(p, ms, ns) + ACC_REL * a_ref + 1e-6
    if bf16_out:
        bound = bound * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y_ref)
    assert_within(y, y_ref, bound, what=what)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 200, 256), (200, 256, 1024), (300, 130, 640),
                                   (512, 512, 2048), (17, 1000, 128), (256, 256, 8192), (40, 128, 2048)])
def test_affine_gemm_matches_oracle(tern, orc, M, N, K):
    p = synth.affine_problem(240 + M, M, N, K, tag=f"m{N}x{K}")
    y = tern.affine_gemm(dev_bf16(p.x), dev_codes(p.codes), dev_scales(p.s), dev_scales(p.b))
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.affine_matmul(p.x, p.codes, p.s, p.b)
    check_prefill(y.cpu().numpy(), p, y_ref, a_ref, False, what=f"affine gemm M={M} N={N} K={K}")


def test_affine_gemm_bf16_and_one_hot(tern, orc):
    M, N, K = 256, 384, 512
    p = synth.affine_problem(250, M, N, K, tag="b16")
    c, s, b = dev_codes(p.codes), dev_scales(p.s), dev_scales(p.b)
    y = tern.affine_gemm(dev_bf16(p.x), c, s, b, out_dtype=torch.bfloat16)
    y_ref, a_ref = orc.affine_matmul(p.x, p.codes, p.s, p.b)
    check_prefill(y.to(torch.float64).cpu().numpy(), p, y_ref, a_ref, True, what="affine gemm bf16")
    # one-hot rows of x pick bf16(fp32(s q + b)) exactly
    q = codes_q(p.codes)
    W32 = (np.repeat(p.s.astype(np.float32), 128, axis=1) * q.astype(np.float32) +
           np.repeat(p.b.astype(np.float32), 128, axis=1))
    Wb = torch.from_numpy(W32).to(torch.bfloat16).to(torch.float64).numpy()
    ks = [(37 * m) % K for m in range(M)]
    y = tern.affine_gemm(dev_bf16(one_hot_rows(ks, K)), c, s, b).cpu().numpy()
    for m in range(M):
        assert np.array_equal(y[m].astype(np.float64), Wb[:, ks[m]]), m


@pytest.mark.parametrize("name,K,N", [(n, k, nn) for (n, k, nn) in synth.PREFILL_LAYER])
def test_affine_gemm_prefill_layer_sampled(tern, orc, name, K, N):
    M = synth.PREFILL_M
    p = synth.affine_problem(260, M, N, K, tag=f"ap{name}")
    c, s, b = dev_codes(p.codes), dev_scales(p.s), dev_scales(p.b)
    y = tern.affine_gemm(dev_bf16(p.x), c, s, b, out_dtype=torch.bfloat16)
    y32 = tern.affine_gemm(dev_bf16(p.x), c, s, b)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    rs = np.random.default_rng(K + N + 7)
    ms, ns = rs.integers(0, M, 3000), rs.integers(0, N, 3000)
    ms[:4], ns[:4] = M - 1, [0, N - 1, N - 2, N // 2]
    y_ref, a_ref = orc.affine_matmul_sampled(p.x, p.codes, p.s, p.b, ms, ns)
    check_prefill(y.to(torch.float64).cpu().numpy()[ms, ns], p, y_ref, a_ref, True, ms, ns,
                  what=f"affine pp512 {name}")
    check_prefill(y32.cpu().numpy()[ms, ns], p, y_ref, a_ref, False, ms, ns, what=f"affine pp512 {name} fp32")
