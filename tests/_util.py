"""Shared test helpers: moving seeded inputs to the device and tolerance checks."""
import numpy as np
import torch


def dev_trits(t: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(t)).cuda()


def dev_scales(s: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(s, dtype=np.float16)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_codes(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint32).view(np.int32)).cuda()


def host_codes(codes: torch.Tensor) -> np.ndarray:
    return codes.cpu().numpy().view(np.uint32)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).cpu().numpy()


def assert_fp32_close(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray, rel: float = 1e-3,
                      abs_: float = 1e-6, what: str = ""):
    """|y - y_ref| <= rel * sum_k |x w| + abs_ per element (the fp32 bound)."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bound = rel * a_ref + abs_
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside the bound; worst ratio "
            f"{np.max(err / bound):.3g}; first {i.tolist()}: got {y_gpu[bad][:5]}, want {y_ref[bad][:5]}")
    return float(np.max(err / bound)) if err.size else 0.0


# ---------------------------------------------------------------------------
# Prefill tolerances.  The prefill kernels fold each group scale into the bf16
# weight operand: a ternary or 1-bit weight is exactly t * bf16(s_g) (the fp16
# scale rounded to nearest even), which is the operand the product is defined
# on.  So the oracle is handed those rounded scales and the fp32 output is held
# to the stated 1e-3 * sum_k |x w| + 1e-6, the bf16 output to
# 8e-3 * max(|y_ref|, ||x (.) w||_2).  A second check against the exact-scale
# oracle bounds the whole difference by what the rounding of each scale
# explains: sum_g |bf16(s_g) - s_g| * |sum_{k in g} x_k t_k|, plus 2^-12 * A
# for the fp32 accumulation.
# ---------------------------------------------------------------------------
ACC_REL = 2.0 ** -12


def f16_to_bf16_f16(s: np.ndarray) -> np.ndarray:
    """fp16 values rounded to bf16 (nearest even), returned as fp16: every such
    value below 65280 is an fp16 value, and the tests use no larger scale."""
    f = np.asarray(s, dtype=np.float16).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    r = (((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)).view(np.float32)
    out = r.astype(np.float16)
    if not np.array_equal(out.astype(np.float32), r):
        raise ValueError("a bf16-rounded scale is not an fp16 value")
    return out


def x_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scale_rounding_bound(x_bits, t, s, ms=None, ns=None):
    """sum_g |bf16(s_g) - s_g| |sum_{k in g} x_k t_k| for every output (ms, ns
    None) or for the outputs (ms[i], ns[i])."""
    x = x_f64(x_bits)
    t = np.asarray(t, dtype=np.float64)
    ds = np.abs(f16_to_bf16_f16(s).astype(np.float64) - np.asarray(s, dtype=np.float16).astype(np.float64))
    M, K = x.shape
    G = K // 128
    if ms is None:
        out = np.zeros((M, t.shape[0]))
        for g in range(G):
            sl = slice(128 * g, 128 * g + 128)
            out += np.abs(x[:, sl] @ t[:, sl].T) * ds[:, g][None, :]
        return out
    xs = x[ms].reshape(len(ms), G, 128)
    ts = t[ns].reshape(len(ns), G, 128)
    return (np.abs((xs * ts).sum(axis=2)) * ds[ns]).sum(axis=1)


def l2_xw(x_bits, t, s, ms=None, ns=None):
    """||x (.) w||_2 per output, w = t * s per group."""
    x2 = x_f64(x_bits) ** 2
    w2 = (np.asarray(t, dtype=np.float64) * np.repeat(np.asarray(s, dtype=np.float16).astype(np.float64), 128,
                                                       axis=1)) ** 2
    if ms is None:
        return np.sqrt(x2 @ w2.T)
    return np.sqrt((x2[ms] * w2[ns]).sum(axis=1))


def assert_bf16_close(y_gpu, y_ref, l2, rel: float = 8e-3, what: str = ""):
    """|y - y_ref| <= rel * max(|y_ref|, ||x (.) w||_2) per element (the bf16-output bound)."""
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    bound = rel * np.maximum(np.abs(y_ref), l2)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside the bf16 bound; worst ratio "
            f"{np.max(err / np.maximum(bound, 1e-300)):.3g}; first {i.tolist()}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def assert_within(y_gpu, y_ref, bound, what: str = ""):
    """|y - y_ref| <= bound per element."""
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside the bound; worst ratio "
                             f"{np.max(err / np.maximum(bound, 1e-300)):.3g}; first {i.tolist()}")
