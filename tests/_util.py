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
