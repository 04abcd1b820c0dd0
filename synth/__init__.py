"""Seeded synthetic inputs for the ternary-g128 product and the rotation.

This module only draws random inputs; it holds none of the method's
arithmetic (no packing, no unpacking, no product, no transform).  It is the one
module that both the CPU oracle's callers and the CUDA path's callers share.

The distributions follow the workloads the pages describe (a 27B hybrid
backbone with ternary g128 weights, decode at batch 1, speculative verify at
k+1 = 5 tokens, prefill of 512 tokens); the exact hidden sizes are stand-ins,
since the pages give none:

* trits t in {-1, 0, +1}: iid, either uniform or with P(0) = 0.4, P(+-1) = 0.3;
* scales: fp16, U[0.005, 0.05] or |N(0, 0.02)| + 1e-3, one per 128 along K;
* activations x: bf16 rounded from N(0, 1) (round to nearest even);
* rotation signs: iid uniform over {-1, +1}, int8;
* the 1-bit sibling format's weights: iid uniform over {-1, +1};
* an affine pack's 2-bit codes: every slot iid uniform over {0, 1, 2, 3}
  (drawn as whole random 32-bit words), and fp16 biases b = -u s with
  u ~ U[1, 2] (a min-max fit of symmetric weights puts b near -1.5 s).

Each tensor draws from its own stream, keyed by (seed, name), so one tensor's
shape never shifts another tensor's values.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

UNIFORM = "uniform"          # P(-1) = P(0) = P(+1) = 1/3
SPARSE40 = "p0=0.4"          # P(0) = 0.4, P(-1) = P(+1) = 0.3
SCALE_UNIFORM = "U[0.005,0.05]"
SCALE_HALFNORMAL = "|N(0,0.02)|+1e-3"


def rng(seed: int, name: str) -> np.random.Generator:
    """An independent PCG64 stream for tensor `name` under `seed`."""
    key = zlib.crc32(name.encode("utf-8"))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), key])))


def binary(seed: int, name: str, shape) -> np.ndarray:
    """int8 array of iid values in {-1, +1}, each with probability 1/2 (the
    1-bit sibling format's weights)."""
    return np.where(rng(seed, name).random(shape) < 0.5, -1, 1).astype(np.int8)


def binary_problem(seed: int, M: int, N: int, K: int, tag: str = "") -> "Problem":
    """A seeded problem of the 1-bit format: t in {-1, +1}."""
    return Problem(M, N, K, binary(seed, f"{tag}b", (N, K)), scales(seed, f"{tag}s", (N, K // 128)),
                   activations(seed, f"{tag}x", (M, K)))


def code_words(seed: int, name: str, shape) -> np.ndarray:
    """uint32 array of iid random words: every 2-bit slot uniform over 0..3."""
    return rng(seed, name).integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)


def biases(seed: int, name: str, s: np.ndarray) -> np.ndarray:
    """float16 group biases b = -u s, u ~ U[1, 2] iid, for fp16 scales s."""
    u = rng(seed, name).uniform(1.0, 2.0, size=s.shape)
    return (-u * s.astype(np.float64)).astype(np.float16)


@dataclass
class AffineProblem:
    """One seeded problem on an affine pack: w = s q + b per group of 128."""
    M: int
    N: int
    K: int
    codes: np.ndarray      # uint32 [N, K/16]
    s: np.ndarray          # float16 [N, K/128]
    b: np.ndarray          # float16 [N, K/128]
    x: np.ndarray          # uint16 bf16 bits [M, K]


def affine_problem(seed: int, M: int, N: int, K: int, tag: str = "") -> AffineProblem:
    """A seeded problem on an affine pack (all four codes, biases near -1.5 s)."""
    s = scales(seed, f"{tag}s", (N, K // 128))
    return AffineProblem(M, N, K, code_words(seed, f"{tag}c", (N, K // 16)), s, biases(seed, f"{tag}b", s),
                         activations(seed, f"{tag}x", (M, K)))


def trits(seed: int, name: str, shape, dist: str = SPARSE40) -> np.ndarray:
    """int8 array of iid values in {-1, 0, +1}."""
    g = rng(seed, name)
    u = g.random(shape, dtype=np.float32)
    if dist == UNIFORM:
        edges = (1.0 / 3.0, 2.0 / 3.0)
    elif dist == SPARSE40:
        edges = (0.3, 0.7)
    else:
        raise ValueError(f"unknown trit distribution {dist!r}")
    out = np.full(shape, 1, dtype=np.int8)
    out[u < edges[1]] = 0
    out[u < edges[0]] = -1
    return out


def scales(seed: int, name: str, shape, dist: str = SCALE_HALFNORMAL) -> np.ndarray:
    """float16 array of positive group scales."""
    g = rng(seed, name)
    if dist == SCALE_UNIFORM:
        v = g.uniform(0.005, 0.05, size=shape)
    elif dist == SCALE_HALFNORMAL:
        v = np.abs(g.normal(0.0, 0.02, size=shape)) + 1e-3
    else:
        raise ValueError(f"unknown scale distribution {dist!r}")
    return v.astype(np.float16)


def float_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(v, dtype=np.float32))
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = r.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def activations(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """bf16 activations as uint16 bit patterns, rounded from N(0, std^2)."""
    g = rng(seed, name)
    return float_to_bf16_bits(g.normal(0.0, std, size=shape).astype(np.float32))


def signs(seed: int, name: str, n: int) -> np.ndarray:
    """int8 vector of iid uniform +-1."""
    g = rng(seed, name)
    return np.where(g.random(n) < 0.5, -1, 1).astype(np.int8)


@dataclass
class Problem:
    """One seeded product problem: y = x W^T with W given by (t, s)."""
    M: int
    N: int
    K: int
    t: np.ndarray          # int8 [N, K]
    s: np.ndarray          # float16 [N, K/128]
    x: np.ndarray          # uint16 bf16 bits [M, K]
    signs: np.ndarray | None = None   # int8 [K] (rotation problems only)


def problem(seed: int, M: int, N: int, K: int, trit_dist: str = SPARSE40,
            scale_dist: str = SCALE_HALFNORMAL, with_signs: bool = False,
            tag: str = "") -> Problem:
    """A seeded problem of the given shape; `tag` separates problems of one seed."""
    t = trits(seed, f"{tag}t", (N, K), trit_dist)
    s = scales(seed, f"{tag}s", (N, K // 128), scale_dist)
    x = activations(seed, f"{tag}x", (M, K))
    sg = signs(seed, f"{tag}signs", K) if with_signs else None
    return Problem(M, N, K, t, s, x, sg)


# The workloads (shapes and distributions) used by the tests and the benchmark.
TINY = dict(M=1, K=512, N=256, trit_dist=UNIFORM, scale_dist=SCALE_UNIFORM, seed=0)
DECODE_SHAPES = [(5120, 17408), (17408, 5120)]          # (K, N): gate/up, down
VERIFY_M = [1, 2, 4, 5, 8, 16]
VERIFY_STEP_M = 5                                         # draft depth k = 4, plus one
VERIFY_SHAPES = [(5120, 17408), (5120, 6144)]
ROTATED = dict(K=4096, N=12288, M=(1, 16))
PREFILL_M = 512
PREFILL_LAYER = [("gate", 5120, 17408), ("up", 5120, 17408), ("qkv", 5120, 6144),
                 ("down", 17408, 5120)]                   # (name, K, N)
PREFILL_LAYERS = 64


# ---------------------------------------------------------------------------
# Device-side draws for the benchmark's multi-gigabyte weight sets (torch's
# seeded CUDA generator; same distributions as above, not the same values).
# ---------------------------------------------------------------------------

def device_generator(seed: int, name: str, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 32) ^ zlib.crc32(name.encode("utf-8")))
    return g


def device_trits(seed: int, name: str, shape, dist: str = SPARSE40, device="cuda"):
    """int8 CUDA tensor of iid trits."""
    import torch
    g = device_generator(seed, name, device)
    u = torch.rand(shape, generator=g, device=device)
    lo, hi = (1.0 / 3.0, 2.0 / 3.0) if dist == UNIFORM else (0.3, 0.7)
    t = (u >= lo).to(torch.int8)
    t += (u >= hi).to(torch.int8)
    t -= 1
    return t


def device_binary(seed: int, name: str, shape, device="cuda"):
    """int8 CUDA tensor of iid weights in {-1, +1} (the 1-bit format), P = 1/2."""
    import torch
    g = device_generator(seed, name, device)
    return torch.where(torch.rand(shape, generator=g, device=device) < 0.5, -1, 1).to(torch.int8)


def device_code_words(seed: int, name: str, shape, device="cuda"):
    """int32 CUDA tensor of iid random words (an affine pack's codes, every
    2-bit slot uniform over 0..3)."""
    import torch
    g = device_generator(seed, name, device)
    return torch.randint(-(1 << 31), 1 << 31, shape, generator=g, device=device, dtype=torch.int32)


def device_biases(seed: int, name: str, s, device="cuda"):
    """fp16 CUDA tensor b = -u s, u ~ U[1, 2] iid, for fp16 scales s."""
    import torch
    g = device_generator(seed, name, device)
    u = torch.rand(s.shape, generator=g, device=device) + 1.0
    return (-u * s.float()).to(torch.float16)


def device_scales(seed: int, name: str, shape, dist: str = SCALE_HALFNORMAL, device="cuda"):
    import torch
    g = device_generator(seed, name, device)
    if dist == SCALE_UNIFORM:
        v = torch.rand(shape, generator=g, device=device) * 0.045 + 0.005
    else:
        v = torch.randn(shape, generator=g, device=device).abs_() * 0.02 + 1e-3
    return v.to(torch.float16)


def device_activations(seed: int, name: str, shape, device="cuda"):
    import torch
    g = device_generator(seed, name, device)
    return torch.randn(shape, generator=g, device=device).to(torch.bfloat16)


def device_signs(seed: int, name: str, n: int, device="cuda"):
    import torch
    g = device_generator(seed, name, device)
    return torch.where(torch.rand(n, generator=g, device=device) < 0.5, -1, 1).to(torch.int8)
