"""CPU oracle for the ternary-g128 matrix product and the Hadamard rotation.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs may import this package.  The CUDA library does
not use it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
compiles it with gcc and exposes numpy-level wrappers.  Every function follows
the definitions on the "prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card
("Weight representation: ternary g128", "Memory requirement", "MLX packaging")
and the "Ternary-Bonsai-2-9B-2bit" article (section 3, "Ternary weights and
Hadamard rotation"); see the header of ``oracle.c`` for the readings taken.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP) and return its path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sig = {
                "orc_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_pack": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_unpack": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_matmul": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _I]),
                "orc_matmul_sampled": (_I, [_P, _P, _P, _I, _P, _P, _I, _P, _P, _I]),
                "orc_bin_pack": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_f3_pack": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_f3_unpack": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_f3_matmul": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _I]),
                "orc_bin_unpack": (_I, [_P, _I, _I, _P]),
                "orc_bin_matmul": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _I]),
                "orc_bin_matmul_sampled": (_I, [_P, _P, _P, _I, _P, _P, _I, _P, _P, _I]),
                "orc_scales_from_g64": (ctypes.c_longlong, [_P, _I, _I, _P]),
                "orc_mlx_affine": (ctypes.c_float, [_I, ctypes.c_float, ctypes.c_float]),
                "orc_affine_matmul": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _I]),
                "orc_affine_matmul_sampled": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _P, _P, _I]),
                "orc_hadamard_explicit": (_I, [_I, _P]),
                "orc_fwht": (_I, [_P, _I]),
                "orc_rotate": (_I, [_P, _P, _I, _I, _I, _P]),
                "orc_unrotate": (_I, [_P, _P, _I, _I, _I, _P]),
                "orc_rotate_matmul": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I]),
                "orc_max_threads": (_I, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().orc_max_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().orc_bf16_to_f64(int(bits)))


def f16_to_f64(bits: int) -> float:
    return float(_load().orc_f16_to_f64(int(bits)))


def pack(t: np.ndarray) -> tuple[np.ndarray, int]:
    """t int8 [N, K] in {-1,0,1} -> (codes uint32 [N, K/16], invalid count)."""
    t = _c(t, np.int8)
    N, K = t.shape
    codes = np.empty((N, K // 16), dtype=np.uint32)
    bad = _load().orc_pack(_ptr(t), N, K, _ptr(codes))
    if bad < 0:
        raise ValueError("K must be a multiple of 16")
    return codes, int(bad)


def unpack(codes: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """codes uint32 [N, K/16] -> (t int8 [N, K], count of invalid code 3)."""
    codes = _c(codes, np.uint32)
    N = codes.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    bad = _load().orc_unpack(_ptr(codes), N, K, _ptr(t))
    if bad < 0:
        raise ValueError("K must be a multiple of 16")
    return t, int(bad)


def bin_pack(t: np.ndarray) -> tuple[np.ndarray, int]:
    """The 1-bit sibling: t int8 [N, K] in {-1, +1} -> (words uint32 [N, K/32],
    count of entries that are not +-1)."""
    t = _c(t, np.int8)
    N, K = t.shape
    words = np.empty((N, K // 32), dtype=np.uint32)
    bad = _load().orc_bin_pack(_ptr(t), N, K, _ptr(words))
    if bad < 0:
        raise ValueError("K must be a multiple of 32")
    return words, int(bad)


def bin_unpack(words: np.ndarray, K: int) -> np.ndarray:
    """words uint32 [N, K/32] -> t int8 [N, K] = 2b - 1."""
    words = _c(words, np.uint32)
    N = words.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    if _load().orc_bin_unpack(_ptr(words), N, K, _ptr(t)) != 0:
        raise ValueError("K must be a multiple of 32")
    return t


def bin_matmul(x_bf16: np.ndarray, words: np.ndarray, scales_f16: np.ndarray,
               nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """y[m, n] = sum_k x[m, k] (2 b[n, k] - 1) s[n, k // 128] in double, and the
    error scale a = sum_k |x w|; returns (y, a)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    words = _c(words, np.uint32)
    M, K = x.shape
    N = words.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    if _load().orc_bin_matmul(_ptr(x), _ptr(words), _ptr(s), M, N, K, _ptr(y), _ptr(a), nthreads) != 0:
        raise ValueError("bad shape")
    return y, a


def bin_matmul_sampled(x_bf16: np.ndarray, words: np.ndarray, scales_f16: np.ndarray,
                       ms: np.ndarray, ns: np.ndarray, nthreads: int = 0):
    """The binary product at outputs (ms[i], ns[i]) only; returns (y, a)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    words = _c(words, np.uint32)
    K = x.shape[1]
    ms = _c(ms, np.int32)
    ns = _c(ns, np.int32)
    y = np.empty(len(ms), dtype=np.float64)
    a = np.empty(len(ms), dtype=np.float64)
    if _load().orc_bin_matmul_sampled(_ptr(x), _ptr(words), _ptr(s), K, _ptr(ms), _ptr(ns), len(ms),
                                      _ptr(y), _ptr(a), nthreads) != 0:
        raise ValueError("bad shape")
    return y, a


def f3_pack(t: np.ndarray) -> tuple[np.ndarray, int]:
    """Native base-3 packing: t int8 [N, K] in {-1,0,1} -> (bytes uint8
    [N, 26 K/128], count of entries outside {-1,0,1}).  Five trits per byte,
    byte = q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4 with q = t + 1; the 26th byte of a
    group holds trits 125..127."""
    t = _c(t, np.int8)
    N, K = t.shape
    out = np.empty((N, 26 * (K // 128)), dtype=np.uint8)
    bad = _load().orc_f3_pack(_ptr(t), N, K, _ptr(out))
    if bad < 0:
        raise ValueError("K must be a multiple of 128")
    return out, int(bad)


def f3_unpack(packed: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """bytes uint8 [N, 26 K/128] -> (t int8 [N, K], count of out-of-range bytes)."""
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    bad = _load().orc_f3_unpack(_ptr(packed), N, K, _ptr(t))
    if bad < 0:
        raise ValueError("K must be a multiple of 128")
    return t, int(bad)


def f3_matmul(x_bf16: np.ndarray, packed: np.ndarray, scales_f16: np.ndarray,
              nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """y[m, n] = sum_k x[m, k] (q[n, k] - 1) s[n, k // 128] in double from the
    base-3 bytes, and a = sum_k |x w|; returns (y, a)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    packed = _c(packed, np.uint8)
    M, K = x.shape
    N = packed.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    if _load().orc_f3_matmul(_ptr(x), _ptr(packed), _ptr(s), M, N, K, _ptr(y), _ptr(a), nthreads) != 0:
        raise ValueError("bad shape")
    return y, a


def scales_from_g64(s64: np.ndarray) -> tuple[np.ndarray, int]:
    """fp16 scales [N, K/64] of the group-size-64 pack -> ([N, K/128], count of
    groups whose two halves differ)."""
    s64 = _bits16(np.ascontiguousarray(s64))
    N, G2 = s64.shape
    out = np.empty((N, G2 // 2), dtype=np.uint16)
    bad = _load().orc_scales_from_g64(_ptr(s64), N, G2 * 64, _ptr(out))
    if bad < 0:
        raise ValueError("K must be a multiple of 128")
    return out.view(np.float16), int(bad)


def _bits16(a: np.ndarray) -> np.ndarray:
    return _c(a.view(np.uint16) if a.dtype != np.uint16 else a, np.uint16)


def matmul(x_bf16: np.ndarray, codes: np.ndarray, scales_f16: np.ndarray,
           K: int | None = None, nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """y[m, n] = sum_k x[m, k] (q[n, k] - 1) s[n, k // 128] in double.

    x_bf16: uint16 bf16 bit patterns [M, K]; codes uint32 [N, K/16];
    scales_f16: float16 (or its uint16 bits) [N, K/128].
    Returns (y, a) with a = sum_k |x w| (the error scale)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    codes = _c(codes, np.uint32)
    M, Kx = x.shape
    K = Kx if K is None else K
    N = codes.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    st = _load().orc_matmul(_ptr(x), _ptr(codes), _ptr(s), M, N, K, _ptr(y), _ptr(a), nthreads)
    if st == -1:
        raise ValueError("invalid code 3 in codes")
    if st != 0:
        raise ValueError("bad shape")
    return y, a


def matmul_sampled(x_bf16: np.ndarray, codes: np.ndarray, scales_f16: np.ndarray,
                   ms: np.ndarray, ns: np.ndarray, nthreads: int = 0):
    """The product at outputs (ms[i], ns[i]) only; returns (y, a) of length len(ms)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    codes = _c(codes, np.uint32)
    K = x.shape[1]
    ms = _c(ms, np.int32)
    ns = _c(ns, np.int32)
    y = np.empty(len(ms), dtype=np.float64)
    a = np.empty(len(ms), dtype=np.float64)
    st = _load().orc_matmul_sampled(_ptr(x), _ptr(codes), _ptr(s), K, _ptr(ms), _ptr(ns),
                                    len(ms), _ptr(y), _ptr(a), nthreads)
    if st == -1:
        raise ValueError("invalid code 3 in codes")
    if st != 0:
        raise ValueError("bad shape")
    return y, a


def affine_matmul(x_bf16: np.ndarray, codes: np.ndarray, scales_f16: np.ndarray, biases_f16: np.ndarray,
                  nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """The affine pack's product: y[m, n] = sum_k x[m, k] (s q[n, k] + b)[n, k // 128]
    in double, every code 0..3 valid; returns (y, a) with a = sum_k |x w|."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    b = _bits16(biases_f16)
    codes = _c(codes, np.uint32)
    M, K = x.shape
    N = codes.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    if _load().orc_affine_matmul(_ptr(x), _ptr(codes), _ptr(s), _ptr(b), M, N, K, _ptr(y), _ptr(a),
                                 nthreads) != 0:
        raise ValueError("bad shape")
    return y, a


def affine_matmul_sampled(x_bf16: np.ndarray, codes: np.ndarray, scales_f16: np.ndarray,
                          biases_f16: np.ndarray, ms: np.ndarray, ns: np.ndarray, nthreads: int = 0):
    """The affine product at outputs (ms[i], ns[i]) only; returns (y, a)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    b = _bits16(biases_f16)
    codes = _c(codes, np.uint32)
    K = x.shape[1]
    ms = _c(ms, np.int32)
    ns = _c(ns, np.int32)
    y = np.empty(len(ms), dtype=np.float64)
    a = np.empty(len(ms), dtype=np.float64)
    if _load().orc_affine_matmul_sampled(_ptr(x), _ptr(codes), _ptr(s), _ptr(b), K, _ptr(ms), _ptr(ns),
                                         len(ms), _ptr(y), _ptr(a), nthreads) != 0:
        raise ValueError("bad shape")
    return y, a


def mlx_affine(q: int, s_mlx: float, bias: float) -> float:
    """MLX affine dequantisation of one code in float32: s_mlx * q + bias."""
    return float(_load().orc_mlx_affine(int(q), float(s_mlx), float(bias)))


def hadamard_explicit(n: int) -> np.ndarray:
    """The n x n Sylvester Hadamard matrix (unnormalized), by recursion."""
    H = np.empty((n, n), dtype=np.float64)
    if _load().orc_hadamard_explicit(n, _ptr(H)) != 0:
        raise ValueError("n must be a power of two")
    return H


def fwht(v: np.ndarray) -> np.ndarray:
    """Unnormalized fast Walsh-Hadamard transform (natural order) of a vector."""
    v = np.array(v, dtype=np.float64, copy=True)
    if _load().orc_fwht(_ptr(v), v.shape[0]) != 0:
        raise ValueError("length must be a power of two")
    return v


def rotate(x_bf16: np.ndarray, signs: np.ndarray, block: int = 4096) -> np.ndarray:
    """x' = H_B (s * x) / sqrt(B) per block of the last dimension, in double."""
    x = _bits16(x_bf16)
    signs = _c(signs, np.int8)
    M, K = x.shape
    out = np.empty((M, K), dtype=np.float64)
    if _load().orc_rotate(_ptr(x), _ptr(signs), M, K, block, _ptr(out)) != 0:
        raise ValueError("bad block size")
    return out


def unrotate(xr: np.ndarray, signs: np.ndarray, block: int = 4096) -> np.ndarray:
    """The inverse rotation x = s * (H_B x' / sqrt(B))."""
    xr = _c(xr, np.float64)
    signs = _c(signs, np.int8)
    M, K = xr.shape
    out = np.empty((M, K), dtype=np.float64)
    if _load().orc_unrotate(_ptr(xr), _ptr(signs), M, K, block, _ptr(out)) != 0:
        raise ValueError("bad block size")
    return out


def rotate_matmul(x_bf16: np.ndarray, signs: np.ndarray, codes: np.ndarray,
                  scales_f16: np.ndarray, block: int = 4096, nthreads: int = 0):
    """y = rotate(x) W^T with the rotated activation kept in double; returns (y, a)."""
    x = _bits16(x_bf16)
    s = _bits16(scales_f16)
    signs = _c(signs, np.int8)
    codes = _c(codes, np.uint32)
    M, K = x.shape
    N = codes.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    st = _load().orc_rotate_matmul(_ptr(x), _ptr(signs), _ptr(codes), _ptr(s), M, N, K, block,
                                   _ptr(y), _ptr(a), nthreads)
    if st == -1:
        raise ValueError("invalid code 3 in codes")
    if st != 0:
        raise ValueError("bad shape")
    return y, a
