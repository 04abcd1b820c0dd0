"""bit_gemv_gemm_gb300 -- Python binding of libtern (GB300 ternary-g128 product).

A thin ctypes layer over the C ABI in ``include/tern.h``: it checks tensor
types, passes ``data_ptr()`` and the current CUDA stream, and turns status codes
into exceptions.  Every step of the computation runs in the library's CUDA
kernels; PyTorch only allocates device memory and supplies streams.  There is
no fallback: if the library is not built, or the device is not an sm_103 GPU,
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtern.so")

TERN_OK = 0
_STATUS = {0: "ok", 1: "null pointer", 2: "bad shape", 3: "misaligned pointer", 4: "workspace too small",
           5: "CUDA error", 6: "device is not sm_103", 7: "device-side error"}

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_LL = ctypes.c_longlong

EXPORTS = {
    "tern_status_str": (ctypes.c_char_p, [_I]),
    "tern_packed_bytes": (_SZ, [_I, _I]),
    "tern_pack": (_I, [_P, _I, _I, _P, _P, _P]),
    "tern_pack_host": (_I, [_P, _I, _I, _P, _P]),
    "tern_unpack_host": (_I, [_P, _I, _I, _P, _P]),
    "tern_validate_host": (_I, [_P, _I, _I, _P]),
    "tern_gemv_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tern_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "tern_fwht": (_I, [_P, _P, _P, _I, _I, _P]),
    "tern_fwht_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "tern_gemm_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tern_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "tern_device_error": (_I, [_P]),
    "tern_last_launch_count": (_I, []),
    "tern_gemv_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "tern_gemv_pair_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "tern_gemv_pair": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "tern_wait_selftest": (_I, [_I, _I, _P]),
    "tern_bin_packed_bytes": (_SZ, [_I, _I]),
    "tern_scales_from_g64": (_I, [_P, _I, _I, _P, _P, _P]),
    "tern_scales_from_g64_host": (_I, [_P, _I, _I, _P, _P]),
    "tern_bin_pack": (_I, [_P, _I, _I, _P, _P, _P]),
    "tern_bin_pack_host": (_I, [_P, _I, _I, _P, _P]),
    "tern_bin_unpack_host": (_I, [_P, _I, _I, _P]),
    "tern_bin_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "tern_bin_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "tern_affine_gemv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "tern_affine_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "tern_f3_packed_bytes": (_SZ, [_I, _I]),
    "tern_f3_pack": (_I, [_P, _I, _I, _P, _P, _P]),
    "tern_f3_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
}


class TernError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown')} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libtern.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtern.so is not built ({LIB_PATH}); run "
                                   "`python -m bit_gemv_gemm_gb300.build` or __graft_entry__.build()")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def _check(fn: str, st: int) -> None:
    if st != TERN_OK:
        raise TernError(fn, st)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _covers(**need) -> None:
    """name=(tensor, elements): each tensor must hold at least the elements the
    call reads or writes through its pointer (the library sees only pointers
    and sizes, so a short tensor would be read or written past its end)."""
    for name, (t, n) in need.items():
        if t is not None and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements; the call needs {n}")


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------

def packed_bytes(N: int, K: int) -> int:
    return int(lib().tern_packed_bytes(N, K))


def gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().tern_gemv_workspace_bytes(M, N, K))


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().tern_gemm_workspace_bytes(M, N, K))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device byte buffer usable as a libtern workspace (torch's
    allocations are 256-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------
# packing
# ---------------------------------------------------------------------------

def pack(t: torch.Tensor, codes: torch.Tensor | None = None, bad_count: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """Device packer: int8 trits [N, K] -> uint32 codes [N, K/16] (as int32 storage).

    If ``bad_count`` (int32 CUDA tensor of one element) is given, the number of
    entries outside {-1, 0, +1} is added to it."""
    N, K = t.shape
    if codes is None:
        codes = torch.empty((N, K // 16), dtype=torch.int32, device=t.device)
    _covers(codes=(codes, N * (K // 16)), bad_count=(bad_count, 1))
    bp = _dev(bad_count, torch.int32, "bad_count") if bad_count is not None else None
    _check("tern_pack", lib().tern_pack(_dev(t, torch.int8, "t"), N, K, _dev(codes, torch.int32, "codes"),
                                        bp, _stream(stream)))
    return codes


def scales_from_g64(s64: torch.Tensor, K: int, mismatch: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Scales of the group-size-64 pack (fp16 [N, K/64], each g128 scale
    repeated) -> g128 scales fp16 [N, K/128]; differing halves are counted."""
    N = s64.shape[0]
    out = torch.empty((N, K // 128), dtype=torch.float16, device=s64.device)
    _covers(s64=(s64, N * (K // 64)), mismatch=(mismatch, 1))
    mp = _dev(mismatch, torch.int32, "mismatch") if mismatch is not None else None
    _check("tern_scales_from_g64", lib().tern_scales_from_g64(_dev(s64, torch.float16, "s64"), N, K,
                                                              _dev(out, torch.float16, "s128"), mp, _stream(stream)))
    return out


def scales_from_g64_host(s64: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    s64 = np.ascontiguousarray(s64, dtype=np.float16)
    N = s64.shape[0]
    out = np.empty((N, K // 128), dtype=np.float16)
    bad = ctypes.c_longlong(0)
    _check("tern_scales_from_g64_host", lib().tern_scales_from_g64_host(s64.ctypes.data, N, K, out.ctypes.data,
                                                                        ctypes.byref(bad)))
    return out, int(bad.value)


def bin_pack(t: torch.Tensor, words: torch.Tensor | None = None, bad_count: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """Device packer of the 1-bit format: int8 [N, K] in {-1, +1} -> uint32
    words [N, K/32] (as int32 storage), bit k%32 of word k/32 set for +1."""
    N, K = t.shape
    if words is None:
        words = torch.empty((N, K // 32), dtype=torch.int32, device=t.device)
    _covers(words=(words, N * (K // 32)), bad_count=(bad_count, 1))
    bp = _dev(bad_count, torch.int32, "bad_count") if bad_count is not None else None
    _check("tern_bin_pack", lib().tern_bin_pack(_dev(t, torch.int8, "t"), N, K, _dev(words, torch.int32, "words"),
                                                bp, _stream(stream)))
    return words


def f3_pack(t: torch.Tensor, packed: torch.Tensor | None = None, bad_count: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Device packer of the base-3 format: int8 [N, K] in {-1, 0, +1} -> uint8
    [N, 26 K/128], five trits per byte (q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4)."""
    N, K = t.shape
    nbytes = int(lib().tern_f3_packed_bytes(N, K))
    if packed is None:
        packed = torch.empty((N, 26 * (K // 128)), dtype=torch.uint8, device=t.device)
    _covers(packed=(packed, nbytes), bad_count=(bad_count, 1))
    bp = _dev(bad_count, torch.int32, "bad_count") if bad_count is not None else None
    _check("tern_f3_pack", lib().tern_f3_pack(_dev(t, torch.int8, "t"), N, K, _dev(packed, torch.uint8, "packed"),
                                              bp, _stream(stream)))
    return packed


def f3_gemv(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """y (fp32 [M, N]) = x W^T on a base-3 pack, M = 1..16; x bf16 [M, K],
    packed uint8 [N, 26 K/128], scales fp16 [N, K/128].  No workspace."""
    M, K = x.shape
    N = packed.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(packed=(packed, N * 26 * (K // 128)), scales=(scales, N * (K // 128)), y=(y, M * N))
    _check("tern_f3_gemv", lib().tern_f3_gemv(
        _dev(x, torch.bfloat16, "x"), _dev(packed, torch.uint8, "packed"), _dev(scales, torch.float16, "scales"),
        _dev(y, torch.float32, "y"), M, N, K, _stream(stream)))
    return y


def bin_pack_host(t: np.ndarray) -> tuple[np.ndarray, int]:
    t = np.ascontiguousarray(t, dtype=np.int8)
    N, K = t.shape
    words = np.empty((N, K // 32), dtype=np.uint32)
    bad = ctypes.c_longlong(0)
    _check("tern_bin_pack_host", lib().tern_bin_pack_host(t.ctypes.data, N, K, words.ctypes.data,
                                                          ctypes.byref(bad)))
    return words, int(bad.value)


def bin_unpack_host(words: np.ndarray, K: int) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    N = words.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    _check("tern_bin_unpack_host", lib().tern_bin_unpack_host(words.ctypes.data, N, K, t.ctypes.data))
    return t


def pack_host(t: np.ndarray) -> tuple[np.ndarray, int]:
    t = np.ascontiguousarray(t, dtype=np.int8)
    N, K = t.shape
    codes = np.empty((N, K // 16), dtype=np.uint32)
    bad = ctypes.c_longlong(0)
    _check("tern_pack_host", lib().tern_pack_host(t.ctypes.data, N, K, codes.ctypes.data, ctypes.byref(bad)))
    return codes, int(bad.value)


def unpack_host(codes: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    N = codes.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    bad = ctypes.c_longlong(0)
    _check("tern_unpack_host", lib().tern_unpack_host(codes.ctypes.data, N, K, t.ctypes.data, ctypes.byref(bad)))
    return t, int(bad.value)


def validate_host(codes: np.ndarray, K: int) -> int:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    bad = ctypes.c_longlong(0)
    _check("tern_validate_host", lib().tern_validate_host(codes.ctypes.data, codes.shape[0], K, ctypes.byref(bad)))
    return int(bad.value)


# ---------------------------------------------------------------------------
# products and rotation
# ---------------------------------------------------------------------------

def gemv(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
         ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y (fp32 [M, N]) = x W^T for M = 1..16; x bf16 [M, K], codes int32 [N, K/16], scales fp16 [N, K/128]."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), y=(y, M * N))
    if ws is None:
        ws = workspace(gemv_workspace_bytes(M, N, K), x.device)
    _check("tern_gemv", lib().tern_gemv(
        _dev(x, torch.bfloat16, "x"), _dev(codes, torch.int32, "codes"), _dev(scales, torch.float16, "scales"),
        _dev(y, torch.float32, "y"), M, N, K, _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def bin_gemv(x: torch.Tensor, words: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
             ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The 1-bit sibling: y (fp32 [M, N]) = x W^T for M = 1..16, W = (2b - 1) s;
    x bf16 [M, K], words int32 [N, K/32], scales fp16 [N, K/128]."""
    M, K = x.shape
    N = words.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(words=(words, N * (K // 32)), scales=(scales, N * (K // 128)), y=(y, M * N))
    if ws is None:
        ws = workspace(gemv_workspace_bytes(M, N, K), x.device)
    _check("tern_bin_gemv", lib().tern_bin_gemv(
        _dev(x, torch.bfloat16, "x"), _dev(words, torch.int32, "words"), _dev(scales, torch.float16, "scales"),
        _dev(y, torch.float32, "y"), M, N, K, _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def gemv_pair(x: torch.Tensor, codes_a: torch.Tensor, scales_a: torch.Tensor, codes_b: torch.Tensor,
              scales_b: torch.Tensor, y_a: torch.Tensor | None = None, y_b: torch.Tensor | None = None,
              ws: torch.Tensor | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Two products of the same activation in one launch: (x W_a^T, x W_b^T)."""
    M, K = x.shape
    Na, Nb = codes_a.shape[0], codes_b.shape[0]
    if y_a is None:
        y_a = torch.empty((M, Na), dtype=torch.float32, device=x.device)
    if y_b is None:
        y_b = torch.empty((M, Nb), dtype=torch.float32, device=x.device)
    _covers(codes_a=(codes_a, Na * (K // 16)), scales_a=(scales_a, Na * (K // 128)), y_a=(y_a, M * Na),
            codes_b=(codes_b, Nb * (K // 16)), scales_b=(scales_b, Nb * (K // 128)), y_b=(y_b, M * Nb))
    if ws is None:
        ws = workspace(int(lib().tern_gemv_pair_workspace_bytes(M, Na, Nb, K)), x.device)
    _check("tern_gemv_pair", lib().tern_gemv_pair(
        _dev(x, torch.bfloat16, "x"), _dev(codes_a, torch.int32, "codes_a"), _dev(scales_a, torch.float16, "scales_a"),
        _dev(y_a, torch.float32, "y_a"), Na, _dev(codes_b, torch.int32, "codes_b"),
        _dev(scales_b, torch.float16, "scales_b"), _dev(y_b, torch.float32, "y_b"), Nb, M, K,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y_a, y_b


def gemv_noalloc(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """tern_gemv without a workspace: the library's fixed scratch array is used."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), y=(y, M * N))
    _check("tern_gemv_noalloc", lib().tern_gemv_noalloc(
        _dev(x, torch.bfloat16, "x"), _dev(codes, torch.int32, "codes"), _dev(scales, torch.float16, "scales"),
        _dev(y, torch.float32, "y"), M, N, K, _stream(stream)))
    return y


def fwht(x: torch.Tensor, signs: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y (bf16 [M, K]) = H_4096 (signs * x) / 64 per 4096-block of the last dimension."""
    M, K = x.shape
    if y is None:
        y = torch.empty_like(x)
    _covers(signs=(signs, K), y=(y, M * K))
    _check("tern_fwht", lib().tern_fwht(_dev(x, torch.bfloat16, "x"), _dev(signs, torch.int8, "signs"),
                                        _dev(y, torch.bfloat16, "y"), M, K, _stream(stream)))
    return y


def fwht_gemm(x: torch.Tensor, signs: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
              y: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y (fp32 [M, N]) = rotate(x) W^T with the rotation fused into the product's prologue."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(signs=(signs, K), codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), y=(y, M * N))
    if ws is None:
        ws = workspace(gemv_workspace_bytes(M, N, K), x.device)
    _check("tern_fwht_gemm", lib().tern_fwht_gemm(
        _dev(x, torch.bfloat16, "x"), _dev(signs, torch.int8, "signs"), _dev(codes, torch.int32, "codes"),
        _dev(scales, torch.float16, "scales"), _dev(y, torch.float32, "y"), M, N, K,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def gemm(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
         out_dtype=torch.float32, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y ([M, N], fp32 or bf16) = x W^T on the tcgen05 tensor cores, any M >= 1."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    _covers(codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), y=(y, M * N))
    if ws is None:
        ws = workspace(gemm_workspace_bytes(M, N, K), x.device)
    _check("tern_gemm", lib().tern_gemm(
        _dev(x, torch.bfloat16, "x"), _dev(codes, torch.int32, "codes"), _dev(scales, torch.float16, "scales"),
        _dev(y, y.dtype, "y"), 1 if y.dtype == torch.bfloat16 else 0, M, N, K,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def device_error() -> int:
    """Reads and clears the device-side error word (synchronizes the device)."""
    code = ctypes.c_int(0)
    _check("tern_device_error", lib().tern_device_error(ctypes.byref(code)))
    return int(code.value)


SELFTEST_RANGE_FLAG, SELFTEST_MBARRIER = 0, 1
DEVERR_GEMM_MMA_WAIT, DEVERR_GEMV_RANGE_FLAG_WAIT, DEVERR_GEMV_ACTIVATION_RANGE = 0x103, 0x202, 0x203


def wait_selftest(which: int, limit_us: int, stream=None) -> None:
    """Runs one bounded wait on something nothing completes (tern_wait_selftest);
    the code it reports is read with device_error()."""
    _check("tern_wait_selftest", lib().tern_wait_selftest(which, limit_us, _stream(stream)))


def last_launch_count() -> int:
    return int(lib().tern_last_launch_count())


def bin_gemm(x: torch.Tensor, words: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
             out_dtype=torch.float32, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The 1-bit sibling format on the tcgen05 tensor cores: y ([M, N], fp32 or
    bf16) = x W^T, W = (2b - 1) s, any M >= 1."""
    M, K = x.shape
    N = words.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    _covers(words=(words, N * (K // 32)), scales=(scales, N * (K // 128)), y=(y, M * N))
    if ws is None:
        ws = workspace(gemm_workspace_bytes(M, N, K), x.device)
    _check("tern_bin_gemm", lib().tern_bin_gemm(
        _dev(x, torch.bfloat16, "x"), _dev(words, torch.int32, "words"), _dev(scales, torch.float16, "scales"),
        _dev(y, y.dtype, "y"), 1 if y.dtype == torch.bfloat16 else 0, M, N, K,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def affine_gemv(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                y: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """An affine pack: y (fp32 [M, N]) = x W^T for M = 1..16, W = s q + b per
    group of 128; x bf16 [M, K], codes int32 [N, K/16] (every code 0..3),
    scales and biases fp16 [N, K/128]."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _covers(codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), biases=(biases, N * (K // 128)),
            y=(y, M * N))
    if ws is None:
        ws = workspace(gemv_workspace_bytes(M, N, K), x.device)
    _check("tern_affine_gemv", lib().tern_affine_gemv(
        _dev(x, torch.bfloat16, "x"), _dev(codes, torch.int32, "codes"), _dev(scales, torch.float16, "scales"),
        _dev(biases, torch.float16, "biases"), _dev(y, torch.float32, "y"), M, N, K,
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y


def affine_gemm(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                y: torch.Tensor | None = None, out_dtype=torch.float32, ws: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """An affine pack on the tcgen05 tensor cores: y ([M, N], fp32 or bf16) =
    x W^T, W = s q + b per group of 128, any M >= 1."""
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    _covers(codes=(codes, N * (K // 16)), scales=(scales, N * (K // 128)), biases=(biases, N * (K // 128)),
            y=(y, M * N))
    if ws is None:
        ws = workspace(gemm_workspace_bytes(M, N, K), x.device)
    _check("tern_affine_gemm", lib().tern_affine_gemm(
        _dev(x, torch.bfloat16, "x"), _dev(codes, torch.int32, "codes"), _dev(scales, torch.float16, "scales"),
        _dev(biases, torch.float16, "biases"), _dev(y, y.dtype, "y"), 1 if y.dtype == torch.bfloat16 else 0,
        M, N, K, _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
    return y
