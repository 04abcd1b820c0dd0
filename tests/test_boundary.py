"""The product path's boundary without a GPU: the binding fails loudly when
the CUDA library is missing (there is no fallback), and nothing on the
product side reaches the oracle."""
import ast
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bit_gemv_gemm_gb300")


def test_binding_fails_loudly_without_the_library(monkeypatch):
    import bit_gemv_gemm_gb300 as t
    monkeypatch.setattr(t, "_lib", None)
    monkeypatch.setattr(t, "LIB_PATH", os.path.join(ROOT, "no-such-dir", "libtern.so"))
    with pytest.raises(RuntimeError, match="not built"):
        t.lib()
    with pytest.raises(RuntimeError, match="not built"):
        t.packed_bytes(16, 128)


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module


def test_product_side_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                for mod in _imports(os.path.join(dirpath, f)):
                    assert not mod.split(".")[0] == "oracle", (f, mod)
    for f in os.listdir(os.path.join(PKG, "csrc")):
        src = open(os.path.join(PKG, "csrc", f)).read()
        assert "oracle" not in src.lower(), f


def test_library_links_no_oracle_code():
    from bit_gemv_gemm_gb300 import build
    lib = build.build()
    out = subprocess.run(["readelf", "-d", lib], capture_output=True, text=True).stdout
    needed = [l for l in out.splitlines() if "NEEDED" in l]
    assert needed and not any("orc" in l for l in needed), needed
    syms = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True).stdout
    assert " orc_" not in syms and "tern_gemv" in syms


def test_binding_refuses_tensors_shorter_than_the_call_needs():
    """A short tensor is refused before any pointer reaches the library (CPU
    tensors: the coverage check comes before the device check)."""
    import torch
    import bit_gemv_gemm_gb300 as t
    M, N, K = 2, 8, 256
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    codes = torch.zeros((N, K // 16), dtype=torch.int32)
    words = torch.zeros((N, K // 32), dtype=torch.int32)
    s = torch.zeros((N, K // 128), dtype=torch.float16)
    with pytest.raises(ValueError, match="codes"):
        t.gemv(x, codes[:, :-1].contiguous(), s)                  # one word short per row
    with pytest.raises(ValueError, match="scales"):
        t.gemv(x, codes, s[:-1])
    with pytest.raises(ValueError, match="y"):
        t.gemv(x, codes, s, y=torch.zeros((M, N - 1)))
    with pytest.raises(ValueError, match="words"):
        t.bin_gemv(x, torch.zeros((N, K // 32 - 1), dtype=torch.int32), s)
    with pytest.raises(ValueError, match="biases"):
        t.affine_gemv(x, codes, s, s[:-1])
    with pytest.raises(ValueError, match="biases"):
        t.affine_gemm(x, codes, s, s[:-1])
    with pytest.raises(ValueError, match="scales"):
        t.gemm(x, codes, s[:-1])
    with pytest.raises(ValueError, match="y_b"):
        t.gemv_pair(x, codes, s, codes, s, y_b=torch.zeros((M, N - 1)))
    with pytest.raises(ValueError, match="signs"):
        t.fwht(torch.zeros((1, 4096), dtype=torch.bfloat16), torch.zeros(4095, dtype=torch.int8))
    with pytest.raises(ValueError, match="codes"):
        t.pack(torch.zeros((N, K), dtype=torch.int8), codes=codes[:-1])
    # full-size CPU tensors pass the coverage check and stop at the device check
    with pytest.raises(TypeError, match="CUDA"):
        t.gemv(x, codes, s, y=torch.zeros((M, N)), ws=torch.zeros(256, dtype=torch.uint8))
