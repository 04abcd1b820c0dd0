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
