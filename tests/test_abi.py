"""The C ABI without a GPU: the library loads, exports every declared entry
point, validates arguments before touching the device, and its host packer,
unpacker and validator agree bit for bit with the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tern():
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "tern.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tern_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("tern_pack", "tern_gemv", "tern_gemm", "tern_fwht", "tern_fwht_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(tern):
    lib = tern.lib()
    names = declared_entry_points()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    # and the binding knows every one of them
    assert set(names) <= set(tern.EXPORTS)


def test_status_strings(tern):
    lib = tern.lib()
    for s in range(8):
        assert lib.tern_status_str(s)
    assert lib.tern_status_str(99) == b"unknown status"


def test_packed_bytes(tern):
    assert tern.packed_bytes(17408, 5120) == 17408 * 5120 // 4 + 17408 * 5120 // 64 == 23674880
    assert tern.packed_bytes(5120, 6144 // 6144 * 6144) == 5120 * 6144 * 17 // 64
    assert tern.packed_bytes(12288, 4096) == 13369344
    assert tern.packed_bytes(256, 512) == 34816
    assert tern.packed_bytes(3, 100) == 0


def test_host_pack_matches_oracle(tern, orc):
    for seed, (N, K) in enumerate([(1, 16), (7, 128), (33, 1024), (64, 4096)]):
        t = synth.trits(seed, "t", (N, K), synth.UNIFORM)
        c_lib, bad = tern.pack_host(t)
        c_orc, bad_o = orc.pack(t)
        assert bad == bad_o == 0
        assert np.array_equal(c_lib, c_orc)
        back, bad2 = tern.unpack_host(c_lib, K)
        assert bad2 == 0 and np.array_equal(back, t)
        assert tern.validate_host(c_lib, K) == 0


def test_host_pack_invalid_entries(tern, orc):
    t = synth.trits(5, "t", (4, 64), synth.UNIFORM)
    t[0, 3] = 2
    t[1, 63] = -128
    t[3, 17] = 5
    c_lib, bad = tern.pack_host(t)
    c_orc, bad_o = orc.pack(t)
    assert bad == bad_o == 3
    assert np.array_equal(c_lib, c_orc)
    assert tern.validate_host(c_lib, 64) == 3
    _, bad_u = tern.unpack_host(c_lib, 64)
    assert bad_u == 3


def test_validate_counts_every_code3_slot(tern):
    words = np.array([[0xFFFFFFFF, 0x55555555, 0xC0000003, 0x00000000]], dtype=np.uint32)
    assert tern.validate_host(words, 64) == 16 + 0 + 2 + 0


def test_argument_errors_never_launch(tern):
    """Shape, NULL, alignment and workspace errors are reported before any
    device call, so they can be checked without a GPU."""
    lib = tern.lib()
    P = 4096  # a fake, 16-byte aligned "device" address; nothing dereferences it
    # shapes
    assert lib.tern_gemv(P, P, P, P, 0, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_gemv(P, P, P, P, 17, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_gemv(P, P, P, P, 1, 16, 100, P, 1 << 20, None) == 2
    assert lib.tern_gemv(P, P, P, P, 1, 0, 128, P, 1 << 20, None) == 2
    assert lib.tern_fwht(P, P, P, 1, 4000, None) == 2
    assert lib.tern_fwht_gemm(P, P, P, P, P, 1, 16, 5120, P, 1 << 20, None) == 2
    assert lib.tern_pack(P, 4, 17, P, None, None) == 2
    assert lib.tern_gemm(P, P, P, P, 0, 0, 16, 128, P, 1 << 20, None) == 2
    # NULL
    assert lib.tern_gemv(None, P, P, P, 1, 16, 128, P, 1 << 20, None) == 1
    assert lib.tern_fwht(P, None, P, 1, 4096, None) == 1
    assert lib.tern_fwht_gemm(P, None, P, P, P, 1, 16, 4096, P, 1 << 20, None) == 1
    # alignment
    assert lib.tern_gemv(P + 2, P, P, P, 1, 16, 128, P, 1 << 20, None) == 3
    assert lib.tern_fwht(P, P + 8, P, 1, 4096, None) == 3
    # workspace: flag words once K spans more than one 1024-wide slice, plus the
    # staged rotated x for the fused call
    need = tern.gemv_workspace_bytes(1, 16, 2048)
    assert need >= 256
    assert lib.tern_gemv(P, P, P, P, 1, 16, 2048, None, need, None) == 4
    assert lib.tern_gemv(P, P, P, P, 1, 16, 2048, P, need - 1, None) == 4
    assert lib.tern_fwht_gemm(P, P, P, P, P, 1, 16, 4096, None, 1 << 30, None) == 4
    need = tern.gemv_workspace_bytes(2, 16, 4096)
    assert lib.tern_fwht_gemm(P, P, P, P, P, 2, 16, 4096, P, need - 1, None) == 4
    assert tern.gemv_workspace_bytes(17, 16, 128) == 0
    assert lib.tern_gemm(P, P, P, P, 0, 64, 256, 512, None, 1 << 30, None) == 4
    need = tern.gemm_workspace_bytes(64, 256, 512)
    assert lib.tern_gemm(P, P, P, P, 0, 64, 256, 512, P, need - 1, None) == 4
    # the bounded-wait self-test: an unknown wait or a limit out of range
    assert lib.tern_wait_selftest(2, 1000, None) == 2
    assert lib.tern_wait_selftest(-1, 1000, None) == 2
    assert lib.tern_wait_selftest(tern.SELFTEST_RANGE_FLAG, 0, None) == 2
    assert lib.tern_wait_selftest(tern.SELFTEST_MBARRIER, 1000001, None) == 2

def test_workspace_sizes(tern):
    # Once K spans more than one chunk of 8 groups (K > 1024): one flag word per
    # 16-row tile (256-byte aligned).  When K % 4096 == 0 the size also covers
    # the fused call, which for M > 2 stages the rotated x there: M x K fp16
    # values and one int32 exponent per token and 128-group (256-byte
    # aligned); for M <= 2 the product rebuilds it in shared memory.
    a256 = lambda v: (v + 255) // 256 * 256

    def rot(M, K):
        return a256(M * K * 2 + M * (K // 128) * 4)

    assert tern.gemv_workspace_bytes(1, 17408, 5120) == a256(1088 * 4)
    assert tern.gemv_workspace_bytes(16, 10, 17408) == 256
    assert tern.gemv_workspace_bytes(2, 12288, 4096) == a256(768 * 4)
    assert tern.gemv_workspace_bytes(3, 12288, 4096) == a256(768 * 4) + rot(3, 4096)
    assert tern.gemv_workspace_bytes(16, 12288, 8192) == a256(768 * 4) + rot(16, 8192)
    assert tern.gemv_workspace_bytes(1, 16, 4096) == 256
    assert tern.gemv_workspace_bytes(3, 100, 1152) == a256(7 * 4)
    assert tern.gemv_workspace_bytes(1, 256, 512) == 256      # one chunk: nothing needed
    assert tern.gemv_workspace_bytes(1, 256, 1024) == 256
    # a pair call counts the tiles of both matrices
    assert lib_pair(tern, 1, 17408, 17408, 5120) == a256(2176 * 4)


def lib_pair(tern, M, Na, Nb, K):
    return int(tern.lib().tern_gemv_pair_workspace_bytes(M, Na, Nb, K))


def test_gemm_workspace_sizes(tern):
    # counters: tiles x 4 uint32 (256-byte aligned); one 256 x 128 fp32 sum per tile
    def want(M, N, K):
        tiles = -(-M // 256) * -(-N // 128)
        return (tiles * 16 + 255) // 256 * 256 + tiles * 256 * 128 * 4
    for M, N, K in [(512, 17408, 5120), (512, 5120, 17408), (1, 128, 128), (300, 130, 640), (17, 1000, 128)]:
        assert tern.gemm_workspace_bytes(M, N, K) == want(M, N, K)
    assert tern.gemm_workspace_bytes(0, 128, 128) == 0


# --------------------------------------------------------------------------
# the 1-bit sibling format
# --------------------------------------------------------------------------

def test_bin_host_pack_matches_oracle(tern, orc):
    t = synth.binary(40, "hp", (33, 1024))
    words, bad = tern.bin_pack_host(t)
    want, wbad = orc.bin_pack(t)
    assert bad == wbad == 0
    assert np.array_equal(words, want)
    assert np.array_equal(tern.bin_unpack_host(words, 1024), t)
    assert tern.lib().tern_bin_packed_bytes(33, 1024) == words.nbytes + 33 * 8 * 2


def test_bin_host_pack_invalid_entries(tern, orc):
    t = synth.binary(41, "inv", (4, 64))
    t[0, 3] = 0
    t[2, 40] = 2
    t[3, 63] = -7
    words, bad = tern.bin_pack_host(t)
    want, wbad = orc.bin_pack(t)
    assert bad == wbad == 3
    assert np.array_equal(words, want)


def test_bin_argument_errors_never_launch(tern):
    lib = tern.lib()
    P = 4096
    assert lib.tern_bin_pack(P, 4, 48, P, None, None) == 2          # K % 32
    assert lib.tern_bin_pack(P, 4, 64, None, None, None) == 1
    assert lib.tern_bin_pack(P + 8, 4, 64, P, None, None) == 3
    assert lib.tern_bin_packed_bytes(4, 96) == 0
    assert lib.tern_bin_gemv(P, P, P, P, 0, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_bin_gemv(P, P, P, P, 17, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_bin_gemv(P, P, P, P, 1, 16, 96, P, 1 << 20, None) == 2
    assert lib.tern_bin_gemv(None, P, P, P, 1, 16, 128, P, 1 << 20, None) == 1
    assert lib.tern_bin_gemv(P, P + 4, P, P, 1, 16, 128, P, 1 << 20, None) == 3
    need = tern.gemv_workspace_bytes(1, 16, 2048)
    assert lib.tern_bin_gemv(P, P, P, P, 1, 16, 2048, None, need, None) == 4
    assert lib.tern_bin_gemv(P, P, P, P, 1, 16, 2048, P, need - 1, None) == 4
    assert lib.tern_bin_gemm(P, P, P, P, 0, 0, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_bin_gemm(P, P, P, P, 0, 4, 16, 96, P, 1 << 20, None) == 2
    assert lib.tern_bin_gemm(P, None, P, P, 0, 4, 16, 128, P, 1 << 20, None) == 1
    need = tern.gemm_workspace_bytes(64, 256, 512)
    assert lib.tern_bin_gemm(P, P, P, P, 0, 64, 256, 512, P, need - 1, None) == 4


def test_scales_from_g64_host_matches_oracle(tern, orc):
    s128 = synth.scales(61, "g64h", (9, 12))
    s64 = np.repeat(s128, 2, axis=1)
    s64[4, 7] = np.float16(1.5)
    out, bad = tern.scales_from_g64_host(s64, 12 * 128)
    want, wbad = orc.scales_from_g64(s64)
    assert bad == wbad == 1
    assert np.array_equal(out.view(np.uint16), want.view(np.uint16))
    lib = tern.lib()
    assert lib.tern_scales_from_g64(4096, 4, 192, 4096, None, None) == 2      # K % 128
    assert lib.tern_scales_from_g64(None, 4, 256, 4096, None, None) == 1


def test_gemv_pair_argument_errors(tern):
    lib = tern.lib()
    P = 4096
    assert lib.tern_gemv_pair(P, P, P, P, 16, P, P, P, 0, 1, 2048, P, 1 << 20, None) == 2     # N_b = 0
    assert lib.tern_gemv_pair(P, P, P, P, 16, None, P, P, 16, 1, 2048, P, 1 << 20, None) == 1
    assert lib.tern_gemv_pair(P, P, P, P, 16, P + 4, P, P, 16, 1, 2048, P, 1 << 20, None) == 3
    need = tern.lib().tern_gemv_pair_workspace_bytes(1, 17408, 17408, 5120)
    assert need == (2 * 1088 * 4 + 255) // 256 * 256
    assert lib.tern_gemv_pair(P, P, P, P, 17408, P, P, P, 17408, 1, 5120, P, need - 1, None) == 4
    assert tern.lib().tern_gemv_pair_workspace_bytes(1, 16, 16, 1024) == 256


def test_affine_argument_errors_never_launch(tern):
    lib = tern.lib()
    P = 4096
    assert lib.tern_affine_gemv(P, P, P, P, P, 0, 16, 128, P, 1 << 20, None) == 2         # M = 0
    assert lib.tern_affine_gemv(P, P, P, P, P, 17, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_affine_gemv(P, P, P, P, P, 1, 16, 96, P, 1 << 20, None) == 2          # K % 128
    assert lib.tern_affine_gemv(P, P, P, None, P, 1, 16, 128, P, 1 << 20, None) == 1      # no biases
    assert lib.tern_affine_gemv(P, P, P, P + 2, P, 1, 16, 128, P, 1 << 20, None) == 3     # misaligned biases
    assert lib.tern_affine_gemv(P, P + 4, P, P, P, 1, 16, 128, P, 1 << 20, None) == 3
    need = tern.gemv_workspace_bytes(1, 16, 2048)
    assert lib.tern_affine_gemv(P, P, P, P, P, 1, 16, 2048, None, need, None) == 4
    assert lib.tern_affine_gemv(P, P, P, P, P, 1, 16, 2048, P, need - 1, None) == 4
    assert lib.tern_affine_gemm(P, P, P, P, P, 0, 0, 16, 128, P, 1 << 20, None) == 2
    assert lib.tern_affine_gemm(P, P, P, P, P, 0, 4, 16, 96, P, 1 << 20, None) == 2
    assert lib.tern_affine_gemm(P, P, P, None, P, 0, 4, 16, 128, P, 1 << 20, None) == 1
    assert lib.tern_affine_gemm(P, P, P, P + 8, P, 0, 4, 16, 128, P, 1 << 20, None) == 3
    assert lib.tern_affine_gemm(P, None, P, P, P, 0, 4, 16, 128, P, 1 << 20, None) == 1
    need = tern.gemm_workspace_bytes(64, 256, 512)
    assert lib.tern_affine_gemm(P, P, P, P, P, 0, 64, 256, 512, P, need - 1, None) == 4
    assert tern.last_launch_count() == 0


def test_header_is_plain_c_and_a_c_program_links_the_library(tern, tmp_path):
    """The boundary needs no CUDA, torch or C++ headers: tern.h compiles as
    C99 and C++17, and a plain C program links libtern.so and calls its
    host-side entry points (no GPU needed for these)."""
    import subprocess
    inc = os.path.join(ROOT, "include")
    hdr = os.path.join(inc, "tern.h")
    for lang, std, cc in (("c", "-std=c99", "gcc"), ("c++", "-std=c++17", "g++")):
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", lang, hdr],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
    src = tmp_path / "use_tern.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "tern.h"
int main(void) {
    int8_t t[2 * 32];
    uint32_t codes[2 * 2];
    int8_t back[2 * 32];
    long long bad = -1;
    for (int i = 0; i < 64; ++i) t[i] = (int8_t)((i % 3) - 1);
    if (tern_pack_host(t, 2, 32, codes, &bad) != TERN_OK || bad != 0) return 1;
    if (tern_unpack_host(codes, 2, 32, back, &bad) != TERN_OK || bad != 0) return 2;
    if (memcmp(t, back, sizeof t) != 0) return 3;
    if (tern_packed_bytes(17408, 5120) != 23674880u) return 4;
    if (tern_gemv(NULL, NULL, NULL, NULL, 0, 1, 128, NULL, 0, NULL) != TERN_ERR_SHAPE) return 5;
    printf("%s\n", tern_status_str(TERN_OK));
    return 0;
}
''')
    lib = tern.LIB_PATH
    exe = tmp_path / "use_tern"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), lib, "-o", str(exe),
                        f"-Wl,-rpath,{os.path.dirname(lib)}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip()
