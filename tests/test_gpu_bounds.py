"""Out-of-bounds writes and failure detection on the GPU, without a fault.

Canaries.  Every device entry point writes its output into the middle of a
larger buffer whose margins hold a known bit pattern; after the call the
margins must be unchanged, bit for bit.  The shapes are ragged (N not a
multiple of a tile, several K-slices, M past the private-partial limit,
stream-K split tiles), the cases where a stray row or token index would land
outside the output.  Workspaces get the same margins, and a product's
workspace must be back at zero when the call completes (the library's
contract: a completed call leaves it ready for the next).

Bounded waits.  Each product wait has a time limit, after which the kernel
stores an error code and returns.  tern_wait_selftest runs the products' own
wait helpers on a flag and an mbarrier that nothing ever completes; the code
must come back through tern_device_error, reading it must clear it, and a
product run afterwards on the same context must still match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import synth
from tests._util import (assert_bf16_close, assert_fp32_close, dev_bf16, dev_codes, dev_scales, dev_trits, f16_to_bf16_f16,
                         host_codes, l2_xw, x_f64)

pytestmark = pytest.mark.gpu

PAD = 1024           # margin bytes on each side (keeps 256-byte alignment)
CANARY = 0xA5


@pytest.fixture(scope="module")
def tern():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_gemv_gemm_gb300 import build
    build.build()
    import bit_gemv_gemm_gb300 as t
    return t


class Guarded:
    """A device tensor of `shape` and `dtype` viewed out of a byte buffer with
    PAD canary bytes before and after it."""

    def __init__(self, shape, dtype, fill=CANARY, inner=None):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.n = nbytes
        self.buf = torch.full((PAD + nbytes + PAD,), fill, dtype=torch.uint8, device="cuda")
        if inner is not None:
            self.buf[PAD:PAD + nbytes] = inner
        self.t = self.buf[PAD:PAD + nbytes].view(dtype).view(*shape) if nbytes else \
            torch.empty(shape, dtype=dtype, device="cuda")

    def margins_intact(self, fill=CANARY) -> bool:
        torch.cuda.synchronize()
        return bool((self.buf[:PAD] == fill).all() and (self.buf[PAD + self.n:] == fill).all())

    def inner_zero(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.buf[PAD:PAD + self.n] == 0).all())


def workspace(n):
    """A zero-filled workspace of n bytes with canary margins."""
    return Guarded((max(n, 1),), torch.uint8, inner=0)


@pytest.mark.parametrize("N,K", [(37, 128), (1000, 2048), (3, 17408)])
def test_pack_writes_only_its_codes(tern, N, K):
    t = synth.trits(1, "canary", (N, K), synth.UNIFORM)
    codes = Guarded((N, K // 16), torch.int32)
    tern.pack(dev_trits(t), codes=codes.t)
    assert codes.margins_intact()
    assert np.array_equal(host_codes(codes.t), tern.pack_host(t)[0])


@pytest.mark.parametrize("M,K", [(1, 4096), (3, 8192), (16, 4096)])
def test_fwht_writes_only_its_output(tern, M, K):
    x = dev_bf16(synth.activations(2, "canary", (M, K)))
    s = torch.from_numpy(synth.signs(2, "canary", K)).cuda()
    y = Guarded((M, K), torch.bfloat16)
    tern.fwht(x, s, y=y.t)
    assert y.margins_intact()
    assert torch.equal(y.t, tern.fwht(x, s))


@pytest.mark.parametrize("M,N,K", [(1, 1000, 5120), (1, 17408, 5120), (3, 777, 17408), (6, 129, 2176),
                                   (16, 200, 512), (5, 16, 128), (8, 300, 2560)])
def test_gemv_writes_only_its_output(tern, orc, M, N, K):
    p = synth.problem(700 + M, M, N, K, tag=f"cv{N}x{K}")
    x, codes, s = dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(p.s)
    ws = workspace(tern.gemv_workspace_bytes(M, N, K))
    y = Guarded((M, N), torch.float32)
    for _ in range(2):
        tern.gemv(x, codes, s, y=y.t, ws=ws.t)
        assert y.margins_intact() and ws.margins_intact()
        assert ws.inner_zero(), "the range flags are not back at zero"
    assert tern.device_error() == 0
    y_ref, a_ref = orc.matmul(p.x, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.t.cpu().numpy(), y_ref, a_ref, what=f"canary gemv M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(1, 1000, 5120), (1, 129, 17408), (5, 77, 2048), (16, 33, 1024), (3, 40, 640)])
def test_f3_gemv_writes_only_its_output(tern, orc, M, N, K):
    """The base-3 product (no workspace: its range flags are file-scope) twice
    into a guarded y: the margins intact, no device error, the second call
    (after the first has returned its flags to zero) against the oracle."""
    p = synth.problem(760 + M, M, N, K, tag=f"c3{N}x{K}")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    y = Guarded((M, N), torch.float32)
    for _ in range(2):
        tern.f3_gemv(dev_bf16(p.x), torch.from_numpy(packed).cuda(), dev_scales(p.s), y=y.t)
        assert y.margins_intact()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.t.cpu().numpy(), y_ref, a_ref, what=f"canary f3 M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 5])
def test_f3_gemv_reports_activation_out_of_range(tern, orc, M):
    """The base-3 tensor-pipe product stages the activation as the decode
    product does: a group whose largest |x| is 2^100 or more is reported as
    TERN_DEVERR_GEMV_ACTIVATION_RANGE, and the next in-range call (after the
    report was read) matches the oracle."""
    N, K = 300, 2048
    p = synth.problem(1750 + M, M, N, K, tag="f3range")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    dp, ds = torch.from_numpy(packed).cuda(), dev_scales(p.s)
    assert tern.device_error() == 0
    x = p.x.copy()
    x[M - 1, 1500] = np.uint16(np.array([2.0 ** 101], dtype=np.float32).view(np.uint32)[0] >> 16)
    tern.f3_gemv(dev_bf16(x), dp, ds)
    torch.cuda.synchronize()
    assert tern.device_error() == tern.DEVERR_GEMV_ACTIVATION_RANGE
    y = tern.f3_gemv(dev_bf16(p.x), dp, ds)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.f3_matmul(p.x, packed, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what=f"f3 after a range report M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 1000, 5120), (3, 777, 17408), (6, 129, 2176), (16, 200, 640)])
def test_bin_gemv_writes_only_its_output(tern, orc, M, N, K):
    p = synth.binary_problem(750 + M, M, N, K, tag=f"cb{N}x{K}")
    words = Guarded((N, K // 32), torch.int32)
    tern.bin_pack(dev_trits(p.t), words=words.t)
    assert words.margins_intact()
    ws = workspace(tern.gemv_workspace_bytes(M, N, K))
    y = Guarded((M, N), torch.float32)
    for _ in range(2):
        tern.bin_gemv(dev_bf16(p.x), words.t, dev_scales(p.s), y=y.t, ws=ws.t)
        assert y.margins_intact() and ws.margins_intact()
        assert ws.inner_zero(), "the range flags are not back at zero"
    assert tern.device_error() == 0
    y_ref, a_ref = orc.bin_matmul(p.x, orc.bin_pack(p.t)[0], p.s)
    assert_fp32_close(y.t.cpu().numpy(), y_ref, a_ref, what=f"canary binary M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 16])
def test_fwht_gemm_writes_only_its_output(tern, orc, M):
    N, K = 600, 4096
    p = synth.problem(800 + M, M, N, K, with_signs=True, tag="cr")
    x, codes, s = dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(p.s)
    ws = workspace(tern.gemv_workspace_bytes(M, N, K))
    y = Guarded((M, N), torch.float32)
    tern.fwht_gemm(x, torch.from_numpy(p.signs).cuda(), codes, s, y=y.t, ws=ws.t)
    assert y.margins_intact() and ws.margins_intact()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.rotate_matmul(p.x, p.signs, orc.pack(p.t)[0], p.s)
    assert_fp32_close(y.t.cpu().numpy(), y_ref, a_ref, what=f"canary fused M={M}")


@pytest.mark.parametrize("M,N,K,dt", [(300, 130, 640, torch.float32), (17, 1000, 128, torch.bfloat16),
                                      (256, 256, 8192, torch.float32), (40, 128, 2048, torch.bfloat16),
                                      (513, 400, 1024, torch.bfloat16)])
def test_gemm_writes_only_its_output(tern, orc, M, N, K, dt):
    p = synth.problem(900 + M, M, N, K, tag=f"cg{N}x{K}")
    x, codes, s = dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(p.s)
    ws = workspace(tern.gemm_workspace_bytes(M, N, K))
    y = Guarded((M, N), dt)
    for _ in range(2):
        tern.gemm(x, codes, s, y=y.t, ws=ws.t)
        assert y.margins_intact() and ws.margins_intact()
        assert ws.inner_zero(), "the stream-K counters or sums are not back at zero"
    assert tern.device_error() == 0
    ocodes, sb = orc.pack(p.t)[0], f16_to_bf16_f16(p.s)   # the prefill's operand: t * bf16(s_g)
    y_b, a_b = orc.matmul(p.x, ocodes, sb)
    got = y.t.to(torch.float64).cpu().numpy()
    if dt == torch.bfloat16:
        assert_bf16_close(got, y_b, l2_xw(p.x, p.t, sb), what=f"canary gemm M={M}")
    else:
        assert_fp32_close(got, y_b, a_b, what=f"canary gemm M={M}")


@pytest.mark.parametrize("which,code", [(0, 0x202), (1, 0x103)])
def test_bounded_wait_reports_and_context_survives(tern, orc, which, code):
    assert which in (tern.SELFTEST_RANGE_FLAG, tern.SELFTEST_MBARRIER)
    assert code in (tern.DEVERR_GEMV_RANGE_FLAG_WAIT, tern.DEVERR_GEMM_MMA_WAIT)
    assert tern.device_error() == 0
    tern.wait_selftest(which, 2000)      # first launch: loads the module
    assert tern.device_error() == code
    t0 = time.perf_counter()
    tern.wait_selftest(which, 2000)      # 2 ms limit
    got = tern.device_error()            # synchronizes
    elapsed = time.perf_counter() - t0
    assert got == code
    # well under the products' 1 s limit: for the mbarrier case this also shows
    # that the second role's 1 s wait ended on the first role's abort flag
    assert elapsed < 0.5, elapsed
    assert tern.device_error() == 0, "reading the error word did not clear it"
    # the context is still usable: a multi-slice decode product (which itself
    # waits on range flags) and a prefill product match the oracle
    M, N, K = 2, 600, 5120
    p = synth.problem(1000 + which, M, N, K, tag="after")
    x, codes, s = dev_bf16(p.x), tern.pack(dev_trits(p.t)), dev_scales(p.s)
    ocodes = orc.pack(p.t)[0]
    y_ref, a_ref = orc.matmul(p.x, ocodes, p.s)
    assert_fp32_close(tern.gemv(x, codes, s).cpu().numpy(), y_ref, a_ref, what="gemv after self-test")
    y_b, a_b = orc.matmul(p.x, ocodes, f16_to_bf16_f16(p.s))
    assert_fp32_close(tern.gemm(x, codes, s).cpu().numpy(), y_b, a_b, what="gemm after self-test")
    assert tern.device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("big", [2.0 ** 100, 2.0 ** 120, float("inf")])
def test_gemv_reports_activation_out_of_range(tern, orc, big):
    """An activation group whose largest |x| is 2^100 or more, or not finite,
    is outside the fp16 staging's exponent range: the call reports
    TERN_DEVERR_GEMV_ACTIVATION_RANGE instead of returning wrong numbers
    silently.  Just below the bound the product is still within tolerance,
    and the next in-range call reports nothing."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 2, 300, 2048
    p = synth.problem(1700, M, N, K, tag="range")
    ocodes, bad = orc.pack(p.t)
    assert bad == 0
    codes, s = dev_codes(ocodes), dev_scales(p.s)
    assert tern.device_error() == 0
    def bf16_bits(v):   # the bf16 bit pattern of a value bf16 holds exactly
        return np.uint16(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)

    x = p.x.copy()   # bf16 bit patterns
    x[1, 777] = bf16_bits(big)
    y = tern.gemv(dev_bf16(x), codes, s)
    torch.cuda.synchronize()
    assert tern.device_error() == tern.DEVERR_GEMV_ACTIVATION_RANGE
    # just below the bound: no report.  The other activations of that group
    # are 2^99 below its largest and drop out of the fp16 staging, which the
    # group term of the stated bound covers: |y - y_ref| <= 1e-3 sum_k |x w|
    # + 2^-22 sum_g |s_g| max_{k in g} |x_k| + 1e-6
    x[1, 777] = bf16_bits(2.0 ** 99 * 1.5)
    y = tern.gemv(dev_bf16(x), codes, s)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.matmul(x, ocodes, p.s)
    xs = np.abs(x_f64(x)).reshape(M, K // 128, 128).max(axis=2)          # [M][G]
    group_term = xs @ np.abs(p.s.astype(np.float64)).T                    # [M][N]
    err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
    assert (err <= 1e-3 * a_ref + 2.0 ** -22 * group_term + 1e-6).all()
    # the rows whose weight at the large activation is not zero meet the plain bound
    rows = np.nonzero(p.t[:, 777] != 0)[0]
    assert rows.size > 0
    assert_fp32_close(y.cpu().numpy()[1, rows], y_ref[1, rows], a_ref[1, rows], what="gemv just below the bound")
    # and with the whole group that large, every row does
    x[1, 768:896] = bf16_bits(2.0 ** 98)
    x[1, 777] = bf16_bits(2.0 ** 99 * 1.5)
    y = tern.gemv(dev_bf16(x), codes, s)
    torch.cuda.synchronize()
    assert tern.device_error() == 0
    y_ref, a_ref = orc.matmul(x, ocodes, p.s)
    assert_fp32_close(y.cpu().numpy(), y_ref, a_ref, what="gemv with a whole group near the bound")
