// tern_decode.cu -- the decode / small-batch ternary-g128 product (M = 1..16)
// on FP8 tensor-core adds, for K a multiple of 1024.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} x[m][k] * (q[n][k] - 1)
//
// ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card: ternary weights with one
// FP16 scale per 128 along K, "Weight representation: ternary g128"; the codes
// are unpacked and scaled inside the product and never expanded to a dense
// tensor, "CUDA (NVIDIA GPUs)"; token generation is the memory-bound phase,
// "Cross-platform throughput".)
//
// Why FP8.  At 2.125 bits per weight an SM must retire ~80 weights per clock
// for HBM to stay busy.  On this part the legacy m16n8k32 e4m3 x e5m2 MMA
// issues every ~4.5 cycles per sub-partition (512 weights of a 16-row tile),
// against ~8 cycles for the f16 m16n8k16 (256 weights), and the logic ops an
// unpack needs run at half rate.  The FP8 path needs four times fewer of both.
//
// Weights (operand A, e4m3).  A code word holds codes 0..15 of a 16-weight
// slice in bits 2j.  Masking a word with 0x03030303 leaves codes 0, 4, 8, 12
// in the low two bits of the four bytes: as e4m3 that byte is the subnormal
// q * 2^-9.  Masking with 0x0C0C0C0C leaves codes 1, 5, 9, 13 in bits 2-3: the
// byte reads q * 2^-7 (bit 2 is the top mantissa bit, bit 3 the exponent's
// lowest), again linear in q = 0, 1, 2 (and 3).  Codes 2, 6, 10, 14 and 3, 7,
// 11, 15 take the same two masks after one shift by 4.  So one logical op per
// four weights gives an MMA A register, and MMA c (c = 0..3) of a 128-weight
// group takes codes c, c+4, c+8, c+12 of each word.  The weight k of the group
// sits, for lane (gid, t), in MMA c = k % 4 at fragment column 4t + b (+16),
// k = 32 t + 16 hh + 4 b + c: the K order is permuted, identically for the
// activation.
//
// Activation (operand B, e5m2).  Per token and group, E is chosen from the
// largest |x| so that |x| 2^E < 2^15.  Every value v = x 2^E (2^(E-2) for the
// odd MMAs, whose A bytes are 4x larger) is split exactly into three terms of
// at most three significant bits: t0 = v truncated to three bits, t1 = (v - t0)
// truncated, t2 = v - t0 - t1 (a bf16 value has eight).  Each term is an e5m2
// value (exact while the term stays above 2^-14; smaller values, below 2^-28 of
// the group's largest, keep an error under 2^-17 in these units).  The three
// terms of token m go to three B columns; with four tokens per lane quad a
// 16-row tile needs ceil(3 H / 2) MMA column tiles for H = ceil(M / 4) token
// slots.  Column tile j, column 2 t' + p holds term tau of token 4 h + t' for
// 3 h + tau = 2 j + p, so the C fragment of lane t holds all three terms of its
// tokens and no shuffle is needed.  Every product q x 2^(E-9) is exact, and
// the tensor core sums them to within ~2^-22 of their absolute sum.
//
// The -1 of q - 1.  Per (token, group) the same chains run once on the
// all-ones code pattern (q = 1) give A1 with the very same rounding, and per
// row y += s_g 2^(9 - E) ((c_tau0 + c_tau1) + c_tau2 - A1): a row of zero
// weights gives exactly 0.
//
// Work split.  K is cut into chunks of 8 groups (1024 weights); the (chunk,
// 16-row tile) pairs are ordered chunk-major and dealt in equal contiguous
// ranges to one CTA per SM, so a CTA sees at most a few chunks (segments).
// A CTA has 8 consumer warps (warp w takes group w of the chunk), a producer
// warp and a reducer warp.  The producer streams stages of U tiles x 8 groups
// (codes with a 128-byte swizzle, and the scales) by TMA into a ring, and
// starts before the programmatic-dependent-launch wait: weights are never the
// previous kernel's output.  A consumer stages its group's activation into
// registers once per segment, then per tile unpacks, runs the MMA chains and
// writes per-row partials for its group.  The reducer sums the 8 groups'
// partials of a stage.  With one chunk it stores y.  With several, y is
// accumulated with global float reductions: the CTA holding a tile's chunk 0
// clears the tile's rows of y at its start and counts the tile into a flag
// word; a CTA holding another chunk of the tile waits (bounded) until the flag
// is non-zero, counts itself in (the S-th count returns the flag to 0, so the
// workspace is back at zero after every call) and adds its sums.  The order in
// which the chunks' sums meet is not fixed: the last bits of y may differ from
// run to run.
//
// Every wait is bounded (1 s).  A wait that runs out raises the CTA's abort
// flag and the sticky device error word; the producer then waits (bounded) for
// its copies in flight before the CTA exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "tern_sm100.cuh"

namespace tern {
namespace {

using namespace sm100;

constexpr int kDecGroup = 128;
constexpr int kDecGroups = 8;                          // groups per K-chunk
constexpr int kDecTileCodeBytes = 16 * 256;            // one 16-row tile x 8 groups of codes
constexpr int kDecTileScaleBytes = 16 * 16;            // its scales
constexpr uint64_t kDecWaitNs = 1000000000ull;         // 1 s: far beyond any real wait
constexpr uint64_t kDecDrainNs = 100000000ull;         // copies in flight after an abort

__device__ int g_decode_error;   // sticky device error word of this translation unit

// Per token-slot count H (M <= 4 H): tiles per stage U, ring stages D, partial buffers PB,
// units whose MMA chains are interleaved NB, reducer warps R, consumer warps CW (a multiple of
// 8: consumer warp w takes group w % 8 and every (CW / 8)-th tile of a stage from tile w / 8).
template <int H> struct DecCfg;
// H = 0: the single-token layout (M = 1), two groups per MMA tile
template <> struct DecCfg<0> { static constexpr int U = 4, D = 5, kMinCtas = 1, PB = 3, R = 1, CW = 16; };
template <> struct DecCfg<1> { static constexpr int U = 4, D = 5, kMinCtas = 1, PB = 3, NB = 2, R = 1, CW = 16; };
template <> struct DecCfg<2> { static constexpr int U = 2, D = 6, kMinCtas = 1, PB = 2, NB = 1, R = 2, CW = 16; };
template <> struct DecCfg<3> { static constexpr int U = 2, D = 6, kMinCtas = 1, PB = 2, NB = 1, R = 4, CW = 8; };
template <> struct DecCfg<4> { static constexpr int U = 2, D = 6, kMinCtas = 1, PB = 2, NB = 1, R = 4, CW = 8; };

struct DecArgs {
    const __nv_bfloat16* x;   // [M][K]
    float* y1;                // [M][N1]
    float* y2;                // [M][N2] (a pair call)
    unsigned* cnt;            // [T] per-tile flag words (S > 1), 0 between calls
    long long L;              // S * T (chunk, tile) pairs
    int M, N1, N2, K, G, S, T1, T, P;
    int mpad;                 // floats per partial row
    uint32_t off_scl, off_part, off_bst, off_est, off_bar;   // from the 1024-aligned base
    uint32_t part_floats;     // floats per partial buffer
};

__device__ __forceinline__ void mma_e4e5(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, bool accumulate) {
    if (accumulate) {
        asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e5m2.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        const float z = 0.0f;
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e5m2.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    }
}

// The A registers of one unit: for MMA c, codes c, c+4, c+8, c+12 of each of
// the lane's four words as e4m3 bytes, q 2^-9 (c even) or q 2^-7 (c odd).
// A[c][0..3] = (row gid word 2t, row gid+8 word 2t, row gid word 2t+1, row
// gid+8 word 2t+1) in the MMA's a0..a3 order.  Written as one block of PTX
// shifts and ANDs: the same masks written as C++ expressions were compiled into
// a sequence that fed the MMAs about five times slower on this part.
__device__ __forceinline__ void unit_regs(uint32_t (&A)[4][4], uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
    asm("{\n.reg .b32 t0, t1, t2, t3;\n"
        "shr.b32 t0, %16, 4;\nshr.b32 t1, %17, 4;\nshr.b32 t2, %18, 4;\nshr.b32 t3, %19, 4;\n"
        "and.b32 %0, %16, 0x03030303;\nand.b32 %1, %18, 0x03030303;\nand.b32 %2, %17, 0x03030303;\nand.b32 %3, %19, 0x03030303;\n"
        "and.b32 %4, %16, 0x0C0C0C0C;\nand.b32 %5, %18, 0x0C0C0C0C;\nand.b32 %6, %17, 0x0C0C0C0C;\nand.b32 %7, %19, 0x0C0C0C0C;\n"
        "and.b32 %8, t0, 0x03030303;\nand.b32 %9, t2, 0x03030303;\nand.b32 %10, t1, 0x03030303;\nand.b32 %11, t3, 0x03030303;\n"
        "and.b32 %12, t0, 0x0C0C0C0C;\nand.b32 %13, t2, 0x0C0C0C0C;\nand.b32 %14, t1, 0x0C0C0C0C;\nand.b32 %15, t3, 0x0C0C0C0C;\n}"
        : "=r"(A[0][0]), "=r"(A[0][1]), "=r"(A[0][2]), "=r"(A[0][3]), "=r"(A[1][0]), "=r"(A[1][1]), "=r"(A[1][2]),
          "=r"(A[1][3]), "=r"(A[2][0]), "=r"(A[2][1]), "=r"(A[2][2]), "=r"(A[2][3]), "=r"(A[3][0]), "=r"(A[3][1]),
          "=r"(A[3][2]), "=r"(A[3][3])
        : "r"(w0), "r"(w1), "r"(w2), "r"(w3));
}

// The chains of NU units (16 rows x one group each) into acc[NU][NT][4]: MMA c
// in order 0..3 for every unit and column tile, the NU x NT chains interleaved
// so that consecutive MMAs are independent.  w[u] = (row gid word 2t, word
// 2t+1, row gid+8 word 2t, word 2t+1) of unit u.
template <int NU, int NT>
__device__ __forceinline__ void unit_chains(float (&acc)[NU][NT][4], const uint32_t (&w)[NU][4],
                                            const uint32_t (&b)[NT][8]) {
    uint32_t A[NU][4][4];
#pragma unroll
    for (int u = 0; u < NU; ++u) unit_regs(A[u], w[u][0], w[u][1], w[u][2], w[u][3]);
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
            for (int j = 0; j < NT; ++j)
                mma_e4e5(acc[u][j], A[u][c][0], A[u][c][1], A[u][c][2], A[u][c][3], b[j][2 * c], b[j][2 * c + 1], c > 0);
}

// Three-significant-bit truncation of an fp32 value (sign, exponent, top two
// mantissa bits).
__device__ __forceinline__ float trunc3(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFE00000u); }

// Two fp32 values to e5m2 (round to nearest even; exact for the terms here):
// hi byte = a, lo byte = b.
__device__ __forceinline__ uint32_t cvt_e5m2x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void sts_u8(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
// Named barrier among `n` threads (a multiple of 32), and the same with an AND
// of a predicate over those threads.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, %2, %3, p;\nselp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
// Counts into a flag word modulo wrap + 1, without waiting for the old value.
__device__ __forceinline__ void red_inc_wrap(unsigned* p, unsigned wrap) {
    asm volatile("red.relaxed.gpu.global.inc.u32 [%0], %1;" ::"l"(p), "r"(wrap) : "memory");
}

// The (chunk, tile) walk of a CTA's range of pairs: a stage is up to U tiles
// of one chunk.  32-bit: the shape limits keep S * T below 2^30.
struct StageWalk {
    int nkc, ntile, left, T, U;   // the next stage starts at (nkc, ntile); `left` pairs remain
    int kc, tile, n;              // the current stage
    __device__ StageWalk(long long L0, long long L1, int T_, int U_) : T(T_), U(U_), kc(0), tile(0), n(0) {
        nkc = (int)(L0 / T_);
        ntile = (int)(L0 - (long long)nkc * T_);
        left = (int)(L1 - L0);
    }
    __device__ bool next() {
        if (left <= 0) return false;
        kc = nkc;
        tile = ntile;
        n = min(U, min(T - ntile, left));
        ntile += n;
        left -= n;
        if (ntile == T) {
            ntile = 0;
            ++nkc;
        }
        return true;
    }
};

// A bounded mbarrier wait for a whole warp: lane 0 polls, the others then
// observe the completed phase once (each lane takes its own acquire), so the
// 32 lanes do not all poll the shared-memory barrier.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag, int lane) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort_flag, kDecWaitNs);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok;
}

template <int H>
constexpr int dec_threads() { return (DecCfg<H>::CW + 1 + DecCfg<H>::R) * 32; }   // + producer + reducers
// B registers a consumer lane holds (in units of 8: one MMA column tile's worth),
// and the partial slots a stage's rows collect: 8 groups, or for M = 1 the
// three busy lanes of each of the 4 group pairs
template <int H>
constexpr int dec_nt() { return H == 0 ? 2 : (3 * H + 1) / 2; }
template <int H>
constexpr int dec_slots() { return H == 0 ? 12 : kDecGroups; }

template <int H>
__global__ void __launch_bounds__(dec_threads<H>(), DecCfg<H>::kMinCtas)
decode_kernel(const __grid_constant__ CUtensorMap mc1, const __grid_constant__ CUtensorMap ms1,
              const __grid_constant__ CUtensorMap mc2, const __grid_constant__ CUtensorMap ms2, const DecArgs a) {
    constexpr int NT = dec_nt<H>(), SLOTS = dec_slots<H>();
    constexpr int U = DecCfg<H>::U, D = DecCfg<H>::D, PB = DecCfg<H>::PB, R = DecCfg<H>::R, CW = DecCfg<H>::CW;
    extern __shared__ __align__(1024) unsigned char dec_smem_raw[];
    // the 1024-aligned base, by pointer arithmetic on the shared array so that
    // every access through it stays a shared-memory access
    unsigned char* smem = dec_smem_raw + ((1024u - (smem_u32(dec_smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t s_codes = sbase;                 // [D][U][2 halves][16 rows][128 B], 128-byte swizzle
    const uint32_t s_scl = sbase + a.off_scl;       // [D][U][16 rows][8 groups] fp16
    float* part = reinterpret_cast<float*>(smem + a.off_part);   // [PB][8 warps][16 U rows][mpad]
    const uint32_t s_bst = sbase + a.off_bst;       // [8 warps][32 lanes][NT][8] uint32 (staging)
    int* est = reinterpret_cast<int*>(smem + a.off_est);          // [8 warps][16] staging exponents
    const uint32_t bar0 = sbase + a.off_bar;
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(D + s); };
    auto pfull_bar = [&](int p) { return bar0 + 8u * (uint32_t)(2 * D + p); };
    auto pempty_bar = [&](int p) { return bar0 + 8u * (uint32_t)(2 * D + PB + p); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a.off_bar + 8 * (2 * D + 2 * PB));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CW);
        }
        for (int p = 0; p < PB; ++p) {
            mbar_init(pfull_bar(p), CW);
            mbar_init(pempty_bar(p), R);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const long long L0 = a.L * blockIdx.x / a.P, L1 = a.L * (blockIdx.x + 1) / a.P;
    auto fail = [&](int code) {
        if (!*abort_flag) {
            *abort_flag = 1;
            report_device_error(&g_decode_error, code);
        }
    };

    if (warp == CW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            tma_prefetch_desc(&mc1);
            tma_prefetch_desc(&ms1);
            if (a.N2 > 0) {
                tma_prefetch_desc(&mc2);
                tma_prefetch_desc(&ms2);
            }
            StageWalk wk(L0, L1, a.T, U);
            int s = 0;
            bool ok = true;
            while (wk.next()) {
                const int slot = s % D;
                if (s >= D && !mbar_wait_bounded(empty_bar(slot), (uint32_t)((s / D) - 1) & 1u, abort_flag,
                                                  kDecWaitNs)) {
                    fail(TERN_DEVERR_DECODE_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(slot), (uint32_t)wk.n * (kDecTileCodeBytes + kDecTileScaleBytes));
                for (int i = 0; i < wk.n; ++i) {
                    const int tl = wk.tile + i;
                    const bool second = tl >= a.T1;
                    const CUtensorMap* mc = second ? &mc2 : &mc1;
                    const CUtensorMap* ms = second ? &ms2 : &ms1;
                    const int row0 = (second ? tl - a.T1 : tl) * 16;
                    const uint32_t dst = s_codes + (uint32_t)((slot * U + i) * kDecTileCodeBytes);
                    tma_load_2d(dst, mc, 64 * wk.kc, row0, full_bar(slot));
                    tma_load_2d(dst + 2048u, mc, 64 * wk.kc + 32, row0, full_bar(slot));
                    tma_load_2d(s_scl + (uint32_t)((slot * U + i) * kDecTileScaleBytes), ms, 8 * wk.kc, row0,
                                full_bar(slot));
                }
                ++s;
            }
            // no copy may still be landing when the CTA exits: wait for the
            // stages issued last (already complete on the normal path)
            for (int q = std::max(0, s - D); q < s; ++q)
                if (!mbar_wait_drain(full_bar(q % D), (uint32_t)(q / D) & 1u, kDecDrainNs)) break;
            (void)ok;
        }
        return;
    }

    const int gid = lane >> 2, t = lane & 3;
    const int M = a.M;

    if (warp > CW) {
        // ---------------- reducers (R warps) ----------------
        const int rl = (warp - CW - 1) * 32 + lane, RT = R * 32;
        pdl_wait();   // the previous kernel may still read y, or use the workspace
        if (a.S > 1) {
            // y starts at zero: this CTA clears the rows of its chunk-0 tiles,
            // then counts each such tile into its flag word.  A chunk other
            // than 0 waits until its tiles' flags are non-zero, counts itself in
            // and then adds into y; the S-th count returns a flag to 0.
            const long long c0end = min(L1, (long long)a.T);
            const int t0 = (int)L0, nt = L0 < c0end ? (int)(c0end - L0) : 0;
            for (int q = rl; q < nt * M; q += RT) {
                const int ti = q / M, m = q - ti * M, tl = t0 + ti;
                const bool second = tl >= a.T1;
                const int Nm = second ? a.N2 : a.N1;
                const int row0 = (second ? tl - a.T1 : tl) * 16;
                float* d = (second ? a.y2 : a.y1) + (size_t)m * Nm + row0;
                const int nr = min(16, Nm - row0);
                for (int r = 0; r < nr; ++r) d[r] = 0.0f;
            }
            __threadfence();
            named_bar_sync(1, RT);
            for (int i = rl; i < nt; i += RT) red_inc_wrap(a.cnt + t0 + i, (unsigned)(a.S - 1));
            // the tiles of the chunks past 0: each flag read, then polled
            bool ok = true;
            for (long long pos = max(L0, (long long)a.T) + rl; ok && pos < L1; pos += RT) {
                const int tl = (int)(pos % a.T);
                ok = ld_acquire_gpu(a.cnt + tl) != 0u || wait_flag_nonzero(a.cnt + tl, kDecWaitNs);
                if (ok) red_inc_wrap(a.cnt + tl, (unsigned)(a.S - 1));
            }
            if (!named_bar_and(1, RT, ok)) {
                if (rl == 0) fail(TERN_DEVERR_DECODE_REDUCER_WAIT);
                return;
            }
        }
        StageWalk wk(L0, L1, a.T, U);
        int s = 0;
        while (wk.next()) {
            const int pb = s % PB;
            if (!warp_wait(pfull_bar(pb), (uint32_t)(s / PB) & 1u, abort_flag, lane)) {
                fail(TERN_DEVERR_DECODE_REDUCER_WAIT);
                return;
            }
            const float* pp = part + (size_t)pb * a.part_floats;
            const int nout = wk.n * 16 * M;
            for (int idx = rl; idx < nout; idx += RT) {
                const int r = idx / M, m = idx - r * M;
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < SLOTS; ++w) v += pp[(w * 16 * U + r) * a.mpad + m];
                const int tl = wk.tile + (r >> 4);
                const bool second = tl >= a.T1;
                const int row = (second ? tl - a.T1 : tl) * 16 + (r & 15);
                const int Nm = second ? a.N2 : a.N1;
                if (row < Nm) {
                    float* dst = (second ? a.y2 : a.y1) + (size_t)m * Nm + row;
                    if (a.S == 1) *dst = v;
                    else red_add_f32(dst, v);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty_bar(pb));
            ++s;
        }
        return;
    }

    // ---------------- consumers ----------------
    if constexpr (H == 0) {
        // One token.  Warp w takes the group pair (2 gp, 2 gp + 1) of the chunk
        // and every (CW / 4)-th tile of a stage from tile w / 4.  The three terms
        // of group 2 gp + z are the B columns 3 z .. 3 z + 2 of one MMA tile (its
        // other columns zero), so one chain of 8 MMAs covers both groups of a
        // 16-row tile and every lane t < 3 holds two columns of it.
        const int gp = warp & 3, ph = warp >> 2;
        constexpr int TS = CW / 4;
        uint32_t b[2][8];
        float A1r[2][2], F2[2];
        const uint32_t my_bst = s_bst + (uint32_t)(warp * 32 * 16) * 4u;
        int* my_est = est + warp * 16;
        const int tq = lane >> 3, hh = (lane >> 2) & 1, bb = lane & 3;   // staging: target t, half, byte
        auto stage_pair = [&](int g0) {
#pragma unroll
            for (int q = 0; q < 16; q += 4)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(my_bst + (uint32_t)(lane * 16 + q) * 4u),
                             "r"(0u)
                             : "memory");
            __syncwarp();
#pragma unroll
            for (int z = 0; z < 2; ++z) {
                const uint2 raw = *reinterpret_cast<const uint2*>(a.x + (size_t)(g0 + z) * kDecGroup + 4 * lane);
                float f[4];
                f[0] = __uint_as_float(raw.x << 16);
                f[1] = __uint_as_float(raw.x & 0xFFFF0000u);
                f[2] = __uint_as_float(raw.y << 16);
                f[3] = __uint_as_float(raw.y & 0xFFFF0000u);
                float mx = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const int E = min(127, 141 - (int)(__float_as_uint(mx) >> 23));   // mx 2^E < 2^15
                if (lane == 0) my_est[z] = E;
                const float fe = __uint_as_float((uint32_t)(E + 127) << 23);
                const float fo = __uint_as_float((uint32_t)(E + 125) << 23);
                float t0[4], t1[4], t2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v = f[e] * ((e & 1) ? fo : fe);
                    t0[e] = trunc3(v);
                    const float r1 = v - t0[e];
                    t1[e] = trunc3(r1);
                    t2[e] = r1 - t1[e];
                }
#pragma unroll
                for (int tau = 0; tau < 3; ++tau) {
                    const float* tv = tau == 0 ? t0 : tau == 1 ? t1 : t2;
                    const int col = 3 * z + tau;
                    const uint32_t p01 = cvt_e5m2x2(tv[0], tv[1]);
                    const uint32_t p23 = cvt_e5m2x2(tv[2], tv[3]);
                    const uint32_t base =
                        my_bst + (uint32_t)((col * 4 + tq) * 16 + z * 8) * 4u + (uint32_t)hh * 4u + (uint32_t)bb;
                    sts_u8(base + 0u * 8u, p01 >> 8);   // MMA c: register 2c + hh of set z
                    sts_u8(base + 1u * 8u, p01);
                    sts_u8(base + 2u * 8u, p23 >> 8);
                    sts_u8(base + 3u * 8u, p23);
                }
            }
            __syncwarp();
#pragma unroll
            for (int z = 0; z < 2; ++z) {
                const uint32_t ad = my_bst + (uint32_t)(lane * 16 + z * 8) * 4u;
                uint4 lo, hi;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w) : "r"(ad));
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                             : "r"(ad + 16u));
                b[z][0] = lo.x; b[z][1] = lo.y; b[z][2] = lo.z; b[z][3] = lo.w;
                b[z][4] = hi.x; b[z][5] = hi.y; b[z][6] = hi.z; b[z][7] = hi.w;
            }
            // the all-ones chain, the same 8 MMAs as a tile's
            uint32_t O[4][4];
            unit_regs(O, 0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
            float acc1[4];
#pragma unroll
            for (int z = 0; z < 2; ++z)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    mma_e4e5(acc1, O[c][0], O[c][1], O[c][2], O[c][3], b[z][2 * c], b[z][2 * c + 1], z + c > 0);
            A1r[0][0] = acc1[0];
            A1r[0][1] = acc1[1];
            A1r[1][0] = acc1[2];
            A1r[1][1] = acc1[3];
            F2[0] = __uint_as_float((uint32_t)(9 - my_est[0] + 127) << 23);   // 2^(9 - E)
            F2[1] = __uint_as_float((uint32_t)(9 - my_est[1] + 127) << 23);
            __syncwarp();
        };
        // the lane's columns 2t, 2t+1 belong to groups z0, z1 (t = 3: none)
        const int z0 = (2 * t) / 3, z1 = (2 * t + 1) / 3;
        auto lane_off_of = [&](int g) {
            return (uint32_t)((g >> 2) * 2048 + gid * 128 + ((((2 * (g & 3)) + (t >> 1)) ^ gid) << 4) + 8 * (t & 1));
        };
        const uint32_t lo0 = lane_off_of(2 * gp), lo1 = lane_off_of(2 * gp + 1);
        bool waited = false;
        StageWalk wk(L0, L1, a.T, U);
        int s = 0, cur_kc = -1;
        while (wk.next()) {
            if (wk.kc != cur_kc) {
                if (!waited) {
                    pdl_wait();   // x may be the previous kernel's output
                    waited = true;
                }
                stage_pair(kDecGroups * wk.kc + 2 * gp);
                cur_kc = wk.kc;
            }
            const int slot = s % D, pb = s % PB;
            if (!warp_wait(full_bar(slot), (uint32_t)(s / D) & 1u, abort_flag, lane) ||
                (s >= PB && !warp_wait(pempty_bar(pb), (uint32_t)((s / PB) - 1) & 1u, abort_flag, lane))) {
                fail(TERN_DEVERR_DECODE_CONSUMER_WAIT);
                return;
            }
            float* pw = part + (size_t)pb * a.part_floats + (size_t)(gp * 3 + min(t, 2)) * 16 * U;
            const unsigned char* cs = smem + (size_t)slot * U * kDecTileCodeBytes;
            const unsigned char* ss = smem + a.off_scl + (size_t)slot * U * kDecTileScaleBytes + gid * 16 + 4 * gp;
#pragma unroll 1
            for (int i = ph; i < wk.n; i += TS) {
                const uint2 ra0 = *reinterpret_cast<const uint2*>(cs + i * kDecTileCodeBytes + lo0);
                const uint2 rb0 = *reinterpret_cast<const uint2*>(cs + i * kDecTileCodeBytes + lo0 + 1024);
                const uint2 ra1 = *reinterpret_cast<const uint2*>(cs + i * kDecTileCodeBytes + lo1);
                const uint2 rb1 = *reinterpret_cast<const uint2*>(cs + i * kDecTileCodeBytes + lo1 + 1024);
                const __half2 sg0 = *reinterpret_cast<const __half2*>(ss + i * kDecTileScaleBytes);         // row gid: groups 2gp, 2gp+1
                const __half2 sg1 = *reinterpret_cast<const __half2*>(ss + i * kDecTileScaleBytes + 128);   // row gid + 8
                uint32_t A0[4][4], A1[4][4];
                unit_regs(A0, ra0.x, ra0.y, rb0.x, rb0.y);
                unit_regs(A1, ra1.x, ra1.y, rb1.x, rb1.y);
                float acc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    mma_e4e5(acc, A0[c][0], A0[c][1], A0[c][2], A0[c][3], b[0][2 * c], b[0][2 * c + 1], c > 0);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    mma_e4e5(acc, A1[c][0], A1[c][1], A1[c][2], A1[c][3], b[1][2 * c], b[1][2 * c + 1], true);
                const float2 sa = __half22float2(sg0), sb = __half22float2(sg1);
                const float ga0 = sa.x * F2[0], gb0 = sa.y * F2[1], ga1 = sb.x * F2[0], gb1 = sb.y * F2[1];
                if (t < 3) {
                    pw[16 * i + gid] = (acc[0] - A1r[0][0]) * (z0 ? gb0 : ga0) + (acc[1] - A1r[0][1]) * (z1 ? gb0 : ga0);
                    pw[16 * i + gid + 8] =
                        (acc[2] - A1r[1][0]) * (z0 ? gb1 : ga1) + (acc[3] - A1r[1][1]) * (z1 ? gb1 : ga1);
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(empty_bar(slot));
                mbar_arrive(pfull_bar(pb));
            }
            ++s;
        }
    } else {
    const int gw = warp & (kDecGroups - 1), ph = warp / kDecGroups;   // group of the chunk, first tile
    constexpr int TS = CW / kDecGroups;                                // tile stride
    const int hlf = gw >> 2, wq = gw & 3;
    uint32_t b[NT][8];
    float A1a[H], A1b[H], F[H];
    const uint32_t my_bst = s_bst + (uint32_t)(warp * 32 * NT * 8) * 4u;
    int* my_est = est + warp * 16;
    bool waited = false;

    // Stage group g of the activation into this warp's B registers.
    auto stage_x = [&](int g) {
        // clear this lane's staging words (absent tokens and terms stay 0)
#pragma unroll
        for (int q = 0; q < NT * 8; q += 4)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(my_bst + (uint32_t)(lane * NT * 8 + q) * 4u),
                         "r"(0u)
                         : "memory");
        __syncwarp();
        const int tq = lane >> 3, hh = (lane >> 2) & 1, bb = lane & 3;   // target t, half, byte
        for (int m = 0; m < M; ++m) {
            const uint2 raw = *reinterpret_cast<const uint2*>(a.x + (size_t)m * a.K + (size_t)g * kDecGroup + 4 * lane);
            float f[4];
            f[0] = __uint_as_float(raw.x << 16);
            f[1] = __uint_as_float(raw.x & 0xFFFF0000u);
            f[2] = __uint_as_float(raw.y << 16);
            f[3] = __uint_as_float(raw.y & 0xFFFF0000u);
            float mx = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const int be = (int)(__float_as_uint(mx) >> 23);   // mx >= 0
            const int E = min(127, 141 - be);                   // mx 2^E < 2^15
            if (lane == 0) my_est[m] = E;
            const float fe = __uint_as_float((uint32_t)(E + 127) << 23);
            const float fo = __uint_as_float((uint32_t)(E + 125) << 23);
            float t0[4], t1[4], t2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = f[e] * ((e & 1) ? fo : fe);
                t0[e] = trunc3(v);
                const float r1 = v - t0[e];
                t1[e] = trunc3(r1);
                t2[e] = r1 - t1[e];
            }
            const int h = m >> 2, tm = m & 3;
#pragma unroll
            for (int tau = 0; tau < 3; ++tau) {
                const float* tv = tau == 0 ? t0 : tau == 1 ? t1 : t2;
                const int i = 3 * h + tau, j = i >> 1, col = 2 * tm + (i & 1);
                const uint32_t p01 = cvt_e5m2x2(tv[0], tv[1]);   // hi = value 0, lo = value 1
                const uint32_t p23 = cvt_e5m2x2(tv[2], tv[3]);
                const uint32_t base =
                    my_bst + (uint32_t)(((col * 4 + tq) * NT + j) * 8) * 4u + (uint32_t)hh * 4u + (uint32_t)bb;
                sts_u8(base + 0u * 8u, p01 >> 8);   // MMA c = 0: register 2c + hh
                sts_u8(base + 1u * 8u, p01);        // c = 1
                sts_u8(base + 2u * 8u, p23 >> 8);   // c = 2
                sts_u8(base + 3u * 8u, p23);        // c = 3
            }
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const uint32_t ad = my_bst + (uint32_t)((lane * NT + j) * 8) * 4u;
            uint4 lo, hi;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w) : "r"(ad));
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                         : "r"(ad + 16u));
            b[j][0] = lo.x; b[j][1] = lo.y; b[j][2] = lo.z; b[j][3] = lo.w;
            b[j][4] = hi.x; b[j][5] = hi.y; b[j][6] = hi.z; b[j][7] = hi.w;
        }
        // the all-ones chains: the -1 of q - 1 with the products' own rounding
        float acc1[1][NT][4];
        const uint32_t ones[1][4] = {{0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u}};
        unit_chains<1, NT>(acc1, ones, b);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int m = 4 * h + t;
            const int i0 = 3 * h, i1 = 3 * h + 1, i2 = 3 * h + 2;
            A1a[h] = (acc1[0][i0 >> 1][i0 & 1] + acc1[0][i1 >> 1][i1 & 1]) + acc1[0][i2 >> 1][i2 & 1];
            A1b[h] = (acc1[0][i0 >> 1][2 + (i0 & 1)] + acc1[0][i1 >> 1][2 + (i1 & 1)]) + acc1[0][i2 >> 1][2 + (i2 & 1)];
            F[h] = m < M ? __uint_as_float((uint32_t)(9 - my_est[m] + 127) << 23) : 0.0f;   // 2^(9 - E)
        }
        __syncwarp();   // the staging words are read before the next segment clears them
    };

    // one unit's rows into the partial buffer (rows rbase + gid, rbase + gid + 8)
    auto epilogue = [&](const float (&acc)[NT][4], float s0, float s1, float* pw, int rbase) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int m = 4 * h + t;
            const int i0 = 3 * h, i1 = 3 * h + 1, i2 = 3 * h + 2;
            const float c0 = (acc[i0 >> 1][i0 & 1] + acc[i1 >> 1][i1 & 1]) + acc[i2 >> 1][i2 & 1];
            const float c1 = (acc[i0 >> 1][2 + (i0 & 1)] + acc[i1 >> 1][2 + (i1 & 1)]) + acc[i2 >> 1][2 + (i2 & 1)];
            if (m < M) {
                pw[(rbase + gid) * a.mpad + m] = (c0 - A1a[h]) * (s0 * F[h]);
                pw[(rbase + gid + 8) * a.mpad + m] = (c1 - A1b[h]) * (s1 * F[h]);
            }
        }
    };

    // this lane's words of a tile: rows gid and gid + 8, words 2t, 2t+1 of
    // group w (128-byte swizzle: 16-byte chunk index ^ (row & 7))
    const uint32_t lane_off =
        (uint32_t)(hlf * 2048 + gid * 128 + (((2 * wq + (t >> 1)) ^ gid) << 4) + 8 * (t & 1));
    StageWalk wk(L0, L1, a.T, U);
    int s = 0, cur_kc = -1;
    while (wk.next()) {
        if (wk.kc != cur_kc) {
            if (!waited) {
                pdl_wait();   // x may be the previous kernel's output
                waited = true;
            }
            stage_x(kDecGroups * wk.kc + gw);
            cur_kc = wk.kc;
        }
        const int slot = s % D, pb = s % PB;
        if (!warp_wait(full_bar(slot), (uint32_t)(s / D) & 1u, abort_flag, lane) ||
            (s >= PB && !warp_wait(pempty_bar(pb), (uint32_t)((s / PB) - 1) & 1u, abort_flag, lane))) {
            fail(TERN_DEVERR_DECODE_CONSUMER_WAIT);
            return;
        }
        float* pw = part + (size_t)pb * a.part_floats + (size_t)gw * 16 * U * a.mpad;
        const unsigned char* cs = smem + (size_t)slot * U * kDecTileCodeBytes + lane_off;
        const unsigned char* ss = smem + a.off_scl + (size_t)slot * U * kDecTileScaleBytes + gid * 16 + 2 * gw;
        // this warp's tiles ph, ph + TS, ...: NB at a time (interleaved chains),
        // then one at a time for the rest
        auto run_units = [&](auto nb_c, int i0) {
            constexpr int NB = decltype(nb_c)::value;
            uint32_t wv[NB][4];
            float s0[NB], s1[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int ti = i0 + u * TS;
                const uint2 ra = *reinterpret_cast<const uint2*>(cs + ti * kDecTileCodeBytes);
                const uint2 rb = *reinterpret_cast<const uint2*>(cs + ti * kDecTileCodeBytes + 1024);
                wv[u][0] = ra.x;
                wv[u][1] = ra.y;
                wv[u][2] = rb.x;
                wv[u][3] = rb.y;
                s0[u] = __half2float(*reinterpret_cast<const __half*>(ss + ti * kDecTileScaleBytes));
                s1[u] = __half2float(*reinterpret_cast<const __half*>(ss + ti * kDecTileScaleBytes + 128));
            }
            float acc[NB][NT][4];
            unit_chains<NB, NT>(acc, wv, b);
#pragma unroll
            for (int u = 0; u < NB; ++u) epilogue(acc[u], s0[u], s1[u], pw, 16 * (i0 + u * TS));
        };
        constexpr int NB = DecCfg<H>::NB;
        int i = ph;
#pragma unroll 1
        for (; i + (NB - 1) * TS < wk.n; i += NB * TS) run_units(std::integral_constant<int, NB>{}, i);
        if (NB > 1) {
#pragma unroll 1
            for (; i < wk.n; i += TS) run_units(std::integral_constant<int, 1>{}, i);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(empty_bar(slot));
            mbar_arrive(pfull_bar(pb));
        }
        ++s;
    }
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 dec_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// codes [N][K/16] uint32: boxes of 32 words x 16 rows, 128-byte swizzle;
// scales [N][G] fp16: boxes of 8 x 16 rows.
bool dec_maps(CUtensorMap* mc, CUtensorMap* ms, const uint32_t* codes, const void* scales, int N, int K) {
    auto enc = dec_encode_fn();
    if (!enc) return false;
    const int G = K / kDecGroup;
    {
        cuuint64_t gdim[2] = {(cuuint64_t)(K / 16), (cuuint64_t)N};
        cuuint64_t gstride[1] = {(cuuint64_t)K / 4};
        cuuint32_t box[2] = {32, 16};
        cuuint32_t es[2] = {1, 1};
        if (enc(mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t gdim[2] = {(cuuint64_t)G, (cuuint64_t)N};
        cuuint64_t gstride[1] = {(cuuint64_t)G * 2};
        cuuint32_t box[2] = {8, 16};
        cuuint32_t es[2] = {1, 1};
        if (enc(ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(scales), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

inline size_t dec_align(size_t v, size_t al) { return (v + al - 1) / al * al; }

// floats per partial row: conflict-free stores of the 8 x 4 lanes of a warp
int dec_mpad(int M) { return M <= 4 ? M : M <= 12 ? 12 : 20; }

// Shared-memory layout of one CTA (offsets from the 1024-aligned base).
template <int H>
size_t dec_layout(DecArgs& a) {
    constexpr int NT = dec_nt<H>();
    constexpr int U = DecCfg<H>::U, D = DecCfg<H>::D;
    size_t off = (size_t)D * U * kDecTileCodeBytes;
    a.off_scl = (uint32_t)off;
    off += (size_t)D * U * kDecTileScaleBytes;
    a.off_part = (uint32_t)dec_align(off, 16);
    a.part_floats = (uint32_t)(dec_slots<H>() * 16 * U * a.mpad);
    off = a.off_part + (size_t)DecCfg<H>::PB * a.part_floats * 4;
    a.off_bst = (uint32_t)dec_align(off, 16);
    off = a.off_bst + (size_t)DecCfg<H>::CW * 32 * NT * 8 * 4;
    a.off_est = (uint32_t)off;
    off += (size_t)DecCfg<H>::CW * 16 * 4;
    a.off_bar = (uint32_t)dec_align(off, 8);
    off = a.off_bar + 8 * (2 * D + 2 * DecCfg<H>::PB) + 16;
    return off + 1024;   // alignment slack of the dynamic base
}

template <int H>
cudaError_t dec_prepare(int dev, size_t smem) {
    static size_t set_for[64] = {};
    if (set_for[dev] >= smem) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(decode_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) set_for[dev] = smem;
    return e;
}

template <int H>
tern_status dec_launch(const CUtensorMap& mc1, const CUtensorMap& ms1, const CUtensorMap& mc2, const CUtensorMap& ms2,
                       DecArgs a, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TERN_ERR_CUDA;
    const size_t smem = dec_layout<H>(a);
    if (smem > 227 * 1024) return TERN_ERR_SHAPE;
    {
        static std::mutex mu;
        std::lock_guard<std::mutex> lk(mu);
        if (dec_prepare<H>(dev, smem) != cudaSuccess) return TERN_ERR_CUDA;
    }
    const cudaError_t e =
        launch_pdl(decode_kernel<H>, dim3(a.P), dim3(dec_threads<H>()), smem, stream, true, mc1, ms1, mc2, ms2, a);
    return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

}  // namespace

// Workspace of the FP8 decode product: one flag word per 16-row tile when K
// spans several chunks (zero between calls).
size_t decode_workspace_bytes(int M, int T, int K) {
    (void)M;
    if (K / kDecGroup <= kDecGroups) return 0;
    return dec_align((size_t)T * 4, 256);
}

bool decode_supported(int K) { (void)K; return false; }   // the f16 mma.sync kernel is faster on sm_103a

// y1 = x W1^T (and y2 = x W2^T for a pair call, N2 > 0) with the FP8 decode
// kernel.  Shapes and pointers are validated by the caller; K % 1024 == 0.
tern_status decode_run(const void* x, const uint32_t* codes1, const void* scales1, float* y1, int N1,
                       const uint32_t* codes2, const void* scales2, float* y2, int N2, int M, int K, void* workspace,
                       size_t workspace_bytes, int sms, cudaStream_t stream) {
    DecArgs a{};
    a.x = reinterpret_cast<const __nv_bfloat16*>(x);
    a.y1 = y1;
    a.y2 = N2 > 0 ? y2 : y1;
    a.M = M;
    a.N1 = N1;
    a.N2 = N2;
    a.K = K;
    a.G = K / kDecGroup;
    a.S = a.G / kDecGroups;
    a.T1 = (N1 + 15) / 16;
    a.T = a.T1 + (N2 + 15) / 16;
    a.L = (long long)a.S * a.T;
    a.P = (int)std::min<long long>(sms, a.L);
    a.mpad = dec_mpad(M);
    const size_t need = decode_workspace_bytes(M, a.T, K);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return TERN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
        a.cnt = reinterpret_cast<unsigned*>(workspace);
    }
    CUtensorMap mc1, ms1, mc2, ms2;
    if (!dec_maps(&mc1, &ms1, codes1, scales1, N1, K)) return TERN_ERR_CUDA;
    if (N2 > 0) {
        if (!dec_maps(&mc2, &ms2, codes2, scales2, N2, K)) return TERN_ERR_CUDA;
    } else {
        mc2 = mc1;
        ms2 = ms1;
    }
    const int H = (M + 3) / 4;
    if (M == 1) return dec_launch<0>(mc1, ms1, mc2, ms2, a, stream);
    switch (H) {
        case 1: return dec_launch<1>(mc1, ms1, mc2, ms2, a, stream);
        case 2: return dec_launch<2>(mc1, ms1, mc2, ms2, a, stream);
        case 3: return dec_launch<3>(mc1, ms1, mc2, ms2, a, stream);
        default: return dec_launch<4>(mc1, ms1, mc2, ms2, a, stream);
    }
}

// Reads and clears the decode product's device error word.
cudaError_t read_decode_device_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int z = 0;
        e = cudaMemcpyToSymbol(g_decode_error, &z, sizeof(int));
        if (e != cudaSuccess) return e;
    }
    *code = v;
    return cudaSuccess;
}

}  // namespace tern
