// tern_gemm.cu -- prefill ternary-g128 product on the tcgen05 tensor cores.
//
//   y[m][n] = sum_k x[m][k] * t[n][k] * s[n][k/128]
//
// ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card: ternary g128 weights,
// "Weight representation"; the packed codes are unpacked and scaled inside the
// matrix product and never expanded to a dense tensor in memory, "CUDA (NVIDIA
// GPUs)"; pp512 prompt processing is the compute-bound phase, "Cross-platform
// throughput".)
//
// Design.  The product is computed as y^T = W x^T so that the unpacked weights
// are the MMA's A operand and can live in tensor memory:
//   * a TMA producer warp streams, per 64-wide K stage, the x tile (256 tokens
//     x 64, bf16, 128-byte swizzle: the MMA's B operand, K-major) and the
//     packed code tile (128 weight rows x 4 words) into a shared-memory ring;
//   * eight unpack warps turn each code into bf16 t * bf16(s_g) in registers
//     (shift + mask puts two codes into bf16 exponent bits, one bf16x2 FMA gives
//     q - 1 exactly, one bf16x2 multiply applies the scale, one byte permute
//     pairs neighbouring k) and store them with tcgen05.st straight into a
//     tensor-memory slot: the weights never touch shared or global memory in
//     unpacked form;
//   * one thread issues tcgen05.mma kind::f16 (M = 128 weight rows, N = 256
//     tokens, K = 16) with A from tensor memory and B from shared memory,
//     accumulating fp32 in tensor memory;
//   * four epilogue warps read the accumulator with tcgen05.ld and store y
//     (fp32 or bf16) with coalesced stores along n.
// The 1-bit sibling format (w = (2b - 1) s) runs the same kernel: its code box
// is 16 bytes per row too, but spans two K stages (starting at the even one, so
// the TMA x coordinate stays 16-byte aligned), and the unpack turns bits j and
// j + 16 of a word into bf16 2b - 1 with one shift and one FMA.
// An affine pack (w = s q + b per group, every 2-bit code valid) runs it too
// (gemm_kernel<true>): per row and group the four weights s q + b are formed
// in fp32 and rounded once to bf16, and each pair of codes picks its two
// weights from that table with one byte permute.
// Scheduling takes whole tiles on a persistent grid, or stream-K where whole
// tiles would leave SMs idle longer than stream-K's tail costs: the (tile,
// 64-wide K stage) iterations, tile-major, are cut into one equal contiguous
// share per CTA, so no SM idles behind a partial last wave.  A CTA's share is a run of segments, each a stretch of
// one tile's K stages; a CTA runs its (at most two) partial segments first and
// its whole tiles after.  A segment that covers its whole tile is written to y
// directly.  A partial one adds its fp32 accumulator into the tile's fp32 sum
// in the workspace with vector reductions, fences and counts itself into the
// tile's counter (one per epilogue warp's 32 rows); the CTA that counts last
// reads the sum, writes y and clears the sum and the counter.  No CTA or warp
// waits for another; the partial sums meet in no fixed order.
// Stage hand-offs use mbarriers (TMA transaction counts, thread arrivals and
// tcgen05.commit).  Every wait is bounded: after a second it raises a CTA abort
// flag and the device error word, every role drains what it issued, tensor
// memory is freed and the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "tern_sm100.cuh"

namespace tern {
namespace {

__device__ int g_gemm_error;

constexpr int kBM = 128;                    // weight rows per tile (tensor-memory lanes)
constexpr int kBN = 256;                    // tokens per tile (MMA N)
constexpr int kBK = 64;                     // K per stage
constexpr int kStages = 6;                  // K stages in flight (34 KB of shared memory each)
constexpr int kXStageBytes = kBN * kBK * 2; // 32 KB
constexpr int kCStageBytes = kBM * kBK / 4; // 2 KB of codes
constexpr int kNumWarps = 14;               // 0 TMA, 1 MMA, 2-5 epilogue, 6-13 unpack
constexpr int kThreads = kNumWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kTmemD = 0;                   // accumulator: columns [0, 256)
constexpr int kTmemA = 256;                 // weight slots: 32 columns per stage
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s
constexpr uint32_t kIdesc = sm100::idesc_bf16_f32(kBM, kBN);

constexpr size_t kSmemX = 0;
constexpr size_t kSmemC = kSmemX + (size_t)kStages * kXStageBytes;
constexpr size_t kSmemBar = kSmemC + (size_t)kStages * kCStageBytes;
// barriers: full[S], afull[S], empty[S], dfull, dempty, drain; then tmem base and abort flag
constexpr size_t kSmemMisc = kSmemBar + (size_t)(3 * kStages + 3) * 8;
constexpr size_t kSmemBytes = kSmemMisc + 16 + 1024;   // + alignment slack

constexpr int kMaxCtas = 160;                 // stream-K shares (the grid) at most
constexpr int kTileFloats = kBM * kBN;         // one tile's fp32 sum: [256 tokens / 4][128 rows][4]

struct GemmArgs {
    const __half* scales;
    const __half* biases;       // an affine pack's [N][K/128] biases, else null
    void* y;
    float* sums;                // [tiles][kTileFloats] fp32 sums of split tiles, 0 between calls
    unsigned* counters;         // [tiles][4 lane quadrants], 0 between calls
    int stream_k;               // 0: whole tiles blockIdx.x, + gridDim.x, ...; 1: stream-K shares
    int y_is_bf16;
    int bin;                    // 1: the 1-bit layout (words [N][K/32]), else 2-bit codes [N][K/16]
    int M, N, K;
};

// The stream-K share of CTA c: iterations [T c / P, T (c + 1) / P).
__host__ __device__ inline long long share_begin(long long T, int P, int c) { return T * c / P; }
// The CTA whose share holds iteration g.
__device__ inline int share_of(long long T, int P, long long g) {
    int c = (int)((g * P) / T);
    while (c + 1 < P && share_begin(T, P, c + 1) <= g) ++c;
    while (c > 0 && share_begin(T, P, c) > g) --c;
    return c;
}
// Segment s of the share [g0, g1): its tile and K stages [ks0, ks1).  The
// share's first and last tiles (the partial ones) come first, then the whole
// tiles between them in order.
struct Segment {
    int tile, ks0, ks1;
};
__device__ inline int segment_count(long long g0, long long g1, int KS) {
    if (g1 <= g0) return 0;   // (whole-tile schedule: see the kernel)
    const int t0 = (int)(g0 / KS), t1 = (int)((g1 - 1) / KS);
    return t1 - t0 + 1;
}
__device__ inline Segment segment_at(long long g0, long long g1, int KS, int s) {
    const int t0 = (int)(g0 / KS), t1 = (int)((g1 - 1) / KS);
    const int first_lo = (int)(g0 - (long long)t0 * KS);
    const int last_hi = (int)(g1 - (long long)t1 * KS);
    if (s == 0) return Segment{t0, first_lo, t0 == t1 ? last_hi : KS};
    if (s == 1) return Segment{t1, 0, last_hi};
    return Segment{t0 + s - 1, 0, KS};   // s >= 2: whole tiles t0 + 1 .. t1 - 1
}
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// 16 codes of one word -> 8 bf16 pairs (k, k+1) of t * s.
// Codes j and j + 8 sit 16 bits apart, so one shift puts both into bit 7 of
// their halves (the bf16 exponent's low bits): the halves read as q * 2^-126,
// and fma(., 2^126, -1) = q - 1 exactly.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t s2, uint32_t (&o)[8]) {
    constexpr uint32_t kTwo126 = 0x7E807E80u;   // bf16 2^126, both halves
    constexpr uint32_t kMinus1 = 0xBF80BF80u;   // bf16 -1, both halves
    uint32_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t m = (j <= 3 ? (w << (7 - 2 * j)) : (w >> (2 * j - 7))) & 0x01800180u;
        v[j] = bf16x2_mul(bf16x2_fma(m, kTwo126, kMinus1), s2);   // (w_j, w_{j+8})
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        o[p] = prmt(v[2 * p], v[2 * p + 1], 0x5410u);       // (w_{2p},   w_{2p+1})
        o[p + 4] = prmt(v[2 * p], v[2 * p + 1], 0x7632u);   // (w_{2p+8}, w_{2p+9})
    }
}

// 32 weights of one word of the 1-bit layout -> 16 bf16 pairs (k, k+1) of
// (2b - 1) * s.  Bits j and j + 16 sit 16 bits apart, so one shift puts both
// at bit 7 of their halves (the bf16 exponent's low bit): the halves read as
// b * 2^-126, and fma(., 2^127, -1) = 2b - 1 exactly.
__device__ __forceinline__ void unpack_word_bin(uint32_t w, uint32_t s2, uint32_t (&o)[16]) {
    constexpr uint32_t kTwo127 = 0x7F007F00u;   // bf16 2^127, both halves
    constexpr uint32_t kMinus1 = 0xBF80BF80u;   // bf16 -1, both halves
    uint32_t v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t m = (j <= 7 ? (w << (7 - j)) : (w >> (j - 7))) & 0x00800080u;
        v[j] = bf16x2_mul(bf16x2_fma(m, kTwo127, kMinus1), s2);   // (w_j, w_{j+16})
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        o[p] = prmt(v[2 * p], v[2 * p + 1], 0x5410u);       // (w_{2p},    w_{2p+1})
        o[p + 8] = prmt(v[2 * p], v[2 * p + 1], 0x7632u);   // (w_{2p+16}, w_{2p+17})
    }
}

// 16 codes of one word of an affine pack -> 8 bf16 pairs (k, k+1) of s q + b,
// looked up in the group's table: lo holds the low bytes of the bf16 weights
// of codes 0..3 (byte q for code q) and hi their high bytes.  Codes j and
// j + 4 sit 8 bits apart, so one shift and mask leave q_j in bits 0-1 and
// q_{j+4} in bits 8-9, and one multiply-add by 0x11, 0x4040 turns that into
// the byte selector [q_j, 4 + q_j, q_{j+4}, 4 + q_{j+4}]: one byte permute
// then gives the pair (w_j, w_{j+4}), at four operations per two weights like
// the ternary unpack.
__device__ __forceinline__ void unpack_word_affine(uint32_t w, uint32_t lo, uint32_t hi, uint32_t (&o)[8]) {
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int j = i < 4 ? i : i + 4;                       // codes j and j + 4: 0-3 and 8-11
        const uint32_t m = (w >> (2 * j)) & 0x0303u;
        v[i] = prmt(lo, hi, m * 0x11u + 0x4040u);             // (w_j, w_{j+4})
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // v[4h + r] = (w_{8h+r}, w_{8h+r+4})
        o[4 * h] = prmt(v[4 * h], v[4 * h + 1], 0x5410u);       // (w_{8h},   w_{8h+1})
        o[4 * h + 1] = prmt(v[4 * h + 2], v[4 * h + 3], 0x5410u); // (w_{8h+2}, w_{8h+3})
        o[4 * h + 2] = prmt(v[4 * h], v[4 * h + 1], 0x7632u);   // (w_{8h+4}, w_{8h+5})
        o[4 * h + 3] = prmt(v[4 * h + 2], v[4 * h + 3], 0x7632u); // (w_{8h+6}, w_{8h+7})
    }
}

// The table of one group of an affine pack: w_q = s q + b in fp32, rounded
// once to bf16; lo gets the four low bytes (byte q of w_q) and hi the four
// high bytes.
__device__ __forceinline__ void affine_table(unsigned short s16, unsigned short b16, uint32_t& lo, uint32_t& hi) {
    const float sf = __half2float(__ushort_as_half(s16)), bf = __half2float(__ushort_as_half(b16));
    const __nv_bfloat162 l = __floats2bfloat162_rn(bf, sf + bf);                         // w_0, w_1
    const __nv_bfloat162 h = __floats2bfloat162_rn(fmaf(sf, 2.0f, bf), fmaf(sf, 3.0f, bf)); // w_2, w_3
    const uint32_t l32 = *reinterpret_cast<const uint32_t*>(&l), h32 = *reinterpret_cast<const uint32_t*>(&h);
    lo = prmt(l32, h32, 0x6420u);
    hi = prmt(l32, h32, 0x7531u);
}

// AFF: an affine pack (a compile-time switch, so that the other layouts'
// unpack loop carries no trace of it).
template <bool AFF>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_c,
            const GemmArgs a) {
    using namespace sm100;
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + (uint32_t)kSmemBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto afull_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    const uint32_t dfull_bar = bar0 + 8u * (3 * kStages);
    const uint32_t dempty_bar = dfull_bar + 8u;
    const uint32_t drain_bar = dfull_bar + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, N = a.N, K = a.K;
    const int G = K / 128;
    const int KS = K / kBK;
    const int m_tiles = (M + kBN - 1) / kBN;
    const int n_tiles = (N + kBM - 1) / kBM;
    const int total = m_tiles * n_tiles;
    const long long TI = (long long)total * KS;   // stream-K iterations
    const int P = gridDim.x;
    const long long g0 = share_begin(TI, P, blockIdx.x), g1 = share_begin(TI, P, blockIdx.x + 1);
    // whole-tile schedule: tiles blockIdx.x, blockIdx.x + P, ...; stream-K: the share's segments
    const int nseg = a.stream_k ? segment_count(g0, g1, KS) : (total - (int)blockIdx.x + P - 1) / P;
    auto segment = [&](int sg) -> Segment {
        return a.stream_k ? segment_at(g0, g1, KS, sg) : Segment{(int)blockIdx.x + sg * P, 0, KS};
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(afull_bar(s), 8);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(dfull_bar, 1);
        mbar_init(dempty_bar, 4);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_c);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // x may be the previous kernel's output
    pdl_wait();

    auto fail = [&](int code) {
        if (!*abort_flag) {
            *abort_flag = 1;
            report_device_error(&g_gemm_error, code);
        }
    };

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int sg = 0; sg < nseg && ok; ++sg) {
                const Segment seg = segment(sg);
                const int tile = seg.tile, ks0 = seg.ks0, ks1 = seg.ks1;
                const int nt = tile / m_tiles, mt = tile - nt * m_tiles;
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kWaitLimitNs)) {
                        fail(kDevErrGemmProducerWait);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), kXStageBytes + kCStageBytes);
                    tma_load_2d(sbase + (uint32_t)(kSmemX + (size_t)s * kXStageBytes), &tmap_x, ks * kBK, mt * kBN,
                                full_bar(s));
                    // the 1-bit layout: a 16-byte box of 128 weights per row (two
                    // stages), starting at the even stage so that x stays 16-byte aligned
                    tma_load_2d(sbase + (uint32_t)(kSmemC + (size_t)s * kCStageBytes), &tmap_c,
                                a.bin ? (ks & ~1) * (kBK / 32) : ks * (kBK / 16), nt * kBM, full_bar(s));
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA goes away
                const uint32_t n = it < (uint32_t)kStages ? it : (uint32_t)kStages;
                for (uint32_t i = 0; i < n; ++i) {
                    const uint32_t k = it - 1 - i;
                    (void)mbar_wait_drain(full_bar(k % kStages), (k / kStages) & 1u, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            for (int sg = 0; sg < nseg && ok; ++sg, ++tc) {
                const Segment seg = segment(sg);
                const int ks0 = seg.ks0, ks1 = seg.ks1;
                if (!mbar_wait_bounded(dempty_bar, (tc & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    fail(kDevErrGemmMmaWait);
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, kWaitLimitNs) ||
                        !mbar_wait_bounded(afull_bar(s), ph, abort_flag, kWaitLimitNs)) {
                        fail(kDevErrGemmMmaWait);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_k_sw128(sbase + (uint32_t)(kSmemX + (size_t)s * kXStageBytes));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // A: 8 columns (16 bf16) per K=16 step; B: advance 32 bytes inside the swizzle atom
                        mma_f16_ts(tmem + kTmemD, tmem + kTmemA + 32u * s + 8u * kk, bdesc + (uint64_t)(2 * kk),
                                   kIdesc, (ks != ks0 || kk != 0) ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit(empty_bar(s));
                }
                if (!ok) break;
                mma_commit(dfull_bar);
            }
            if (!ok && issued) {
                // wait for every MMA issued so far before tensor memory is freed
                mma_commit(drain_bar);
                (void)mbar_wait_drain(drain_bar, 0u, 100000000ull);
            }
        }
    } else if (warp < 6) {
        // ------------------------------ epilogue ------------------------------
        const int q = warp & 3;
        const int rl = q * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + kTmemD;
        uint32_t tc = 0;
        for (int sg = 0; sg < nseg; ++sg, ++tc) {
            const Segment seg = segment(sg);
            const int tile = seg.tile, ks0 = seg.ks0, ks1 = seg.ks1;
            const int nt = tile / m_tiles, mt = tile - nt * m_tiles;
            const int row = nt * kBM + rl;
            if (!mbar_wait_bounded(dfull_bar, tc & 1u, abort_flag, kWaitLimitNs)) {
                fail(kDevErrGemmEpilogueWait);
                break;
            }
            tc_fence_after();
            auto put = [&](int m, float v) {
                if (a.y_is_bf16)
                    reinterpret_cast<__nv_bfloat16*>(a.y)[(size_t)m * N + row] = __float2bfloat16_rn(v);
                else
                    reinterpret_cast<float*>(a.y)[(size_t)m * N + row] = v;
            };
            if (ks0 == 0 && ks1 == KS) {
                // the whole tile: straight to y
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_x32(trow + 32u * c, v);
                    tmem_ld_wait();
                    if (c == kBN / 32 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dempty_bar);
                    }
                    if (row < N) {
                        const int m0 = mt * kBN + 32 * c;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (m0 + i < M) put(m0 + i, __uint_as_float(v[i]));
                    }
                }
                continue;
            }
            // part of the tile: add the accumulator into the tile's fp32 sum (laid out
            // [token / 4][row][4], so a warp's lanes cover 512 contiguous bytes)
            float* sum = a.sums + (size_t)tile * kTileFloats;
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t v[32];
                tmem_ld_x32(trow + 32u * c, v);
                tmem_ld_wait();
                if (c == kBN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dempty_bar);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    red_add_v4(sum + ((size_t)(8 * c + i) * kBM + rl) * 4, __uint_as_float(v[4 * i]),
                               __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                               __uint_as_float(v[4 * i + 3]));
            }
            // each warp counts its own 32 rows (one counter per tile and lane
            // quadrant), so the four warps never wait for one another
            __threadfence();
            __syncwarp();
            const int c_lo = share_of(TI, P, (long long)tile * KS), c_hi = share_of(TI, P, (long long)tile * KS + KS - 1);
            unsigned last = 0;
            if (lane == 0) last = atomicAdd(a.counters + 4 * tile + q, 1u) == (unsigned)(c_hi - c_lo);
            if (!__shfl_sync(0xffffffffu, last, 0)) continue;
            // the last of the tile's CTAs for these rows: the sum is complete
            __threadfence();
            for (int c = 0; c < kBN / 64; ++c) {
                float4 t[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    t[i] = __ldcg(reinterpret_cast<const float4*>(sum + ((size_t)(16 * c + i) * kBM + rl) * 4));
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    __stcg(reinterpret_cast<float4*>(sum + ((size_t)(16 * c + i) * kBM + rl) * 4),
                           make_float4(0.0f, 0.0f, 0.0f, 0.0f));
                    const int m0 = mt * kBN + 64 * c + 4 * i;
                    if (row < N) {
                        if (m0 < M) put(m0, t[i].x);
                        if (m0 + 1 < M) put(m0 + 1, t[i].y);
                        if (m0 + 2 < M) put(m0 + 2, t[i].z);
                        if (m0 + 3 < M) put(m0 + 3, t[i].w);
                    }
                }
            }
            if (lane == 0) a.counters[4 * tile + q] = 0u;
        }
    } else {
        // ------------------------------ unpack ------------------------------
        const int q = warp & 3;             // tensor-memory lane quadrant
        const int h = (warp - 6) >> 2;      // K half of the stage: 0 -> k 0..31, 1 -> k 32..63
        const int rl = q * 32 + lane;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + kTmemA + 16u * h;
        constexpr bool aff = AFF;
        uint32_t it = 0;
        bool ok = true;
        for (int sg = 0; sg < nseg && ok; ++sg) {
            const Segment seg = segment(sg);
            const int tile = seg.tile, ks0 = seg.ks0, ks1 = seg.ks1;
            const int nt = tile / m_tiles;
            const int row = nt * kBM + rl;
            const __half* srow = a.scales + (size_t)(row < N ? row : 0) * G;
            const __half* brow = aff ? a.biases + (size_t)(row < N ? row : 0) * G : srow;
            uint32_t s2 = 0, lut_lo = 0, lut_hi = 0;
            // the segment's first group scale (and bias), then each next one a group ahead
            unsigned short s_next = row < N ? __half_as_ushort(__ldg(srow + (ks0 >> 1))) : (unsigned short)0;
            unsigned short b_next = aff && row < N ? __half_as_ushort(__ldg(brow + (ks0 >> 1))) : (unsigned short)0;
            for (int ks = ks0; ks < ks1; ++ks, ++it) {
                if (ks == ks0 || (ks & 1) == 0) {
                    // this group's scale as a bf16 pair; fetch the next group's
                    if constexpr (AFF) {
                        affine_table(s_next, b_next, lut_lo, lut_hi);
                    } else {
                        const float sf = __half2float(__ushort_as_half(s_next));
                        const __nv_bfloat16 sb = __float2bfloat16_rn(sf);
                        const uint32_t sbits = __bfloat16_as_ushort(sb);
                        s2 = sbits | (sbits << 16);
                    }
                    const int gn = (ks >> 1) + 1;
                    if (gn < G && row < N) {
                        s_next = __half_as_ushort(__ldg(srow + gn));
                        if (aff) b_next = __half_as_ushort(__ldg(brow + gn));
                    }
                }
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                // the MMAs of this slot's previous round are done (tensor-memory slot free)
                // and this round's codes have landed
                if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kWaitLimitNs) ||
                    !mbar_wait_bounded(full_bar(s), ph, abort_flag, kWaitLimitNs)) {
                    fail(kDevErrGemmUnpackWait);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned char* crow = smem + kSmemC + (size_t)s * kCStageBytes + (size_t)rl * 16;
                uint32_t o[16];
                if (a.bin) {
                    // word (ks odd ? 2 : 0) + h of the row's two-stage box
                    unpack_word_bin(*reinterpret_cast<const uint32_t*>(crow + 8 * (ks & 1) + 4 * h), s2, o);
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(crow + 8 * h);
                    uint32_t o0[8], o1[8];
                    if (aff) {
                        unpack_word_affine(w.x, lut_lo, lut_hi, o0);
                        unpack_word_affine(w.y, lut_lo, lut_hi, o1);
                    } else {
                        unpack_word(w.x, s2, o0);
                        unpack_word(w.y, s2, o1);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        o[i] = o0[i];
                        o[8 + i] = o1[i];
                    }
                }
                tmem_st_x16(tbase + 32u * s, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(s));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps through the driver entry point (no libcuda link).
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t gdim[2] = {inner, outer};
    cuuint64_t gstride[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t read_gemm_device_error(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemm_error, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
}

// Two roles of a CTA waiting on mbarriers that nobody arrives at, as the
// prefill roles wait on each other: warp 0's wait runs out after limit_ns, it
// raises the CTA's abort flag and reports; warp 1, in a wait with the products'
// own 1 s limit, sees the flag and returns at once instead of running out.
__global__ void __launch_bounds__(64) mbar_wait_selftest_kernel(uint64_t limit_ns) {
    using namespace sm100;
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ volatile int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (lane == 0 && !mbar_wait_bounded(smem_u32(&bars[warp]), 0u, &abort_flag, warp == 0 ? limit_ns : kWaitLimitNs) &&
        !abort_flag) {
        abort_flag = 1;
        report_device_error(&g_gemm_error, kDevErrGemmMmaWait);
    }
}
cudaError_t launch_mbar_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    mbar_wait_selftest_kernel<<<1, 64, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace tern

using namespace tern;

// Workspace: [counters: tiles x 4 uint32, 256-byte aligned | fp32 sums: one
// kBN x kBM tile per output tile].  The grid never exceeds kMaxCtas shares nor
// the number of iterations.
namespace tern {
namespace {
int gemm_tiles(int M, int N) { return ((M + kBN - 1) / kBN) * ((N + kBM - 1) / kBM); }
int gemm_shares(int M, int N, int K, int sms) {
    const long long it = (long long)gemm_tiles(M, N) * (K / kBK);
    long long p = sms < kMaxCtas ? sms : kMaxCtas;
    if (p > it) p = it;
    return (int)p;
}
// Stream-K pays for its split tiles with a tail: the fp32 sums' reductions,
// the fence and the last CTA's read-back, measured on GB300 at about the time
// of 30 K stages.  It is used when the whole-tile waves would idle longer.
constexpr int kStreamKTailStages = 30;
bool use_stream_k(int M, int N, int K, int P) {
    const long long tiles = gemm_tiles(M, N), KS = K / kBK;
    const long long whole = (tiles + P - 1) / P * KS;
    const long long shared = (tiles * KS + P - 1) / P + kStreamKTailStages;
    return shared < whole;
}
size_t gemm_counter_bytes(int M, int N) { return ((size_t)gemm_tiles(M, N) * 4 * 4 + 255) / 256 * 256; }
}  // namespace
}  // namespace tern

extern "C" size_t tern_gemm_workspace_bytes(int M, int N, int K) {
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return 0;
    return gemm_counter_bytes(M, N) + (size_t)gemm_tiles(M, N) * kTileFloats * 4;
}

namespace {
tern_status run_gemm(const void* x, const uint32_t* codes, const void* scales, void* y, int y_is_bf16, int M, int N,
                     int K, void* workspace, size_t workspace_bytes, tern_stream_t stream, bool bin,
                     const void* biases = nullptr) {
    set_launch_count(0);
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return TERN_ERR_SHAPE;
    if ((long long)M * N >= (1LL << 40) || (long long)N * K >= (1LL << 40)) return TERN_ERR_SHAPE;
    if (!x || !codes || !scales || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y)) return TERN_ERR_ALIGN;
    if (!workspace || workspace_bytes < tern_gemm_workspace_bytes(M, N, K)) return TERN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;

    CUtensorMap mx, mc;
    if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, kBK, kBN,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, codes, (uint64_t)(K / (bin ? 32 : 16)), (uint64_t)N,
                     (uint64_t)(K / (bin ? 32 : 16)) * 4, kBK / 16, kBM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return TERN_ERR_CUDA;

    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TERN_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes) != cudaSuccess)
            return TERN_ERR_CUDA;
        attr_set[dev] = true;
    }
    GemmArgs args;
    args.scales = reinterpret_cast<const __half*>(scales);
    args.biases = reinterpret_cast<const __half*>(biases);
    args.y = y;
    args.y_is_bf16 = y_is_bf16 ? 1 : 0;
    args.bin = bin ? 1 : 0;
    args.M = M;
    args.N = N;
    args.K = K;
    args.counters = reinterpret_cast<unsigned*>(workspace);
    args.sums = reinterpret_cast<float*>(static_cast<char*>(workspace) + gemm_counter_bytes(M, N));
    const int shares = gemm_shares(M, N, K, sms);
    args.stream_k = use_stream_k(M, N, K, shares) ? 1 : 0;
    const int tiles = gemm_tiles(M, N);
    const int grid = args.stream_k ? shares : (tiles < shares ? tiles : shares);
    cudaError_t e = launch_pdl(biases ? gemm_kernel<true> : gemm_kernel<false>, dim3(grid), dim3(kThreads),
                               kSmemBytes, (cudaStream_t)stream, true, mx, mc, args);
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}
}  // namespace

extern "C" tern_status tern_gemm(const void* x, const uint32_t* codes, const void* scales, void* y,
                                 int y_is_bf16, int M, int N, int K, void* workspace,
                                 size_t workspace_bytes, tern_stream_t stream) {
    return run_gemm(x, codes, scales, y, y_is_bf16, M, N, K, workspace, workspace_bytes, stream, false);
}

extern "C" tern_status tern_affine_gemm(const void* x, const uint32_t* codes, const void* scales,
                                        const void* biases, void* y, int y_is_bf16, int M, int N, int K,
                                        void* workspace, size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return TERN_ERR_SHAPE;
    if (!biases) return TERN_ERR_NULL;
    if (!aligned16(biases)) return TERN_ERR_ALIGN;
    return run_gemm(x, codes, scales, y, y_is_bf16, M, N, K, workspace, workspace_bytes, stream, false, biases);
}

extern "C" tern_status tern_bin_gemm(const void* x, const uint32_t* words, const void* scales, void* y,
                                     int y_is_bf16, int M, int N, int K, void* workspace,
                                     size_t workspace_bytes, tern_stream_t stream) {
    return run_gemm(x, words, scales, y, y_is_bf16, M, N, K, workspace, workspace_bytes, stream, true);
}
