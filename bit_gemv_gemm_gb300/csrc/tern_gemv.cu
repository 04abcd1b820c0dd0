// tern_gemv.cu -- decode / small-batch ternary-g128 product, M = 1..16.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} x[m][k] * (q[n][k] - 1)
//
// ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card: ternary g128 weights,
// "Weight representation"; codes unpacked and scaled inside the product,
// "CUDA (NVIDIA GPUs)"; decode is the memory-bandwidth-bound phase,
// "Cross-platform throughput".)
//
// Arithmetic.  At 2.125 bits per weight an M = 1 product must retire ~25 G
// weights per ms to keep HBM busy, more than the CUDA cores can afford at the
// two or three ALU operations a scalar unpack-and-add costs.  So the adds run
// on the tensor pipe (mma.sync m16n8k16, f16 in, f32 accumulate) and the unpack
// is ONE logical AND per two weights:
//
//   * a word holds codes j and j + 8 of a 16-weight slice in bits 2j and
//     2j + 16.  `word & (0x00030003 << 2j)` leaves, in each 16-bit half, the
//     bit pattern q << 2j.  Read as fp16 that is exactly q * 2^(2j - 24) for
//     j <= 4 (a subnormal) and q * 2^-14 for j = 5 (the two low exponent
//     bits), i.e. q * 2^(2j - 24) for every j <= 5.  Codes 6, 7, 14, 15 take
//     one shift by 12 and reuse the j = 0 and j = 1 masks.  The result is the
//     MMA A-fragment register directly; q = 0, 1, 2 is exact.
//   * the activation is staged as fp16 B fragments, each value pre-multiplied
//     by the power of two 2^(E + 10 - 2j') that undoes its slot's
//     2^(2j' - 24) (j' = j or j - 6), with a per-(token, group) exponent E
//     chosen from the group's max |x| so the largest staged value is below
//     2^15.  bf16 values stage exactly (8 significant bits into 11).  One MMA
//     per slot position j accumulates acc = 2^(E - 14) sum_k q_k x_k over 16
//     weights of 16 rows.
//   * the -1 of q - 1: the same eight-MMA chain run once per (token, group)
//     on the all-ones code pattern gives acc1 = 2^(E - 14) sum_k x_k with the
//     very same rounding, and per row and group
//         y += s_g * (2^(14 - E) * acc - 2^(14 - E) * acc1),
//     so a row of zero weights (q = 1 everywhere) gives exactly 0.
//
// Work split.  K is cut into slices of up to 8 groups; a CTA owns one slice
// and a contiguous range of 16-row tiles.  Warp w of the CTA owns group w of
// the slice: it stages that group's activation once, into registers, and then
// keeps it for the whole range.  A ninth warp streams the slice's codes of one
// tile (16 rows x 8 groups = 4 KB) per TMA load into a shared-memory ring (the
// first loads go out before the programmatic-dependent-launch wait); each
// compute warp reads its 32-byte column of every tile and runs two tiles per
// step as two independent MMA chains.  Row partial sums go to shared-memory
// accumulators.  With one slice the CTA writes y; with several, each CTA
// stores its partial tile sums to the workspace and the last CTA to finish a
// tile (an arrival counter) adds the slices in slice order and writes y.  y is
// written exactly once per element: no pre-zeroing, no global float atomics.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "tern_fwht.cuh"
#include "tern_sm100.cuh"

namespace tern {
namespace {

__device__ int g_gemv_error;

constexpr int kGroup = 128;            // weights per scale
constexpr int kSliceGroups = 8;        // groups per K-slice = compute warps per CTA
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;   // + the TMA producer warp
constexpr int kTileBytes = 16 * 128 * 2;   // 16 rows x 8 groups x 32 B, as two 128-B-wide halves
constexpr int kTileScaleBytes = 16 * 8 * 2;   // 16 rows x 8 groups of fp16 scales
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr size_t kSmemPerSm = 227 * 1024;    // shared memory a GB300 SM offers its CTAs

template <int MT> struct GemvCfg;
template <> struct GemvCfg<1> { static constexpr int kCtasPerSm = 2; };
template <> struct GemvCfg<2> { static constexpr int kCtasPerSm = 2; };

struct GemvArgs {
    const void* x;              // bf16 [M][K], or fp32 [M][K] when the rotation prologue ran
    const __half* scales;       // [N][K/128]
    float* y;                   // [M][N]
    float* partial;             // [S][T][M][16]
    unsigned* counter;          // [T]
    int M, N, K, G, T, S, cps, rmax;
    int ring;                   // ring slots (one per tile of the range whenever shared memory allows)
    int scale_tma;              // scales stream through the ring (needs K % 1024 == 0)
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// dynamic shared memory: [code ring | scale ring | barriers | row accumulators | finalize flags]
__host__ __device__ inline size_t smem_scl(int ring) { return (size_t)ring * kTileBytes; }
__host__ __device__ inline size_t smem_bar(int ring) { return smem_scl(ring) + (size_t)ring * kTileScaleBytes; }
__host__ __device__ inline size_t smem_acc(int ring) { return align_up(smem_bar(ring) + (size_t)ring * 16 + 16, 16); }
__host__ __device__ inline size_t smem_fin(int ring, int rmax, int MP) {
    return smem_acc(ring) + (size_t)rmax * 16 * MP * 4;
}
__host__ __device__ inline size_t smem_total(int ring, int rmax, int MP) {
    return smem_fin(ring, rmax, MP) + (size_t)rmax * 4 + 1024;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, bool accumulate) {
    if (accumulate) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        const float z = 0.0f;
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    }
}

// Slot j's A registers from the four code words by one AND (codes 6, 7, 14, 15
// after a shift by 12).
__device__ __forceinline__ void slot_regs(int j, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                          uint32_t (&r)[4]) {
    if (j < 6) {
        const uint32_t mk = 0x00030003u << (2 * j);
        r[0] = w0 & mk;
        r[1] = w1 & mk;
        r[2] = w2 & mk;
        r[3] = w3 & mk;
    } else {
        const uint32_t mk = 0x00030003u << (2 * (j - 6));
        r[0] = (w0 >> 12) & mk;
        r[1] = (w1 >> 12) & mk;
        r[2] = (w2 >> 12) & mk;
        r[3] = (w3 >> 12) & mk;
    }
}

// The chain of one token tile alone (the same j order, hence the same rounding,
// as unit_mmas and unit_mmas2 give each token tile).
__device__ __forceinline__ void mma_chain1(float (&acc)[4], const uint32_t (&w)[4], const uint32_t (&b)[16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[4];
        slot_regs(j, w[0], w[1], w[2], w[3], r);
        mma16816(acc, r[0], r[1], r[2], r[3], b[2 * j], b[2 * j + 1], j > 0);
    }
}

// Reads this lane's four code words of group gl of one tile from the ring (two
// rows x two words; the tile is two 128-byte-swizzled halves of four groups:
// 16-byte chunk c of row r sits at chunk c ^ (r % 8)).
__device__ __forceinline__ void read_codes(const unsigned char* tile, int gl, int gid, int t, uint32_t (&w)[4]) {
    const unsigned char* half = tile + (gl >> 2) * (kTileBytes / 2);
    const int c = 2 * (gl & 3) + (t >> 1);
    const int off = ((c ^ (gid & 7)) << 4) + 8 * (t & 1);
    const uint2 v0 = *reinterpret_cast<const uint2*>(half + gid * 128 + off);
    const uint2 v1 = *reinterpret_cast<const uint2*>(half + (gid + 8) * 128 + off);
    w[0] = v0.x;   // row gid,     word 2t      (MMA rows 0-7,  k-slots 2t, 2t+1)
    w[1] = v1.x;   // row gid + 8, word 2t      (MMA rows 8-15)
    w[2] = v0.y;   // row gid,     word 2t + 1  (k-slots 2t+8, 2t+9)
    w[3] = v1.y;   // row gid + 8, word 2t + 1
}

// Two tiles of the warp's group at once: 2 x MT independent MMA chains sharing
// the B fragments, each in the slot order of mma_chain1 (so each keeps the
// ones-pass rounding).
template <int MT>
__device__ __forceinline__ void pair_mmas(float (&acc)[2][MT][4], const uint32_t (&w)[2][4],
                                          const uint32_t (&b)[MT][16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[2][4];
#pragma unroll
        for (int q = 0; q < 2; ++q) slot_regs(j, w[q][0], w[q][1], w[q][2], w[q][3], r[q]);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int nt = 0; nt < MT; ++nt)
                mma16816(acc[q][nt], r[q][0], r[q][1], r[q][2], r[q][3], b[nt][2 * j], b[nt][2 * j + 1], j > 0);
    }
}

template <int MT, bool XF32>
__global__ void __launch_bounds__(kThreads, GemvCfg<MT>::kCtasPerSm)
gemv_kernel(const __grid_constant__ CUtensorMap tmap_codes, const __grid_constant__ CUtensorMap tmap_scales,
            const GemvArgs a) {
    using namespace sm100;
    constexpr int MP = 8 * MT;
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int rmax = a.rmax, ring = a.ring;
    const uint32_t bar0 = sbase + (uint32_t)smem_bar(ring);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (ring + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + smem_bar(ring) + 16 * ring);
    float* accs = reinterpret_cast<float*>(smem + smem_acc(ring));                      // [rmax][16][MP]
    int* fin = reinterpret_cast<int*>(smem + smem_fin(ring, rmax, MP));                 // [rmax]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int M = a.M, N = a.N, G = a.G, T = a.T, S = a.S;
    const int sigma = blockIdx.x / a.cps, cslot = blockIdx.x - sigma * a.cps;
    const int g0 = sigma * kSliceGroups;
    const int gs = min(kSliceGroups, G - g0);
    const int tile_lo = (int)((long long)T * cslot / a.cps);
    const int tile_hi = (int)((long long)T * (cslot + 1) / a.cps);
    const int R = tile_hi - tile_lo;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ring; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kComputeWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmap_codes);
        if (a.scale_tma) tma_prefetch_desc(&tmap_scales);
    }
    __syncthreads();
    pdl_launch_dependents();

    auto fail = [&](int code) {
        if (!*abort_flag) {
            *abort_flag = 1;
            report_device_error(&g_gemv_error, code);
        }
    };

    if (warp == kComputeWarps) {
        // ------------------------------ TMA producer ------------------------------
        // codes and scales are never the previous kernel's output: stream them
        // before the PDL wait; with one slot per tile every load goes out at once
        if (lane == 0) {
            const uint32_t bytes = (gs > 4 ? (uint32_t)kTileBytes : (uint32_t)kTileBytes / 2) +
                                   (a.scale_tma ? (uint32_t)kTileScaleBytes : 0u);
            int issued = 0;
            for (int i = 0; i < R; ++i, ++issued) {
                const int s = i % ring;
                const uint32_t ph = (uint32_t)(i / ring) & 1u;
                if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kWaitLimitNs)) {
                    fail(kDevErrGemvProducerWait);
                    break;
                }
                const uint32_t dst = sbase + (uint32_t)(s * kTileBytes);
                const int row = (tile_lo + i) * 16;
                mbar_arrive_expect_tx(full_bar(s), bytes);
                tma_load_2d(dst, &tmap_codes, g0 * 8, row, full_bar(s));
                if (gs > 4) tma_load_2d(dst + kTileBytes / 2, &tmap_codes, g0 * 8 + 32, row, full_bar(s));
                if (a.scale_tma)
                    tma_load_2d(sbase + (uint32_t)(smem_scl(ring) + (size_t)s * kTileScaleBytes), &tmap_scales, g0,
                                row, full_bar(s));
            }
            if (*abort_flag) {
                const int n = issued < ring ? issued : ring;
                for (int k = issued - n; k < issued; ++k)
                    (void)mbar_wait_drain(full_bar(k % ring), (uint32_t)(k / ring) & 1u, 100000000ull);
            }
        }
        pdl_wait();
    } else {
        // ------------------------------ compute warps ------------------------------
        pdl_wait();
        // warp w owns group g0 + w of the slice for every tile of the range: it
        // stages that group's activation B fragments and (F, F * acc1) into
        // registers once
        const bool active = warp < gs;
        const int g = g0 + warp;
        uint32_t b[MT][16];
        float4 f[MT];   // (F, F*acc1) of tokens 2t and 2t+1 of each token tile
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
            const int m = nt * 8 + gid;
            float v[32];
            if (active && m < M) {
                const size_t off = (size_t)m * a.K + (size_t)g * kGroup + 32 * t;
                if (XF32) {
                    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.x) + off);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 u = src[q];
                        v[4 * q] = u.x;
                        v[4 * q + 1] = u.y;
                        v[4 * q + 2] = u.z;
                        v[4 * q + 3] = u.w;
                    }
                } else {
                    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + off);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u = src[q];
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[8 * q + 2 * e] = __uint_as_float(uw[e] << 16);
                            v[8 * q + 2 * e + 1] = __uint_as_float(uw[e] & 0xFFFF0000u);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.0f;
            }
            float mx = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(v[e]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            int E = 0;
            if (mx > 0.0f && mx <= 3.0e38f) {
                int ex;
                frexpf(mx, &ex);                       // mx < 2^ex
                E = max(-100, min(5 - ex, 150));       // mx * 2^(E + 10) < 2^15
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float c = ldexpf(1.0f, E + 10 - 2 * (j < 6 ? j : j - 6));   // exact power of two
                const __half2 lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);       // k = 32t+j, +8
                const __half2 hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c); // k = 32t+16+j, +24
                b[nt][2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
                b[nt][2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            // the -1 correction: the same chain on the all-ones pattern; every
            // row of the result is the same, lane (gid, t) holds tokens 2t, 2t+1
            float acc1[4];
            const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
            mma_chain1(acc1, ones, b[nt]);
            const float F = (m < M) ? ldexpf(1.0f, 14 - E) : 0.0f;
            const float F0 = __shfl_sync(0xffffffffu, F, (2 * t) * 4);
            const float F1 = __shfl_sync(0xffffffffu, F, (2 * t + 1) * 4);
            f[nt] = make_float4(F0, F0 * acc1[0], F1, F1 * acc1[1]);
        }
        for (int i = threadIdx.x; i < R * 16 * MP; i += kComputeWarps * 32) accs[i] = 0.0f;
        // zeroed accumulators visible to every compute warp
        asm volatile("bar.sync 1, %0;" ::"r"(kComputeWarps * 32) : "memory");

        // every warp walks every tile in order (the ring is consumed in order)
        auto epilogue = [&](int i, const float (&acc)[MT][4], float s0, float s1) {
            float* row = accs + (size_t)i * 16 * MP;
#pragma unroll
            for (int nt = 0; nt < MT; ++nt) {
                const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
                if (nt * 8 < M) {
                    if (m0 < M) {
                        atomicAdd(row + gid * MP + m0, s0 * fmaf(f[nt].x, acc[nt][0], -f[nt].y));
                        atomicAdd(row + (gid + 8) * MP + m0, s1 * fmaf(f[nt].x, acc[nt][2], -f[nt].y));
                    }
                    if (M > 1 && m1 < M) {
                        atomicAdd(row + gid * MP + m1, s0 * fmaf(f[nt].z, acc[nt][1], -f[nt].w));
                        atomicAdd(row + (gid + 8) * MP + m1, s1 * fmaf(f[nt].z, acc[nt][3], -f[nt].w));
                    }
                }
            }
        };
        auto tile_scales = [&](int i, int s, float& s0, float& s1) {
            if (a.scale_tma) {
                const unsigned char* tscale = smem + smem_scl(ring) + (size_t)s * kTileScaleBytes;
                s0 = __half2float(*reinterpret_cast<const __half*>(tscale + gid * 16 + 2 * warp));
                s1 = __half2float(*reinterpret_cast<const __half*>(tscale + (gid + 8) * 16 + 2 * warp));
            } else {
                const int row0 = (tile_lo + i) * 16 + gid;
                s0 = row0 < N ? __half2float(a.scales[(size_t)row0 * G + g]) : 0.0f;
                s1 = row0 + 8 < N ? __half2float(a.scales[(size_t)(row0 + 8) * G + g]) : 0.0f;
            }
        };
        for (int i = 0; i < R; i += 2) {
            const bool two = i + 1 < R;
            const int sA = i % ring, sB = (i + 1) % ring;
            if (!mbar_wait_bounded(full_bar(sA), (uint32_t)(i / ring) & 1u, abort_flag, kWaitLimitNs) ||
                (two && !mbar_wait_bounded(full_bar(sB), (uint32_t)((i + 1) / ring) & 1u, abort_flag, kWaitLimitNs))) {
                fail(kDevErrGemvConsumerWait);
                break;
            }
            if (active) {
                uint32_t w2[2][4];
                float sc[2][2];
                read_codes(smem + sA * kTileBytes, warp, gid, t, w2[0]);
                tile_scales(i, sA, sc[0][0], sc[0][1]);
                if (two) {
                    read_codes(smem + sB * kTileBytes, warp, gid, t, w2[1]);
                    tile_scales(i + 1, sB, sc[1][0], sc[1][1]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) w2[1][e] = 0x55555555u;
                    sc[1][0] = sc[1][1] = 0.0f;
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar(sA));
                    if (two) mbar_arrive(empty_bar(sB));
                }
                float acc[2][MT][4];
                pair_mmas<MT>(acc, w2, b);
                epilogue(i, acc[0], sc[0][0], sc[0][1]);
                if (two) epilogue(i + 1, acc[1], sc[1][0], sc[1][1]);
            } else {
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar(sA));
                    if (two) mbar_arrive(empty_bar(sB));
                }
            }
        }
    }
    __syncthreads();
    if (*abort_flag) return;

    // ---- write y (one slice) or the partials and the cross-slice fix-up ----
    const int nvals = R * 16 * M;
    if (S == 1) {
        for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
            const int m = i / (R * 16), rr = i - m * (R * 16);
            const int r = tile_lo * 16 + rr;
            if (r < N) a.y[(size_t)m * N + r] = accs[(size_t)rr * MP + m];
        }
        return;
    }
    float* P = a.partial + ((size_t)sigma * T + tile_lo) * 16 * M;
    for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
        const int tl = i / (16 * M), rem = i - tl * 16 * M;
        const int m = rem / 16, r = rem - m * 16;
        P[i] = accs[((size_t)tl * 16 + r) * MP + m];   // [tile][m][16]
    }
    __threadfence();
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += blockDim.x)
        fin[i] = (atomicAdd(a.counter + tile_lo + i, 1u) == (unsigned)(S - 1));
    __syncthreads();
    __threadfence();
    for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
        const int tl = i / (16 * M);
        if (!fin[tl]) continue;
        const int rem = i - tl * 16 * M;
        const int m = rem / 16, r = rem - m * 16;
        const int tile_g = tile_lo + tl;
        const size_t off = (size_t)tile_g * 16 * M + rem;
        float sum = 0.0f;
        for (int sg = 0; sg < S; ++sg) sum += __ldcg(a.partial + (size_t)sg * T * 16 * M + off);
        const int row = tile_g * 16 + r;
        if (row < N) a.y[(size_t)m * N + row] = sum;
    }
    for (int i = threadIdx.x; i < R; i += blockDim.x)
        if (fin[i]) a.counter[tile_lo + i] = 0u;
}

// Rotation prologue for the fused path: xr (fp32 [M][K]) = H_4096 (s (.) x) / 64,
// kept in fp32 (never rounded to bf16) for the product's staging.
__global__ void __launch_bounds__(kFwhtThreads)
rotate_f32_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs, float* __restrict__ xr,
                  int K) {
    __shared__ float sm[kFwhtSmemFloats];
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x, m = blockIdx.y;
    const size_t off = (size_t)m * K + (size_t)b * kFwhtN;
    fwht4096_block(x + off, signs + (size_t)b * kFwhtN, sm);
    float4* out = reinterpret_cast<float4*>(xr + off);
    for (int i = threadIdx.x; i < kFwhtN / 4; i += blockDim.x) {
        const int e = 4 * i;
        out[i] = make_float4(sm[fwht_pos(e)], sm[fwht_pos(e + 1)], sm[fwht_pos(e + 2)], sm[fwht_pos(e + 3)]);
    }
}

// ---------------------------------------------------------------------------
// Host side.
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

struct Plan {
    int G, T, S, cps, ctas, rmax, ring, MT;
    size_t smem;
    size_t off_xr, off_partial, off_counter, bytes;
};

Plan make_plan(int M, int N, int K, bool rot, int sms) {
    Plan p{};
    p.G = K / kGroup;
    p.T = (N + 15) / 16;
    p.S = (p.G + kSliceGroups - 1) / kSliceGroups;
    p.MT = (M + 7) / 8;
    const int MP = 8 * p.MT;
    const int per_sm = p.MT == 1 ? GemvCfg<1>::kCtasPerSm : GemvCfg<2>::kCtasPerSm;
    const int cmax = sms * per_sm;
    // ring slots that fit next to the fixed shared memory: one per tile of the
    // CTA's range whenever possible, so every code load can be in flight at once
    const size_t budget = kSmemPerSm / per_sm;
    const size_t fixed = smem_total(0, 0, MP);
    const size_t slot = (size_t)kTileBytes + kTileScaleBytes + 16;
    const size_t acc_per_tile = (size_t)16 * MP * 4 + 4;
    p.cps = p.S >= cmax ? 1 : cmax / p.S;
    if (p.cps > p.T) p.cps = p.T;
    for (;;) {
        p.rmax = (p.T + p.cps - 1) / p.cps;
        const size_t left = budget - fixed;
        const long long fit = left > p.rmax * acc_per_tile
                                  ? (long long)((left - p.rmax * acc_per_tile) / slot) : 0;
        p.ring = (int)(fit < p.rmax ? fit : p.rmax);
        if (p.ring >= p.rmax || (p.ring >= 8 && p.ring * 4 >= p.rmax * 3) || p.cps >= p.T) break;
        p.cps = p.cps * 5 / 4 + 1;   // more, shorter ranges
        if (p.cps > p.T) p.cps = p.T;
    }
    if (p.ring < 1) p.ring = 1;
    p.ctas = p.S * p.cps;
    p.smem = smem_total(p.ring, p.rmax, MP);
    size_t off = 0;
    p.off_xr = off;
    if (rot) off = align_up(off + (size_t)M * K * 4, 256);
    p.off_partial = off;
    if (p.S > 1) off = align_up(off + (size_t)p.S * p.T * 16 * M * 4, 256);
    p.off_counter = off;
    if (p.S > 1) off = align_up(off + (size_t)p.T * 4, 256);
    p.bytes = off > 0 ? off : 256;
    return p;
}

tern_status validate(const void* x, const uint32_t* codes, const void* scales, const float* y, int M, int N, int K) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return TERN_ERR_SHAPE;
    if ((long long)N * (K / 16) >= (1LL << 40) || (long long)M * K >= (1LL << 31) || N >= (1 << 28))
        return TERN_ERR_SHAPE;
    if (!x || !codes || !scales || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

size_t workspace_bytes(int M, int N, int K, bool rot) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return 0;
    // partials and counters depend on (S, T) only, never on the device
    return make_plan(M, N, K, rot, 1 << 20).bytes;
}

template <int MT, bool XF32>
cudaError_t launch_gemv(const CUtensorMap& tmap, const CUtensorMap& tmap_s, const GemvArgs& args, const Plan& p,
                        cudaStream_t stream) {
    static int attr_bytes[64] = {};   // the attribute is per function and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_bytes[dev] < (int)p.smem) {
        e = cudaFuncSetAttribute(gemv_kernel<MT, XF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return e;
        attr_bytes[dev] = (int)p.smem;
    }
    return launch_pdl(gemv_kernel<MT, XF32>, dim3(p.ctas), dim3(kThreads), p.smem, stream, true, tmap, tmap_s,
                      args);
}

tern_status run(const void* x, const int8_t* signs, const uint32_t* codes, const void* scales, float* y, int M,
                int N, int K, void* workspace, size_t workspace_bytes_, cudaStream_t stream) {
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const Plan p = make_plan(M, N, K, signs != nullptr, sms);
    if (p.bytes > 256 || signs) {
        if (!workspace || workspace_bytes_ < p.bytes) return TERN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
    }
    auto enc = get_encode();
    if (!enc) return TERN_ERR_CUDA;
    CUtensorMap tmap, tmap_s;
    memset(&tmap_s, 0, sizeof(tmap_s));
    {
        cuuint64_t gdim[2] = {(cuuint64_t)(K / 16), (cuuint64_t)N};
        cuuint64_t gstride[1] = {(cuuint64_t)(K / 16) * 4};
        cuuint32_t box[2] = {32, 16};
        cuuint32_t es[2] = {1, 1};
        if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TERN_ERR_CUDA;
    }
    // scales ride along with the codes when a scale row is a multiple of 16 bytes
    const bool scale_tma = (p.G % 8) == 0;
    if (scale_tma) {
        cuuint64_t gdim[2] = {(cuuint64_t)p.G, (cuuint64_t)N};
        cuuint64_t gstride[1] = {(cuuint64_t)p.G * 2};
        cuuint32_t box[2] = {8, 16};
        cuuint32_t es[2] = {1, 1};
        if (enc(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(scales), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TERN_ERR_CUDA;
    }
    char* ws = reinterpret_cast<char*>(workspace);
    GemvArgs args;
    args.x = x;
    args.scales = reinterpret_cast<const __half*>(scales);
    args.y = y;
    args.partial = p.S > 1 ? reinterpret_cast<float*>(ws + p.off_partial) : nullptr;
    args.counter = p.S > 1 ? reinterpret_cast<unsigned*>(ws + p.off_counter) : nullptr;
    args.M = M;
    args.N = N;
    args.K = K;
    args.G = p.G;
    args.T = p.T;
    args.S = p.S;
    args.cps = p.cps;
    args.rmax = p.rmax;
    args.ring = p.ring;
    args.scale_tma = scale_tma ? 1 : 0;
    int launches = 1;
    cudaError_t e;
    if (signs) {
        float* xr = reinterpret_cast<float*>(ws + p.off_xr);
        e = launch_pdl(rotate_f32_kernel, dim3(K / kFwhtN, M), dim3(kFwhtThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), signs, xr, K);
        if (e != cudaSuccess) return TERN_ERR_CUDA;
        args.x = xr;
        launches = 2;
        e = p.MT == 1 ? launch_gemv<1, true>(tmap, tmap_s, args, p, stream)
                      : launch_gemv<2, true>(tmap, tmap_s, args, p, stream);
    } else {
        e = p.MT == 1 ? launch_gemv<1, false>(tmap, tmap_s, args, p, stream)
                      : launch_gemv<2, false>(tmap, tmap_s, args, p, stream);
    }
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(launches);
    return TERN_OK;
}

}  // namespace

cudaError_t read_gemv_device_error(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemv_error, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(int));
}

}  // namespace tern

using namespace tern;

extern "C" size_t tern_gemv_workspace_bytes(int M, int N, int K) {
    // covers both the plain and the rotation-fused call of the same shape
    return workspace_bytes(M, N, K, (K % kFwhtN) == 0);
}

extern "C" tern_status tern_gemv(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                 int N, int K, void* workspace, size_t workspace_bytes_, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    const size_t need = workspace_bytes(M, N, K, false);
    if (need > 256 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
    return run(x, nullptr, codes, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream);
}

extern "C" tern_status tern_fwht_gemm(const void* x, const int8_t* signs, const uint32_t* codes,
                                      const void* scales, float* y, int M, int N, int K, void* workspace,
                                      size_t workspace_bytes_, tern_stream_t stream) {
    set_launch_count(0);
    if (K % kFwhtN != 0) return TERN_ERR_SHAPE;
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (!signs) return TERN_ERR_NULL;
    if (!aligned16(signs)) return TERN_ERR_ALIGN;
    if (!workspace || workspace_bytes_ < workspace_bytes(M, N, K, true)) return TERN_ERR_WORKSPACE;
    return run(x, signs, codes, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream);
}
