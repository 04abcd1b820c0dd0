// tern_f3.cu -- native base-3 packing: five trits per byte, and the decode
// product on it.
//
// The card gives the information content of a trit (log2 3 bits) and the 1.71
// bits/weight it implies with the FP16 scale, and names packing at that
// density as future work ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card,
// "Weight representation: ternary g128" and "Memory requirement").  Layout
// (the pages give none): byte j < 25 of a 128-weight group holds trits
// 5 j .. 5 j + 4 as q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4 (q = t + 1, values 0..242),
// byte 25 holds trits 125..127 as q0 + 3 q1 + 9 q2; rows are [N][26 K/128]
// bytes, 1.75 bits per weight with the scale.
//
// The product runs on the CUDA cores (a byte's five trits are not separable by
// masks).  For one or two tokens it reads per-lane dot-product tables (below);
// for more, each byte is looked up in a 243-entry table of its five weights
// (-1, 0, +1 as fp32) and its activations are summed with fp32 FMAs.  A warp
// owns two rows; lane j < 26 takes byte j of every group, so the lane's K
// offsets within a group are fixed and a group's 26 bytes are read by one
// coalesced load.  The activation is staged in shared memory (fp32) one
// 1024-wide chunk at a time for all tokens, and each lane loads the next
// chunk's bytes and scales while it sums the current one; each row's sums stay
// in registers over the whole of K, so every output is written once (no
// workspace).
#include <algorithm>
#include <mutex>

#include "tern_common.cuh"
#include "tern_mma.cuh"

namespace tern {
namespace {

constexpr int kF3Threads = 256;
constexpr int kF3Warps = kF3Threads / 32;
constexpr int kF3RowsPerWarp = 2;
constexpr int kF3Chunk = 1024;          // activation values staged per token and pass
constexpr int kF3Lut = 243 * 8;         // table floats: five weights per byte, padded to 8
constexpr int kF3MaxM = 16;

// One thread per output byte: its 5 (or 3) trits, an invalid entry written as
// q = 0 and counted.
__global__ void __launch_bounds__(256)
f3_pack_kernel(const int8_t* __restrict__ t, uint8_t* __restrict__ out, int N, int K, int* __restrict__ bad_count) {
    const int G = K / 128;
    const long long total = (long long)N * G * 26;
    int bad = 0;
    for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < total;
         b += (long long)gridDim.x * blockDim.x) {
        const long long rg = b / 26;              // row * G + group
        const int j = (int)(b - rg * 26);
        const int n = (int)(rg / G), g = (int)(rg - (long long)n * G);
        const int8_t* src = t + (size_t)n * K + (size_t)g * 128 + 5 * j;
        const int cnt = j < 25 ? 5 : 3;
        int v = 0, p = 1;
        for (int i = 0; i < cnt; ++i) {
            int q = (int)src[i] + 1;
            if (q < 0 || q > 2) {
                ++bad;
                q = 0;
            }
            v += q * p;
            p *= 3;
        }
        out[b] = (uint8_t)v;
    }
    if (bad_count) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(bad_count, bad);
    }
}

__global__ void __launch_bounds__(kF3Threads, 2)
f3_gemv_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ packed,
               const __half* __restrict__ scales, float* __restrict__ y, int M, int N, int K) {
    extern __shared__ __align__(16) float f3_smem[];
    float* lut = f3_smem;                 // [243][8]: weights q_i - 1 of byte v at lut[8 v + i]
    float* xs = f3_smem + kF3Lut;         // [M][kF3Chunk]
    for (int v = threadIdx.x; v < 243; v += kF3Threads) {
        int r = v;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            lut[8 * v + i] = (float)(r % 3 - 1);
            r /= 3;
        }
        lut[8 * v + 5] = lut[8 * v + 6] = lut[8 * v + 7] = 0.0f;
    }
    pdl_launch_dependents();
    pdl_wait();   // x may be the previous kernel's output, y still read by it
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / 128;
    const size_t pitch = (size_t)26 * G;
    const int row0 = (blockIdx.x * kF3Warps + warp) * kF3RowsPerWarp;
    float acc[kF3RowsPerWarp][kF3MaxM];
#pragma unroll
    for (int r = 0; r < kF3RowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < kF3MaxM; ++m) acc[r][m] = 0.0f;
    const bool five = lane < 25, byte_lane = lane < 26;
    // A chunk's bytes of this lane (byte `lane` of each of up to 8 groups, four
    // to a register) and its scales (lane g < 8: group g), per row: the next
    // chunk's are loaded while the current one is summed.
    uint32_t cb[kF3RowsPerWarp][2], nb[kF3RowsPerWarp][2];
    float cs[kF3RowsPerWarp], ns[kF3RowsPerWarp];
    auto load_chunk = [&](int k0, uint32_t (&bytes)[kF3RowsPerWarp][2], float (&sc)[kF3RowsPerWarp]) {
        const int gb = k0 / 128, gc = min(kF3Chunk, K - k0) / 128;
#pragma unroll
        for (int r = 0; r < kF3RowsPerWarp; ++r) {
            const int n = row0 + r;
            const uint8_t* prow = packed + (size_t)n * pitch + (size_t)gb * 26;
            uint32_t w[2] = {0u, 0u};
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                // 121 = five zero trits for the slots past the chunk
                const uint32_t v = (n < N && byte_lane && g < gc) ? (uint32_t)prow[g * 26 + lane] : 121u;
                w[g >> 2] |= v << (8 * (g & 3));
            }
            bytes[r][0] = w[0];
            bytes[r][1] = w[1];
            sc[r] = (n < N && lane < gc) ? __half2float(scales[(size_t)n * G + gb + lane]) : 0.0f;
        }
    };
    load_chunk(0, cb, cs);
    for (int k0 = 0; k0 < K; k0 += kF3Chunk) {
        const int kc = min(kF3Chunk, K - k0), gc = kc / 128;
        __syncthreads();   // the previous chunk is no longer read
        for (int i = threadIdx.x; i < M * kc; i += kF3Threads) {
            const int m = i / kc, k = i - m * kc;
            xs[m * kF3Chunk + k] = __bfloat162float(x[(size_t)m * K + k0 + k]);
        }
        if (k0 + kF3Chunk < K) load_chunk(k0 + kF3Chunk, nb, ns);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kF3RowsPerWarp; ++r) {
            if (row0 + r >= N) continue;   // warp-uniform
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= gc) break;
                const float sg = __shfl_sync(0xffffffffu, cs[r], g);
                if (byte_lane) {
                    const int v = (int)((cb[r][g >> 2] >> (8 * (g & 3))) & 0xFFu);
                    const float4 c = *reinterpret_cast<const float4*>(lut + 8 * v);
                    const float c4 = lut[8 * v + 4];
                    const float* xp = xs + 128 * g + 5 * lane;
#pragma unroll
                    for (int m = 0; m < kF3MaxM; ++m) {
                        if (m < M) {
                            const float* xm = xp + m * kF3Chunk;
                            float d = c.x * xm[0];
                            d = fmaf(c.y, xm[1], d);
                            d = fmaf(c.z, xm[2], d);
                            if (five) {
                                d = fmaf(c.w, xm[3], d);
                                d = fmaf(c4, xm[4], d);
                            }
                            acc[r][m] = fmaf(sg, d, acc[r][m]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kF3RowsPerWarp; ++r) {
            cb[r][0] = nb[r][0];
            cb[r][1] = nb[r][1];
            cs[r] = ns[r];
        }
    }
#pragma unroll
    for (int r = 0; r < kF3RowsPerWarp; ++r) {
        const int n = row0 + r;
#pragma unroll
        for (int m = 0; m < kF3MaxM; ++m) {
            if (m < M) {
                float v = acc[r][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0 && n < N) y[(size_t)m * N + n] = v;
            }
        }
    }
}

// ---- one or two tokens: per-lane dot-product tables ----
// A byte v splits into hi = v / 9 (trits 2..4 of the byte, 27 values) and
// lo = v % 9 (trits 0..1, 9 values).  For every group g of a 1024-wide chunk
// and byte position (lane) l, the CTA tabulates for each token
//   T[g][hi][l]      = sum_{i = 2..4} (digit_i(hi) - 1) x[128 g + 5 l + i]
//   T[g][27 + lo][l] = sum_{i = 0..1} (digit_i(lo) - 1) x[128 g + 5 l + i]
// (byte 25 holds trits 125..127 only: its hi is trit 127 alone), so a byte's
// five products are two table reads and an add.  A thread builds the 36
// entries of one (token, group, byte position) from its five activations; the
// tables are laid out
// [g][entry][32 lanes], so a warp's reads fall on 26 distinct banks.  The grid
// is persistent (four CTAs per SM), each CTA taking a contiguous range of rows
// and building each chunk's tables once for all of them; each warp loads the
// next chunk's bytes while it sums the current one.
constexpr int kF3TabMaxM = 2;
constexpr int kF3TabRowsPerWarp = 4;                  // rows a warp keeps sums for
constexpr int kF3TabCtasPerSm = 4;
constexpr int kF3TabPerToken = 8 * 36 * 32;            // floats per token and chunk

__global__ void __launch_bounds__(kF3Threads, kF3TabCtasPerSm)
f3_gemv_table_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ packed,
                     const __half* __restrict__ scales, float* __restrict__ y, int M, int N, int K, int rows_per_cta) {
    extern __shared__ __align__(16) float f3_tab[];   // [M][8 groups][36][32]
    pdl_launch_dependents();
    pdl_wait();   // x may be the previous kernel's output, y still read by it
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / 128;
    const size_t pitch = (size_t)26 * G;
    const int r0 = blockIdx.x * rows_per_cta, r1 = min(N, r0 + rows_per_cta);
    // this warp's rows: r0 + warp, + 8, ... (at most kF3TabRowsPerWarp)
    float acc[kF3TabRowsPerWarp][kF3TabMaxM];
#pragma unroll
    for (int r = 0; r < kF3TabRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < kF3TabMaxM; ++m) acc[r][m] = 0.0f;
    const bool byte_lane = lane < 26;
    // a chunk's bytes (byte `lane` of each group, four to a register) and
    // scales (lane g: group g) of the warp's rows; the next chunk's are
    // loaded while the current one is summed
    uint32_t bytes[kF3TabRowsPerWarp][2], nbytes[kF3TabRowsPerWarp][2];
    float sc[kF3TabRowsPerWarp], nsc[kF3TabRowsPerWarp];
    auto load_chunk = [&](int k0, uint32_t (&bt)[kF3TabRowsPerWarp][2], float (&st)[kF3TabRowsPerWarp]) {
        const int gb = k0 / 128, gc = min(kF3Chunk, K - k0) / 128;
#pragma unroll
        for (int r = 0; r < kF3TabRowsPerWarp; ++r) {
            const int n = r0 + warp + 8 * r;
            const uint8_t* prow = packed + (size_t)n * pitch + (size_t)gb * 26;
            uint32_t w[2] = {0u, 0u};
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t v = (n < r1 && byte_lane && g < gc) ? (uint32_t)prow[g * 26 + lane] : 121u;
                w[g >> 2] |= v << (8 * (g & 3));
            }
            bt[r][0] = w[0];
            bt[r][1] = w[1];
            st[r] = (n < r1 && lane < gc) ? __half2float(scales[(size_t)n * G + gb + lane]) : 0.0f;
        }
    };
    load_chunk(0, bytes, sc);
    for (int k0 = 0; k0 < K; k0 += kF3Chunk) {
        const int gc = min(kF3Chunk, K - k0) / 128;
        __syncthreads();   // the previous chunk's tables are no longer read
        // one (token, group, byte position) per thread: its five activations
        // (trits 3 and 4 absent for byte 25), then all 36 entries as sums
        for (int it = threadIdx.x; it < M * 8 * 26; it += kF3Threads) {
            const int m = it / 208, rem = it - m * 208;
            const int g = rem / 26, l = rem - g * 26;
            float xv[5] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            if (g < gc) {
                const __nv_bfloat16* xp = x + (size_t)m * K + k0 + 128 * g + 5 * l;
#pragma unroll
                for (int i = 0; i < 5; ++i)
                    if (i < 3 || l < 25) xv[i] = __bfloat162float(xp[i]);
            }
            float* tb = f3_tab + (size_t)(m * 8 + g) * 36 * 32 + l;
            // hi = d2 + 3 d3 + 9 d4: (d2 - 1) x2 + ((d3 - 1) x3 + (d4 - 1) x4)
#pragma unroll
            for (int d4 = 0; d4 < 3; ++d4)
#pragma unroll
                for (int d3 = 0; d3 < 3; ++d3) {
                    const float t34 = (float)(d3 - 1) * xv[3] + (float)(d4 - 1) * xv[4];
#pragma unroll
                    for (int d2 = 0; d2 < 3; ++d2) tb[(d2 + 3 * d3 + 9 * d4) * 32] = (float)(d2 - 1) * xv[2] + t34;
                }
            // lo = d0 + 3 d1
#pragma unroll
            for (int d1 = 0; d1 < 3; ++d1)
#pragma unroll
                for (int d0 = 0; d0 < 3; ++d0) tb[(27 + d0 + 3 * d1) * 32] = (float)(d0 - 1) * xv[0] + (float)(d1 - 1) * xv[1];
        }
        if (k0 + kF3Chunk < K) load_chunk(k0 + kF3Chunk, nbytes, nsc);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kF3TabRowsPerWarp; ++r) {
            if (r0 + warp + 8 * r >= r1) break;   // warp-uniform
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g >= gc) break;
                const float sg = __shfl_sync(0xffffffffu, sc[r], g);
                if (byte_lane) {
                    const uint32_t v = (bytes[r][g >> 2] >> (8 * (g & 3))) & 0xFFu;
                    const uint32_t hi = (v * 57u) >> 9, lo = v - 9u * hi;   // v / 9 and v % 9 for v < 256
#pragma unroll
                    for (int m = 0; m < kF3TabMaxM; ++m) {
                        if (m < M) {
                            const float* tb = f3_tab + (size_t)(m * 8 + g) * 36 * 32 + lane;
                            acc[r][m] = fmaf(sg, tb[hi * 32] + tb[(27 + lo) * 32], acc[r][m]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kF3TabRowsPerWarp; ++r) {
            bytes[r][0] = nbytes[r][0];
            bytes[r][1] = nbytes[r][1];
            sc[r] = nsc[r];
        }
    }
#pragma unroll
    for (int r = 0; r < kF3TabRowsPerWarp; ++r) {
        const int n = r0 + warp + 8 * r;
#pragma unroll
        for (int m = 0; m < kF3TabMaxM; ++m) {
            if (m < M) {
                float v = acc[r][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0 && n < r1) y[(size_t)m * N + n] = v;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// One token on the tensor pipe.
//
// A byte's five trits become five 2-bit codes through a 256-entry table
// (q0 | q1 << 2 | ... | q4 << 8; bytes above 242 are not a pack's and give
// undefined weights), the codes of a lane's 32 weights are assembled into the
// two 2-bit code words the decode product reads (16 codes per word, code i at
// bits 2i), and from there the unit is the decode product's: one AND per two
// weights into fp16 A fragments, the `mma.sync` chain against the staged
// activation, the all-ones correction, the group scale.  Lane (gid, t) takes
// weights 32 t .. 32 t + 31 of a group: bytes from b0 = 32 t / 5 on, the first
// 2 (32 t mod 5) bits of b0's codes dropped; seven bytes hold them, eight for
// t = 2 (weights 64 .. 95 start at b0's last trit and end at byte 19's
// first).  The table's 32-bit entries ([v][lane % 16]) hold the codes already
// shifted for the lane's offset in b0, so the assembly takes fixed shifts;
// lanes l and l + 16 share a copy, so a warp's lookups conflict at most two
// ways.
//
// Work split (as the tile-major decode loop): K-slices of whole quads of
// groups, ranges of 16-row tiles, a warp owning whole tiles and walking its
// slice four groups (16 rows x 104 bytes and the 16 x 4 scales, 8-byte
// copies) at a time, the row sums in registers.  The slices meet in y through
// the range flags of the decode product, here in a file-scope array (the call
// takes no workspace): the slice-0 CTA clears its rows and counts itself in;
// the others add once they have seen the count; the S-th count returns the
// word to 0, so the array is all zeros between calls.
// ---------------------------------------------------------------------------
constexpr int kF3mQuad = 4;                                    // groups per stage
constexpr int kF3mDepth = 4;                                   // stages in flight per warp (a power of 2)
constexpr int kF3mRowBytes = 26 * kF3mQuad;                    // a row's bytes per stage
constexpr int kF3mCodeBytes = 16 * kF3mRowBytes;
constexpr int kF3mStageBytes = kF3mCodeBytes + 16 * kF3mQuad * 2;   // and the tile's 16 x 4 scales
constexpr int kF3mRingBytes = 8 * kF3mDepth * kF3mStageBytes;
constexpr int kF3mLutBytes = 256 * 16 * 4;                    // [byte][lane % 16] words
constexpr int kF3mCtasPerSm = 2;
constexpr int kF3mMaxRanges = 4096;                           // range flags in the file-scope array

__device__ unsigned g_f3_flags[kF3mMaxRanges];   // zero between calls (see above)
__device__ int g_f3_error;                       // sticky device error word of this translation unit

struct F3mArgs {
    const __nv_bfloat16* x;
    const uint8_t* packed;
    const __half* scales;
    float* y;
    int M, N, K, G, T, S, cps;
};

__device__ __forceinline__ void f3_check_stage_range(float mx) {
    if (!(mx < 0x1p100f)) report_device_error(&g_f3_error, kDevErrGemvActivationRange);
}

// ONE: a single token (the staged activation read by broadcast, 256 bytes a
// group); otherwise MT token tiles of eight, each group's fragments per lane
// (2 KB a group and token tile) with (F, F acc1) of the lane's two tokens.
template <int MT, bool ONE>
__global__ void __launch_bounds__(kF3Threads, kF3mCtasPerSm) f3_mma_kernel(const F3mArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int G = a.G, S = a.S, N = a.N, M = ONE ? 1 : a.M;
    constexpr int kFrag = ONE ? 256 : MT * 2048;   // staged activation bytes per group
    const size_t pitch = (size_t)26 * G;   // bytes per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int sigma = blockIdx.x / a.cps, clu = blockIdx.x - sigma * a.cps;   // slice, range
    const int Gq = G / kF3mQuad;
    const int qA = (int)((long long)Gq * sigma / S);
    const int nq = (int)((long long)Gq * (sigma + 1) / S) - qA;
    const int gA = kF3mQuad * qA, Gs = kF3mQuad * nq;
    const int tile_lo = (int)((long long)a.T * clu / a.cps);
    const int R = (int)((long long)a.T * (clu + 1) / a.cps) - tile_lo;
    const int n_items = warp < R ? (R - 1 - warp) / 8 + 1 : 0;
    const int n_st = n_items * nq;

    unsigned char* const ring = smem + (size_t)warp * kF3mDepth * kF3mStageBytes;
    const uint32_t* const lut = reinterpret_cast<const uint32_t*>(smem + kF3mRingBytes);
    // ONE: [Gs][4][t][4 words] and [Gs] (F, F acc1); else [Gs][MT][4][32 lanes][16 B] and [Gs][MT][t] float4
    unsigned char* const frag = smem + kF3mRingBytes + kF3mLutBytes;
    unsigned char* const corr = frag + (size_t)Gs * kFrag;
    uint32_t* const bfr = reinterpret_cast<uint32_t*>(frag);
    float2* const fcs = reinterpret_cast<float2*>(corr);

    // ---- this warp's copies: lanes 0-25 take 8-byte piece l % 13 of rows
    // 8 (l / 13) .. + 7, lanes 26-31 the scales of rows l - 26, + 6, + 12.
    // Rows past N read row N - 1; their sums are never written. ----
    const uint32_t ring_s = smem_addr(ring);
    const int cpart = lane % 13, chalf = lane / 13;
    int i_item = 0, i_q = 0, issued = 0, row0 = 0;
    auto item_rows = [&](int it) { row0 = (tile_lo + warp + 8 * it) * 16; };
    if (n_items > 0) item_rows(0);
    auto issue = [&](int slot) {
        if (issued < n_st) {
            const uint32_t base = ring_s + (uint32_t)(slot * kF3mStageBytes);
            const int g0 = gA + kF3mQuad * i_q;
            if (lane < 26) {
                const uint8_t* src = a.packed + (size_t)g0 * 26 + cpart * 8;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int rr = 8 * chalf + r;
                    cp_async8(base + (uint32_t)(rr * kF3mRowBytes + cpart * 8),
                              src + (size_t)min(row0 + rr, N - 1) * pitch);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int rr = lane - 26 + 6 * k;
                    if (rr < 16)
                        cp_async8(base + (uint32_t)(kF3mCodeBytes + rr * 8),
                                  a.scales + (size_t)min(row0 + rr, N - 1) * G + g0);
                }
            }
            ++issued;
            if (++i_q == nq) {
                i_q = 0;
                if (++i_item < n_items) item_rows(i_item);
            }
        }
        cp_async_commit();   // one group per stage, empty past the end, so the waits count uniformly
    };

    pdl_launch_dependents();
    // the weights are never the previous kernel's output: the first stages go
    // out before the PDL wait
#pragma unroll
    for (int i = 0; i < kF3mDepth; ++i) issue(i);

    // the byte table, a copy per lane l % 16 (lanes l and l + 16 share theirs):
    // entry v of lane (gid, t) holds v's five codes shifted left by 8 - r0(t),
    // where r0(t) = 2 (32 t mod 5) is the number of bits of the lane's first
    // byte that belong to the lane before it (0, 4, 8, 2 for t = 0..3), so
    // that the assembly below shifts by amounts that are the same for every
    // lane
    for (int v = threadIdx.x; v < 256; v += kF3Threads) {
        int c = 0, r = v;
#pragma unroll
        for (int d = 0; d < 5; ++d) {
            c |= ((r % 3) & 3) << (2 * d);
            r /= 3;
        }
        if (v >= 243) c = v & 0x3FF;   // not a pack's byte: some codes, never out of bounds
        uint32_t* row = reinterpret_cast<uint32_t*>(smem + kF3mRingBytes) + v * 16;
        const uint32_t sh4[4] = {(uint32_t)c << 8, (uint32_t)c << 4, (uint32_t)c, (uint32_t)c << 6};
#pragma unroll
        for (int l = 0; l < 16; ++l) row[l] = sh4[l & 3];
    }
    pdl_wait();

    __shared__ unsigned cleared_warps, seen_warps;
    const bool clearer = S > 1 && sigma == 0;
    const bool adder = S > 1 && sigma != 0;
    unsigned* const flag = g_f3_flags + clu;
    if (threadIdx.x == 0) {
        cleared_warps = 0u;
        seen_warps = 0u;
    }
    if (clearer)
        for (int it = 0; it < n_items; ++it) {
            const int row0c = (tile_lo + warp + 8 * it) * 16;
            for (int i = lane; i < 16 * M; i += 32) {
                const int m = i >> 4, r = row0c + (i & 15);
                if (r < N) a.y[(size_t)m * N + r] = 0.0f;
            }
        }

    // ---- the slice's activation, as the decode product stages it.  One
    // token: lane (gid, t) of a warp takes group gA + 8 b + gid of block b.
    // Several: item (g, nt) of the Gs x MT, warp w taking items w, w + 8, ...;
    // lane (gid, t) holds token 8 nt + gid. ----
    if constexpr (ONE) {
        for (int blk = warp; blk * 8 < Gs; blk += 8) {
            const int gl = blk * 8 + gid;
            const bool ok = gl < Gs;
            float v[32];
            if (ok) {
                const uint4* s4 = reinterpret_cast<const uint4*>(a.x + (size_t)(gA + gl) * 128 + 32 * t);
    #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = s4[q];
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * q + 2 * e] = __uint_as_float(uw[e] << 16);
                        v[8 * q + 2 * e + 1] = __uint_as_float(uw[e] & 0xFFFF0000u);
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
            f3_check_stage_range(mx);
            const int E = stage_exponent(mx);
            uint32_t b[16];
    #pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float c = stage_multiplier(E, j);
                const __half2 lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);
                const __half2 hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c);
                b[2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
                b[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            if (ok) {
    #pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(bfr + gl * 64 + q * 16 + t * 4) =
                        make_uint4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
            }
            // the ones pass of the block's eight groups: column n is group 8 b + n
            float acc1[4];
            const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
            unit_chain(acc1, ones, b);
            const float c_lo = __shfl_sync(0xffffffffu, acc1[0], gid >> 1);
            const float c_hi = __shfl_sync(0xffffffffu, acc1[1], gid >> 1);
            const float F = __uint_as_float((uint32_t)(14 - E + 127) << 23);   // 2^(14-E)
            if (ok && t == 0) fcs[gl] = make_float2(F, F * ((gid & 1) ? c_hi : c_lo));
        }
    } else {
        for (int item = warp; item < Gs * MT; item += 8) {
            const int g = item / MT, nt = item - g * MT;
            const int m = nt * 8 + gid;
            float v[32];
            if (m < M) {
                const uint4* s4 =
                    reinterpret_cast<const uint4*>(a.x + (size_t)m * a.K + (size_t)(gA + g) * 128 + 32 * t);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = s4[q];
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * q + 2 * e] = __uint_as_float(uw[e] << 16);
                        v[8 * q + 2 * e + 1] = __uint_as_float(uw[e] & 0xFFFF0000u);
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
            f3_check_stage_range(mx);
            const int E = stage_exponent(mx);
            uint32_t b[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float c = stage_multiplier(E, j);
                const __half2 lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);
                const __half2 hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c);
                b[2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
                b[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            unsigned char* fp = frag + (size_t)item * 2048 + lane * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(fp + q * 512) = make_uint4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
            // the all-ones pass: column n is token 8 nt + n; lane (., t) holds
            // tokens 2t and 2t + 1, whose F the lanes of rows 2t and 2t + 1 hold
            float acc1[4];
            const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
            unit_chain(acc1, ones, b);
            const float F = __uint_as_float((uint32_t)(14 - E + 127) << 23);
            const float F0 = __shfl_sync(0xffffffffu, F, (2 * t) * 4);
            const float F1 = __shfl_sync(0xffffffffu, F, (2 * t + 1) * 4);
            if (gid == 0)
                *reinterpret_cast<float4*>(corr + ((size_t)item * 4 + t) * 16) =
                    make_float4(F0, F0 * acc1[0], F1, F1 * acc1[1]);
        }
    }
    __syncthreads();

    auto count_cleared = [&]() {
        __threadfence();
        __syncwarp();
        if (lane == 0 && atomicAdd(&cleared_warps, 1u) == 7u) red_inc(flag, (unsigned)(S - 1));
    };
    auto count_seen = [&]() {
        if (lane == 0 && atomicAdd(&seen_warps, 1u) == 7u) red_inc(flag, (unsigned)(S - 1));
    };
    if (clearer && n_st == 0) count_cleared();
    if (adder && n_st == 0) count_seen();

    // ---- the stages ----
    // this lane's bytes of a group: b0 .. b0 + 7, the first r0(t) bits of b0's
    // codes dropped (the table's shift accounts for them)
    const int b0 = (32 * t) / 5;
    const uint32_t* const lut_l = lut + (lane & 15);
    unsigned flag_seen = 0u;
    bool add_ok = true;
    int s = 0;
    for (int it = 0; it < n_items; ++it) {
        // rows gid and gid + 8; several tokens: tokens 8 nt + 2t and 8 nt + 2t + 1
        float y0 = 0.0f, y1 = 0.0f;
        float yt[MT][4];
#pragma unroll
        for (int nt = 0; nt < MT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) yt[nt][e] = 0.0f;
        for (int q = 0; q < nq; ++q, ++s) {
            const int slot = s & (kF3mDepth - 1);
            cp_async_wait<kF3mDepth - 1>();
            __syncwarp();
            const unsigned char* st = ring + slot * kF3mStageBytes;
            const uint2 sc0 = *reinterpret_cast<const uint2*>(st + kF3mCodeBytes + gid * 8);
            const uint2 sc1 = *reinterpret_cast<const uint2*>(st + kF3mCodeBytes + (gid + 8) * 8);
            const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sc0.x));
            const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sc0.y));
            const float2 r01 = __half22float2(*reinterpret_cast<const __half2*>(&sc1.x));
            const float2 r23 = __half22float2(*reinterpret_cast<const __half2*>(&sc1.y));
            const float s0[4] = {s01.x, s01.y, s23.x, s23.y};
            const float s1[4] = {r01.x, r01.y, r23.x, r23.y};
#pragma unroll
            for (int u = 0; u < kF3mQuad; ++u) {
                // the two code words of rows gid and gid + 8
                uint32_t wd[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int off = (gid + 8 * h) * kF3mRowBytes + 26 * u + b0;
                    const uint32_t* wp = reinterpret_cast<const uint32_t*>(st + (off & ~3));
                    const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
                    const uint32_t sh = (uint32_t)(off & 3) * 8u;
                    const uint32_t x0 = __funnelshift_r(w0, w1, sh), x1 = __funnelshift_r(w1, w2, sh);
                    uint32_t L[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t byte = __byte_perm(i < 4 ? x0 : x1, 0u, 0x4440u | (uint32_t)(i & 3));
                        L[i] = lut_l[byte * 16];
                    }
                    // L[i] = byte i's codes << (8 - r0): they sit at bits
                    // 10 i - r0 of the lane's 64-bit code stream, so each
                    // part lands by a fixed shift and the parts never overlap
                    // (a sum is their OR); byte 7 reaches bits 30-31 of the
                    // second word only when r0 = 8 and shifts out otherwise
                    wd[h][0] = (L[0] >> 8) + (L[1] << 2) + (L[2] << 12) + (L[3] << 22);
                    wd[h][1] = (L[3] >> 10) + L[4] + (L[5] << 10) + (L[6] << 20) + (L[7] << 30);
                }
                const uint32_t w[4] = {wd[0][0], wd[1][0], wd[0][1], wd[1][1]};
                const int gl = kF3mQuad * q + u;
                if constexpr (ONE) {
                    const uint4* bp = reinterpret_cast<const uint4*>(bfr + gl * 64 + t * 4);
                    uint32_t b[16];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint4 z = bp[qq * 4];
                        b[4 * qq] = z.x;
                        b[4 * qq + 1] = z.y;
                        b[4 * qq + 2] = z.z;
                        b[4 * qq + 3] = z.w;
                    }
                    float acc[4];
                    unit_chain(acc, w, b);
                    const float2 fc = fcs[gl];
                    y0 = fmaf(s0[u], fmaf(fc.x, acc[0], -fc.y), y0);
                    y1 = fmaf(s1[u], fmaf(fc.x, acc[2], -fc.y), y1);
                } else {
                    uint32_t b[MT][16];
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        const unsigned char* fp = frag + (size_t)(gl * MT + nt) * 2048 + lane * 16;
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const uint4 z = *reinterpret_cast<const uint4*>(fp + qq * 512);
                            b[nt][4 * qq] = z.x;
                            b[nt][4 * qq + 1] = z.y;
                            b[nt][4 * qq + 2] = z.z;
                            b[nt][4 * qq + 3] = z.w;
                        }
                    }
                    float acc[MT][4];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t r[4];
                        slot_regs<false>(j, w[0], w[1], w[2], w[3], r);
#pragma unroll
                        for (int nt = 0; nt < MT; ++nt)
                            mma16816(acc[nt], r[0], r[1], r[2], r[3], b[nt][2 * j], b[nt][2 * j + 1], j > 0);
                    }
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        const float4 f = *reinterpret_cast<const float4*>(corr + ((size_t)(gl * MT + nt) * 4 + t) * 16);
                        yt[nt][0] = fmaf(s0[u], fmaf(f.x, acc[nt][0], -f.y), yt[nt][0]);   // row gid,     token 2t
                        yt[nt][1] = fmaf(s0[u], fmaf(f.z, acc[nt][1], -f.w), yt[nt][1]);   // row gid,     token 2t+1
                        yt[nt][2] = fmaf(s1[u], fmaf(f.x, acc[nt][2], -f.y), yt[nt][2]);   // row gid + 8, token 2t
                        yt[nt][3] = fmaf(s1[u], fmaf(f.z, acc[nt][3], -f.w), yt[nt][3]);   // row gid + 8, token 2t+1
                    }
                }
            }
            __syncwarp();
            issue(slot);
            if (s == 0) {
                if (clearer) count_cleared();
                if (adder && lane == 0) flag_seen = ld_acquire_gpu(flag);
            }
        }
        const int row = (tile_lo + warp + 8 * it) * 16 + gid;
        if (adder && it == 0) {
            int ok = 1;
            if (lane == 0) {
                ok = flag_seen != 0u || wait_flag_nonzero(flag, kFlagWaitNs);
                if (!ok) report_device_error(&g_f3_error, kDevErrGemvConsumerWait);
            }
            add_ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (add_ok) count_seen();
        }
        auto put = [&](int m, int r, float v) {
            if (m < M && r < N) {
                float* p = a.y + (size_t)m * N + r;
                if (S == 1) *p = v;
                else atomicAdd(p, v);
            }
        };
        if (add_ok) {
            if constexpr (ONE) {
                if (t == 0) {
                    put(0, row, y0);
                    put(0, row + 8, y1);
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < MT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) put(nt * 8 + 2 * t + (e & 1), row + 8 * (e >> 1), yt[nt][e]);
            }
        }
    }
    cp_async_wait<0>();
}


// per group: the staged activation and its correction (one token: 256 + 8
// bytes; MT token tiles: MT x (2048 + 64))
size_t f3m_smem(int Gs, int per_group) { return (size_t)kF3mRingBytes + kF3mLutBytes + (size_t)Gs * per_group; }

// The one-token plan: slices of whole quads and ranges of tiles, as the
// tile-major decode loop plans them (the longest warp's stages against the
// extra CTAs and additions of more slices), at most kF3mMaxRanges ranges;
// several slices only when K spans more than one 1024-wide slice.
struct F3mPlan {
    int S, cps, ctas;
    size_t smem;
};
bool f3m_plan(int N, int K, int per_group, int sms, int optin, F3mPlan* out) {
    const int G = K / 128, Gq = G / kF3mQuad, T = (N + 15) / 16;
    double best = 0.0;
    F3mPlan bp{};
    for (int S = 1; S <= Gq && S <= 64; ++S) {
        if (S > 1 && G <= 8) break;
        const int qmax = (Gq + S - 1) / S;
        const size_t sm = f3m_smem(kF3mQuad * qmax, per_group);
        if (sm > (size_t)optin) continue;
        const int per_sm = std::min(kF3mCtasPerSm, (int)((228 * 1024) / (sm + 1024)));
        if (per_sm < 1) continue;
        const int slots = sms * per_sm;
        const int cps = std::max(1, std::min(std::min(T, kF3mMaxRanges), slots / S));
        const int rmax = (T + cps - 1) / cps;
        const int items = (rmax + 7) / 8;
        const long long waves = ((long long)S * cps + slots - 1) / slots;
        const double cost = (double)waves * (items * (qmax + 0.5) + 1.0 + (S > 1 ? 0.5 : 0.0));
        if (bp.ctas == 0 || cost < best) {
            best = cost;
            bp = F3mPlan{S, cps, S * cps, sm};
        }
    }
    if (bp.ctas == 0) return false;
    *out = bp;
    return true;
}

size_t f3_smem_bytes(int M) { return (size_t)(kF3Lut + M * kF3Chunk) * sizeof(float); }

}  // namespace
}  // namespace tern

using namespace tern;

namespace tern {
// Reads and clears the base-3 product's device error word.  A reported error
// may have stopped a call before its range flags counted back to 0 (a slice
// that gave up its wait never counts), so the flags are cleared with it: the
// next call starts from zeros again.  The caller has synchronised the device.
cudaError_t read_f3_device_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_f3_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int z = 0;
        e = cudaMemcpyToSymbol(g_f3_error, &z, sizeof(int));
        if (e != cudaSuccess) return e;
        void* flags = nullptr;
        e = cudaGetSymbolAddress(&flags, g_f3_flags);
        if (e != cudaSuccess) return e;
        e = cudaMemset(flags, 0, sizeof(g_f3_flags));
        if (e != cudaSuccess) return e;
    }
    *code = v;
    return cudaSuccess;
}
}  // namespace tern

extern "C" size_t tern_f3_packed_bytes(int N, int K) {
    if (N < 0 || K < 0 || K % 128 != 0) return 0;
    return (size_t)N * 26 * (K / 128);
}

extern "C" tern_status tern_f3_pack(const int8_t* t, int N, int K, uint8_t* packed, int* bad_count,
                                    tern_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || K < 0 || K % 128 != 0) return TERN_ERR_SHAPE;
    if ((long long)N * K >= (1LL << 40)) return TERN_ERR_SHAPE;
    if (N == 0 || K == 0) return TERN_OK;
    if (!t || !packed) return TERN_ERR_NULL;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const long long bytes = (long long)N * 26 * (K / 128);
    const int grid = (int)std::min<long long>((bytes + 255) / 256, (long long)sms * 16);
    f3_pack_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(t, packed, N, K, bad_count);
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}

extern "C" tern_status tern_f3_gemv(const void* x, const uint8_t* packed, const void* scales, float* y, int M,
                                    int N, int K, tern_stream_t stream) {
    set_launch_count(0);
    if (M < 1 || M > kF3MaxM || N < 1 || K < 128 || K % 128 != 0) return TERN_ERR_SHAPE;
    if ((long long)N * K >= (1LL << 40)) return TERN_ERR_SHAPE;
    if (!x || !packed || !scales || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales) || !aligned16(y)) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const size_t smem = f3_smem_bytes(M);
    static bool set_for[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TERN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!set_for[dev]) {
            if (cudaFuncSetAttribute(f3_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)f3_smem_bytes(kF3MaxM)) != cudaSuccess ||
                cudaFuncSetAttribute(f3_gemv_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kF3TabMaxM * kF3TabPerToken * sizeof(float))) != cudaSuccess)
                return TERN_ERR_CUDA;
            set_for[dev] = true;
        }
    }
    cudaError_t e;
    if (K % (kF3mQuad * 128) == 0) {
        // the tensor pipe: one token, one token tile (up to 8) or two
        const int kind = M == 1 ? 0 : (M <= 8 ? 1 : 2);
        const int per_group = kind == 0 ? 256 + 8 : (kind == 1 ? 2048 + 64 : 2 * (2048 + 64));
        auto kern = kind == 0 ? f3_mma_kernel<1, true> : (kind == 1 ? f3_mma_kernel<1, false> : f3_mma_kernel<2, false>);
        static int optin_of[64][3] = {};
        static F3mPlan plan_of[64][16];
        static int plan_key[64][16][3];
        static int plan_n[64] = {};
        F3mPlan p{};
        bool have = false;
        {
            std::lock_guard<std::mutex> lk(mu);
            if (!optin_of[dev][kind]) {
                int optin = 0;
                cudaFuncAttributes fa;
                if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
                    cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
                    return TERN_ERR_CUDA;
                optin -= (int)fa.sharedSizeBytes;
                if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
                    return TERN_ERR_CUDA;
                optin_of[dev][kind] = optin;
            }
            for (int i = 0; i < plan_n[dev]; ++i)
                if (plan_key[dev][i][0] == N && plan_key[dev][i][1] == K && plan_key[dev][i][2] == kind) {
                    p = plan_of[dev][i];
                    have = true;
                }
            if (!have) {
                if (!f3m_plan(N, K, per_group, sms, optin_of[dev][kind], &p)) return TERN_ERR_SHAPE;
                const int slot = plan_n[dev] < 16 ? plan_n[dev]++ : (N + K + kind) % 16;
                plan_key[dev][slot][0] = N;
                plan_key[dev][slot][1] = K;
                plan_key[dev][slot][2] = kind;
                plan_of[dev][slot] = p;
            }
        }
        F3mArgs args{reinterpret_cast<const __nv_bfloat16*>(x), packed, reinterpret_cast<const __half*>(scales), y,
                     M, N, K, K / 128, (N + 15) / 16, p.S, p.cps};
        e = launch_pdl(kern, dim3(p.ctas), dim3(kF3Threads), p.smem, (cudaStream_t)stream, true, args);
    } else if (M <= kF3TabMaxM) {
        // persistent: kF3TabCtasPerSm CTAs per SM, at most kF3TabRowsPerWarp rows per warp
        const int per_cta_cap = kF3Warps * kF3TabRowsPerWarp;
        const int ctas = std::max((N + per_cta_cap - 1) / per_cta_cap, std::min(N, kF3TabCtasPerSm * sms));
        const int rows_per_cta = (N + ctas - 1) / ctas;
        const int grid = (N + rows_per_cta - 1) / rows_per_cta;
        e = launch_pdl(f3_gemv_table_kernel, dim3(grid), dim3(kF3Threads),
                       (size_t)M * kF3TabPerToken * sizeof(float), (cudaStream_t)stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), packed, reinterpret_cast<const __half*>(scales), y,
                       M, N, K, rows_per_cta);
    } else {
        const int rows_per_cta = kF3Warps * kF3RowsPerWarp;
        const int grid = (N + rows_per_cta - 1) / rows_per_cta;
        e = launch_pdl(f3_gemv_kernel, dim3(grid), dim3(kF3Threads), smem, (cudaStream_t)stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), packed, reinterpret_cast<const __half*>(scales), y, M,
                       N, K);
    }
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}
