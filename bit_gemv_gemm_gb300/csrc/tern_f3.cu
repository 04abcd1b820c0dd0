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

size_t f3_smem_bytes(int M) { return (size_t)(kF3Lut + M * kF3Chunk) * sizeof(float); }

}  // namespace
}  // namespace tern

using namespace tern;

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
    if (M <= kF3TabMaxM) {
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
