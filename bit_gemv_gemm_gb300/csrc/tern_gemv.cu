// tern_gemv.cu -- decode / small-batch ternary-g128 product, M = 1..16.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} x[m][k] * (q[n][k] - 1)
//
// ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card: ternary g128 weights,
// "Weight representation"; codes unpacked and scaled inside the product,
// "CUDA (NVIDIA GPUs)"; decode is the memory-bandwidth-bound phase,
// "Cross-platform throughput".)
//
// Design.  At 2.125 bits per weight an M = 1 product must retire ~25 G
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
//   * the activation is staged once per call (the prologue kernel) as fp16 in
//     the MMA B-fragment order, with each value pre-multiplied by the power of
//     two 2^(E + 10 - 2j') that undoes its slot's 2^(2j' - 24) (j' = j or j - 6)
//     and a per-(token, group) exponent E chosen from the group's max |x| so the
//     largest staged value is below 2^15.  Every staged value is exact (bf16
//     has 8 significant bits, fp16 11).  One MMA per slot position j then
//     accumulates 2^(E - 14) * sum q x over 16 weights of 16 rows.
//   * per 128-weight group and row, y += s_g * (2^(14 - E) * acc - sum_{k in g} x_k):
//     the -1 of q - 1 becomes a per-(token, group) sum of x shared by all rows.
//
// Work split: stream-K over (16-row tile, group) units, a contiguous range per
// warp of a persistent grid, partial row sums combined with fp32 atomics into
// y (zeroed by the prologue).  Codes and scales are streamed with 8-byte loads
// straight into registers, D groups ahead; the first D are issued before the
// programmatic-dependent-launch wait, so the stream starts while the prologue
// (and the previous kernel) finish.
#include "tern_fwht.cuh"

namespace tern {
namespace {

constexpr int kGroup = 128;            // weights per scale
constexpr int kWordsPerGroup = 8;      // uint32 words of codes per group per row
constexpr int kXsfWords = 64;          // staged fp16x2 words per (token, group)
constexpr int kPrepThreads = 256;      // 8 warps = 8 groups per prologue CTA

constexpr int kGemvWarps = 8;          // warps per CTA
constexpr int kGemvDepth = 4;          // groups in flight per warp
// resident CTAs per SM: 3 for one 8-token tile (<= 85 registers), 2 for two
template <int MT> constexpr int gemv_ctas_per_sm() { return MT == 1 ? 3 : 2; }

struct Workspace {
    uint32_t* xsf;   // [M][G][4][16] staged activation, fp16x2
    float2* fs;      // [G][MP]: (2^(14-E), sum of x over the group)
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ inline size_t ws_xsf_bytes(int M, int G) { return (size_t)M * G * kXsfWords * 4; }
__host__ inline size_t ws_fs_bytes(int MP, int G) { return (size_t)G * MP * sizeof(float2); }

// ---------------------------------------------------------------------------
// Prologue: stage one (token, group) from the four values each lane holds.
// Lane l = 8 t + j holds x[128 g + 32 t + j + 8 u], u = 0..3 (v[u]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stage_group(const float (&v)[4], int lane, uint32_t* __restrict__ xsf_mg,
                                            float2* __restrict__ fs_gm) {
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    float sx = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sx += __shfl_xor_sync(0xffffffffu, sx, o);
    }
    int E = 0;
    if (mx > 0.0f && mx <= 3.0e38f) {
        int ex;
        frexpf(mx, &ex);            // mx < 2^ex
        E = 5 - ex;                 // mx * 2^(E + 10) < 2^15
        E = max(-100, min(E, 150));
    }
    const int t = lane >> 3, j = lane & 7;
    const int jp = j < 6 ? j : j - 6;
    const float c = ldexpf(1.0f, E + 10 - 2 * jp);   // exact power of two
    const __half2 lo = __floats2half2_rn(v[0] * c, v[1] * c);  // k = 32t+j, 32t+j+8
    const __half2 hi = __floats2half2_rn(v[2] * c, v[3] * c);  // k = 32t+16+j, 32t+24+j
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t*>(&lo);
    out.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(xsf_mg + t * 16 + 2 * j) = out;
    if (lane == 0) *fs_gm = make_float2(ldexpf(1.0f, 14 - E), sx);
}

// Zeroes the padded (token >= M) entries of fs and this CTA's share of y.
__device__ __forceinline__ void prologue_zero(float* __restrict__ y, float2* __restrict__ fs, int M, int MP,
                                              int N, int G, int cta, int ctas) {
    const int tid = threadIdx.x;
    if (cta == 0) {
        for (int i = tid; i < G * (MP - M); i += blockDim.x) {
            const int g = i / (MP - M), m = M + i % (MP - M);
            fs[(size_t)g * MP + m] = make_float2(0.0f, 0.0f);
        }
    }
    const size_t total = (size_t)M * N;
    const size_t per = (total + ctas - 1) / ctas;
    const size_t lo = per * cta, hi = min(total, lo + per);
    for (size_t i = lo + tid; i < hi; i += blockDim.x) y[i] = 0.0f;
}

// Plain prologue: grid (ceil(G/8), M); one warp per (token, group).
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(const __nv_bfloat16* __restrict__ x, Workspace ws, float* __restrict__ y, int M, int MP,
            int N, int K) {
    pdl_launch_dependents();
    pdl_wait();
    const int G = K / kGroup;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.y;
    const int g = blockIdx.x * (kPrepThreads / 32) + warp;
    if (g < G) {
        const int t = lane >> 3, j = lane & 7;
        const __nv_bfloat16* xg = x + (size_t)m * K + (size_t)g * kGroup + 32 * t + j;
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __bfloat162float(xg[8 * u]);
        stage_group(v, lane, ws.xsf + ((size_t)m * G + g) * kXsfWords, ws.fs + (size_t)g * MP + m);
    }
    prologue_zero(y, ws.fs, M, MP, N, G, blockIdx.y * gridDim.x + blockIdx.x, gridDim.x * gridDim.y);
}

// Rotation-fused prologue: grid (K/4096, M).  The CTA rotates its 4096-block
// in shared memory (fp32), then stages the block's 32 groups from there, so the
// rotated activation is never rounded to bf16 nor written out.
__global__ void __launch_bounds__(kFwhtThreads)
prep_rot_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs, Workspace ws,
                float* __restrict__ y, int M, int MP, int N, int K) {
    __shared__ float sm[kFwhtSmemFloats];
    pdl_launch_dependents();
    pdl_wait();
    const int G = K / kGroup;
    const int b = blockIdx.x, m = blockIdx.y;
    fwht4096_block(x + (size_t)m * K + (size_t)b * kFwhtN, signs + (size_t)b * kFwhtN, sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = lane >> 3, j = lane & 7;
    for (int gl = warp; gl < kFwhtN / kGroup; gl += kFwhtThreads / 32) {
        const int g = b * (kFwhtN / kGroup) + gl;
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = sm[fwht_pos(gl * kGroup + 32 * t + j + 8 * u)];
        stage_group(v, lane, ws.xsf + ((size_t)m * G + g) * kXsfWords, ws.fs + (size_t)g * MP + m);
    }
    prologue_zero(y, ws.fs, M, MP, N, G, blockIdx.y * gridDim.x + blockIdx.x, gridDim.x * gridDim.y);
}

// ---------------------------------------------------------------------------
// Main kernel.
// ---------------------------------------------------------------------------
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

__device__ __forceinline__ uint2 ldg_stream_u2(const uint32_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

struct Stage {
    uint2 c0, c1;        // codes: row r0 words (2t, 2t+1), row r1 words (2t, 2t+1)
    uint32_t s0, s1;     // fp16 scale bits of rows r0, r1
};

template <int MT, int D>
__global__ void __launch_bounds__(kGemvWarps * 32, gemv_ctas_per_sm<MT>())
gemv_kernel(const uint32_t* __restrict__ codes, const __half* __restrict__ scales, Workspace ws,
            float* __restrict__ y, int M, int N, int K) {
    pdl_launch_dependents();
    const int G = K / kGroup;
    const int W = K / 16;
    const int MP = MT * 8;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int T = (N + 15) >> 4;
    const long long U = (long long)T * G;
    const long long TW = (long long)gridDim.x * kGemvWarps;
    const long long gw = (long long)blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    const int u0 = (int)(U * gw / TW), u1 = (int)(U * (gw + 1) / TW);
    const int n_units = u1 - u0;
    if (n_units <= 0) return;

    // load cursor
    int ld_tile = u0 / G, ld_g = u0 - ld_tile * G;
    Stage st[D];
    auto load_stage = [&](Stage& s) {
        const int r0 = ld_tile * 16 + gid, r1 = r0 + 8;
        const int w = ld_g * kWordsPerGroup + 2 * t;
        if (r0 < N) {
            s.c0 = ldg_stream_u2(codes + (size_t)r0 * W + w);
            s.s0 = ldg_stream_u16(scales + (size_t)r0 * G + ld_g);
        } else {
            s.c0 = make_uint2(0u, 0u);
            s.s0 = 0u;
        }
        if (r1 < N) {
            s.c1 = ldg_stream_u2(codes + (size_t)r1 * W + w);
            s.s1 = ldg_stream_u16(scales + (size_t)r1 * G + ld_g);
        } else {
            s.c1 = make_uint2(0u, 0u);
            s.s1 = 0u;
        }
        if (++ld_g == G) { ld_g = 0; ++ld_tile; }
    };
#pragma unroll
    for (int s = 0; s < D; ++s)
        if (s < n_units) load_stage(st[s]);

    // The activation staging (and y's zeroing) come from the prologue kernel.
    pdl_wait();

    int tile = u0 / G, g = u0 - tile * G;
    float ysum[MT][4];
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) ysum[nt][i] = 0.0f;

    for (int base = 0; base < n_units; base += D) {
#pragma unroll
        for (int s = 0; s < D; ++s) {
            const int i = base + s;
            if (i < n_units) {
                // B fragments and (2^(14-E), sum x) for this group
                uint32_t b[MT][16];
                float4 fsv[MT];
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) {
                    const int m = nt * 8 + gid;
                    if (m < M) {
                        const uint4* src = reinterpret_cast<const uint4*>(
                            ws.xsf + ((size_t)m * G + g) * kXsfWords + t * 16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = __ldg(src + q);
                            b[nt][4 * q + 0] = v.x;
                            b[nt][4 * q + 1] = v.y;
                            b[nt][4 * q + 2] = v.z;
                            b[nt][4 * q + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) b[nt][q] = 0u;
                    }
                    fsv[nt] = __ldg(reinterpret_cast<const float4*>(ws.fs + (size_t)g * MP + nt * 8 + 2 * t));
                }
                const Stage cur = st[s];
                if (i + D < n_units) load_stage(st[s]);

                float acc[MT][4];
                const uint32_t sh0x = cur.c0.x >> 12, sh1x = cur.c1.x >> 12;
                const uint32_t sh0y = cur.c0.y >> 12, sh1y = cur.c1.y >> 12;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t a0, a1, a2, a3;
                    if (j < 6) {
                        const uint32_t mk = 0x00030003u << (2 * j);
                        a0 = cur.c0.x & mk;
                        a1 = cur.c1.x & mk;
                        a2 = cur.c0.y & mk;
                        a3 = cur.c1.y & mk;
                    } else {
                        const uint32_t mk = 0x00030003u << (2 * (j - 6));
                        a0 = sh0x & mk;
                        a1 = sh1x & mk;
                        a2 = sh0y & mk;
                        a3 = sh1y & mk;
                    }
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt)
                        mma16816(acc[nt], a0, a1, a2, a3, b[nt][2 * j], b[nt][2 * j + 1], j > 0);
                }
                const float sc0 = __half2float(__ushort_as_half((unsigned short)cur.s0));
                const float sc1 = __half2float(__ushort_as_half((unsigned short)cur.s1));
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) {
                    const float4 f = fsv[nt];   // (F, Sx) of tokens 2t and 2t+1
                    ysum[nt][0] = fmaf(sc0, fmaf(f.x, acc[nt][0], -f.y), ysum[nt][0]);
                    ysum[nt][1] = fmaf(sc0, fmaf(f.z, acc[nt][1], -f.w), ysum[nt][1]);
                    ysum[nt][2] = fmaf(sc1, fmaf(f.x, acc[nt][2], -f.y), ysum[nt][2]);
                    ysum[nt][3] = fmaf(sc1, fmaf(f.z, acc[nt][3], -f.w), ysum[nt][3]);
                }
                // end of this tile's range: fold the partial sums into y
                if (g == G - 1 || i == n_units - 1) {
                    const int r0 = tile * 16 + gid, r1 = r0 + 8;
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
                        if (r0 < N) {
                            if (m0 < M) atomicAdd(y + (size_t)m0 * N + r0, ysum[nt][0]);
                            if (m1 < M) atomicAdd(y + (size_t)m1 * N + r0, ysum[nt][1]);
                        }
                        if (r1 < N) {
                            if (m0 < M) atomicAdd(y + (size_t)m0 * N + r1, ysum[nt][2]);
                            if (m1 < M) atomicAdd(y + (size_t)m1 * N + r1, ysum[nt][3]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) ysum[nt][q] = 0.0f;
                    }
                }
                if (++g == G) { g = 0; ++tile; }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
tern_status validate(const void* x, const uint32_t* codes, const void* scales, const float* y, int M, int N,
                     int K, void* workspace, size_t workspace_bytes, size_t need) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return TERN_ERR_SHAPE;
    // unit counts and indices stay in 32 bits
    if ((long long)((N + 15) / 16) * (K / kGroup) >= (1LL << 31) || (long long)N * (K / 16) >= (1LL << 40))
        return TERN_ERR_SHAPE;
    if (!x || !codes || !scales || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y)) return TERN_ERR_ALIGN;
    if (!workspace || workspace_bytes < need) return TERN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
    return TERN_OK;
}

template <int MT>
cudaError_t launch_gemv(const uint32_t* codes, const __half* scales, Workspace ws, float* y, int M, int N,
                        int K, int sms, cudaStream_t stream) {
    const long long U = (long long)((N + 15) / 16) * (K / kGroup);
    long long ctas = (long long)sms * gemv_ctas_per_sm<MT>();
    const long long need = (U + kGemvWarps - 1) / kGemvWarps;
    if (ctas > need) ctas = need;
    return launch_pdl(gemv_kernel<MT, kGemvDepth>, dim3((unsigned)ctas), dim3(kGemvWarps * 32), 0, stream,
                      true, codes, scales, ws, y, M, N, K);
}

tern_status run(const void* x, const int8_t* signs, const uint32_t* codes, const void* scales, float* y,
                int M, int N, int K, void* workspace, cudaStream_t stream) {
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const int G = K / kGroup, MT = (M + 7) / 8, MP = 8 * MT;
    Workspace ws;
    ws.xsf = reinterpret_cast<uint32_t*>(workspace);
    ws.fs = reinterpret_cast<float2*>(reinterpret_cast<char*>(workspace) + align_up(ws_xsf_bytes(M, G), 256));
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
    cudaError_t e;
    if (signs) {
        e = launch_pdl(prep_rot_kernel, dim3(K / kFwhtN, M), dim3(kFwhtThreads), 0, stream, true, xb, signs, ws,
                       y, M, MP, N, K);
    } else {
        e = launch_pdl(prep_kernel, dim3((G + 7) / 8, M), dim3(kPrepThreads), 0, stream, true, xb, ws, y, M, MP,
                       N, K);
    }
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    const __half* sc = reinterpret_cast<const __half*>(scales);
    e = MT == 1 ? launch_gemv<1>(codes, sc, ws, y, M, N, K, sms, stream)
                : launch_gemv<2>(codes, sc, ws, y, M, N, K, sms, stream);
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(2);
    return TERN_OK;
}

}  // namespace
}  // namespace tern

using namespace tern;

extern "C" size_t tern_gemv_workspace_bytes(int M, int N, int K) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return 0;
    const int G = K / kGroup, MP = 8 * ((M + 7) / 8);
    return align_up(ws_xsf_bytes(M, G), 256) + align_up(ws_fs_bytes(MP, G), 256);
}

extern "C" tern_status tern_gemv(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                 int N, int K, void* workspace, size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K, workspace, workspace_bytes,
                                   tern_gemv_workspace_bytes(M, N, K));
    if (v != TERN_OK) return v;
    return run(x, nullptr, codes, scales, y, M, N, K, workspace, (cudaStream_t)stream);
}

extern "C" tern_status tern_fwht_gemm(const void* x, const int8_t* signs, const uint32_t* codes,
                                      const void* scales, float* y, int M, int N, int K, void* workspace,
                                      size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    if (K % kFwhtN != 0) return TERN_ERR_SHAPE;
    const tern_status v = validate(x, codes, scales, y, M, N, K, workspace, workspace_bytes,
                                   tern_gemv_workspace_bytes(M, N, K));
    if (v != TERN_OK) return v;
    if (!signs) return TERN_ERR_NULL;
    if (!aligned16(signs)) return TERN_ERR_ALIGN;
    return run(x, signs, codes, scales, y, M, N, K, workspace, (cudaStream_t)stream);
}
