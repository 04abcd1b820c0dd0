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
//   * the activation is staged as fp16 in the MMA B-fragment order, each value
//     pre-multiplied by the power of two 2^(E + 10 - 2j') that undoes its
//     slot's 2^(2j' - 24) (j' = j or j - 6), with a per-(token, group) exponent
//     E chosen from the group's max |x| so the largest staged value is below
//     2^15.  bf16 values stage exactly (8 significant bits into 11).  One MMA
//     per slot position j then accumulates acc = 2^(E - 14) sum_k q_k x_k over
//     16 weights of 16 rows.
//   * the -1 of q - 1: the same eight-MMA chain run once per (token, group)
//     on the all-ones code pattern gives acc1 = 2^(E - 14) sum_k x_k with the
//     very same rounding, and per row and group
//         y += s_g * (2^(14 - E) * acc - 2^(14 - E) * acc1),
//     so a row of zero weights (q = 1 everywhere) gives exactly 0.
//
// Work split.  K is cut into slices of up to 8 groups; a CTA owns one slice
// and a contiguous range of 16-row tiles.  The CTA stages its slice of the
// activation into shared memory once (warp w stages group w), then its eight
// warps split the (tile, group) units of the range, streaming codes and scales
// with 8-byte loads straight into registers, D units ahead (the first D are
// issued before the programmatic-dependent-launch wait).  Row partial sums go
// to shared-memory accumulators; with several slices, each CTA stores its
// partial tile sums to the workspace and the last CTA to finish a tile (an
// arrival counter) adds the slices in slice order and writes y.  y is written
// exactly once per element; no pre-zeroing and no global float atomics.
#include "tern_fwht.cuh"

namespace tern {
namespace {

constexpr int kGroup = 128;            // weights per scale
constexpr int kWordsPerGroup = 8;      // uint32 words of codes per group per row
constexpr int kFragWords = 64;         // staged fp16x2 words per (group, token)
constexpr int kSliceGroups = 8;        // groups per K-slice
constexpr int kWarps = 8;              // warps per CTA
constexpr int kMaxTiles = 32;          // row tiles per CTA chunk (shared accumulators)

template <int MT> struct GemvCfg;
template <> struct GemvCfg<1> { static constexpr int kCtasPerSm = 2, kDepth = 6; };
template <> struct GemvCfg<2> { static constexpr int kCtasPerSm = 1, kDepth = 6; };

template <int MT> constexpr size_t gemv_smem_bytes() {
    return (size_t)kSliceGroups * (8 * MT) * kFragWords * 4    // staged activation
           + (size_t)kSliceGroups * (8 * MT) * 8                // (F, F*acc1)
           + (size_t)kMaxTiles * 16 * (8 * MT) * 4              // row accumulators
           + (size_t)kMaxTiles * 4;                             // finalize flags
}

struct GemvArgs {
    const void* x;              // bf16 [M][K], or fp32 [M][K] when the rotation prologue ran
    const uint32_t* codes;      // [N][K/16]
    const __half* scales;       // [N][K/128]
    float* y;                   // [M][N]
    float* partial;             // [S][T][M][16]
    unsigned* counter;          // [T]
    int M, N, K, G, T, S, ks, cps;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

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

// Loads the B fragments (16 words) of one token from the staged slice.
__device__ __forceinline__ void load_frag(const uint32_t* __restrict__ src, bool valid, uint32_t (&b)[16]) {
    if (valid) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = s4[q];
            b[4 * q + 0] = v.x;
            b[4 * q + 1] = v.y;
            b[4 * q + 2] = v.z;
            b[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) b[q] = 0u;
    }
}

// The eight MMAs of one (16-row, 128-weight) unit: slot j's A registers come
// from the four code words by one AND (codes 6, 7, 14, 15 after a shift by 12).
__device__ __forceinline__ void unit_mmas(float (&acc)[4], uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                          const uint32_t (&b)[16]) {
    const uint32_t h0 = w0 >> 12, h1 = w1 >> 12, h2 = w2 >> 12, h3 = w3 >> 12;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t a0, a1, a2, a3;
        if (j < 6) {
            const uint32_t mk = 0x00030003u << (2 * j);
            a0 = w0 & mk;
            a1 = w1 & mk;
            a2 = w2 & mk;
            a3 = w3 & mk;
        } else {
            const uint32_t mk = 0x00030003u << (2 * (j - 6));
            a0 = h0 & mk;
            a1 = h1 & mk;
            a2 = h2 & mk;
            a3 = h3 & mk;
        }
        mma16816(acc, a0, a1, a2, a3, b[2 * j], b[2 * j + 1], j > 0);
    }
}

struct Stage {
    uint2 c0, c1;        // codes: row r0 words (2t, 2t+1), row r1 words (2t, 2t+1)
    uint32_t s0, s1;     // fp16 scale bits of rows r0, r1
};

template <int MT, bool XF32>
__global__ void __launch_bounds__(kWarps * 32, GemvCfg<MT>::kCtasPerSm)
gemv_kernel(const GemvArgs a) {
    constexpr int MP = 8 * MT;
    constexpr int D = GemvCfg<MT>::kDepth;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint32_t* bsm = reinterpret_cast<uint32_t*>(smem_raw);                       // [8][MP][64]
    float2* fcs = reinterpret_cast<float2*>(bsm + kSliceGroups * MP * kFragWords);  // [8][MP]
    float* accs = reinterpret_cast<float*>(fcs + kSliceGroups * MP);             // [kMaxTiles][16][MP]
    int* fin = reinterpret_cast<int*>(accs + kMaxTiles * 16 * MP);               // [kMaxTiles]

    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int M = a.M, N = a.N, G = a.G, T = a.T, S = a.S;
    const int W = a.K / 16;
    const int sigma = blockIdx.x / a.cps, cslot = blockIdx.x - sigma * a.cps;
    const int g0 = sigma * a.ks;
    const int gs = min(a.ks, G - g0);
    const int tile_lo = (int)((long long)T * cslot / a.cps);
    const int tile_hi = (int)((long long)T * (cslot + 1) / a.cps);

    // ---- per-chunk unit range of this warp, and the code prefetch cursor ----
    int chunk_lo = tile_lo;
    int R = min(kMaxTiles, tile_hi - chunk_lo);
    int U = R * gs;
    int u0 = U * warp / kWarps, u1 = U * (warp + 1) / kWarps;
    int ld_tile = 0, ld_g = 0;   // chunk-local cursor of the next unit to load
    Stage st[D];
    auto load_stage = [&](Stage& s) {
        const int r0 = (chunk_lo + ld_tile) * 16 + gid, r1 = r0 + 8;
        const int g = g0 + ld_g;
        const int w = g * kWordsPerGroup + 2 * t;
        if (r0 < N) {
            s.c0 = ldg_stream_u2(a.codes + (size_t)r0 * W + w);
            s.s0 = ldg_stream_u16(a.scales + (size_t)r0 * G + g);
        } else {
            s.c0 = make_uint2(0x55555555u, 0x55555555u);
            s.s0 = 0u;
        }
        if (r1 < N) {
            s.c1 = ldg_stream_u2(a.codes + (size_t)r1 * W + w);
            s.s1 = ldg_stream_u16(a.scales + (size_t)r1 * G + g);
        } else {
            s.c1 = make_uint2(0x55555555u, 0x55555555u);
            s.s1 = 0u;
        }
        if (++ld_g == gs) { ld_g = 0; ++ld_tile; }
    };
    auto start_chunk_prefetch = [&]() {
        ld_tile = u0 / gs;
        ld_g = u0 - ld_tile * gs;
#pragma unroll
        for (int s = 0; s < D; ++s)
            if (u0 + s < u1) load_stage(st[s]);
    };
    start_chunk_prefetch();

    // ---- everything below reads what the previous kernel may have written ----
    pdl_wait();

    // ---- stage this CTA's slice of the activation (warp w: group g0 + w) ----
    for (int i = threadIdx.x; i < kSliceGroups * MP; i += blockDim.x) fcs[i] = make_float2(0.0f, 0.0f);
    __syncthreads();
    if (warp < gs) {
        const int g = g0 + warp;
        const int tt = lane >> 3, j = lane & 7;
        const int jp = j < 6 ? j : j - 6;
        for (int mb = 0; mb < M; mb += 8) {
            float v[8][4];
#pragma unroll
            for (int mi = 0; mi < 8; ++mi) {
                const int m = mb + mi;
                if (m < M) {
                    const size_t off = (size_t)m * a.K + (size_t)g * kGroup + 32 * tt + j;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (XF32)
                            v[mi][u] = reinterpret_cast<const float*>(a.x)[off + 8 * u];
                        else
                            v[mi][u] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.x)[off + 8 * u]);
                    }
                }
            }
#pragma unroll
            for (int mi = 0; mi < 8; ++mi) {
                const int m = mb + mi;
                if (m < M) {
                    float mx = fmaxf(fmaxf(fabsf(v[mi][0]), fabsf(v[mi][1])), fmaxf(fabsf(v[mi][2]), fabsf(v[mi][3])));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    int E = 0;
                    if (mx > 0.0f && mx <= 3.0e38f) {
                        int ex;
                        frexpf(mx, &ex);            // mx < 2^ex
                        E = max(-100, min(5 - ex, 150));   // mx * 2^(E + 10) < 2^15
                    }
                    const float c = ldexpf(1.0f, E + 10 - 2 * jp);   // exact power of two
                    const __half2 lo = __floats2half2_rn(v[mi][0] * c, v[mi][1] * c);  // k = 32tt+j, +8
                    const __half2 hi = __floats2half2_rn(v[mi][2] * c, v[mi][3] * c);  // k = 32tt+16+j, +24
                    uint2 out;
                    out.x = *reinterpret_cast<const uint32_t*>(&lo);
                    out.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(bsm + ((size_t)warp * MP + m) * kFragWords + tt * 16 + 2 * j) = out;
                    if (lane == 0) fcs[warp * MP + m].x = ldexpf(1.0f, 14 - E);
                }
            }
        }
        __syncwarp();
        // the -1 correction: the same MMA chain on the all-ones code pattern
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
            uint32_t b[16];
            const int m = nt * 8 + gid;
            load_frag(bsm + ((size_t)warp * MP + m) * kFragWords + t * 16, m < M, b);
            float acc1[4];
            const uint32_t ones = 0x55555555u;
            unit_mmas(acc1, ones, ones, ones, ones, b);
            if (gid == 0) {
                const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
                if (m0 < M) fcs[warp * MP + m0].y = fcs[warp * MP + m0].x * acc1[0];
                if (m1 < M) fcs[warp * MP + m1].y = fcs[warp * MP + m1].x * acc1[1];
            }
        }
    }

    for (;;) {
        // ---- zero the accumulators of this chunk ----
        for (int i = threadIdx.x; i < R * 16 * MP; i += blockDim.x) accs[i] = 0.0f;
        __syncthreads();

        // ---- main loop over this warp's units ----
        int tile = u0 / max(gs, 1), gl = u0 - tile * max(gs, 1);
        float ysum[MT][4];
#pragma unroll
        for (int nt = 0; nt < MT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) ysum[nt][q] = 0.0f;
        const int n_units = u1 - u0;
        for (int base = 0; base < n_units; base += D) {
#pragma unroll
            for (int s = 0; s < D; ++s) {
                const int i = base + s;
                if (i < n_units) {
                    const Stage cur = st[s];
                    if (i + D < n_units) load_stage(st[s]);
                    float4 f[MT];
                    float acc[MT][4];
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        uint32_t b[16];
                        const int m = nt * 8 + gid;
                        load_frag(bsm + ((size_t)gl * MP + m) * kFragWords + t * 16, m < M, b);
                        f[nt] = *reinterpret_cast<const float4*>(fcs + gl * MP + nt * 8 + 2 * t);
                        unit_mmas(acc[nt], cur.c0.x, cur.c1.x, cur.c0.y, cur.c1.y, b);
                    }
                    const float sc0 = __half2float(__ushort_as_half((unsigned short)cur.s0));
                    const float sc1 = __half2float(__ushort_as_half((unsigned short)cur.s1));
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        // f = (F, F*acc1) of tokens 2t and 2t+1
                        ysum[nt][0] = fmaf(sc0, fmaf(f[nt].x, acc[nt][0], -f[nt].y), ysum[nt][0]);
                        ysum[nt][1] = fmaf(sc0, fmaf(f[nt].z, acc[nt][1], -f[nt].w), ysum[nt][1]);
                        ysum[nt][2] = fmaf(sc1, fmaf(f[nt].x, acc[nt][2], -f[nt].y), ysum[nt][2]);
                        ysum[nt][3] = fmaf(sc1, fmaf(f[nt].z, acc[nt][3], -f[nt].w), ysum[nt][3]);
                    }
                    if (gl == gs - 1 || i == n_units - 1) {
                        float* row = accs + (size_t)tile * 16 * MP;
#pragma unroll
                        for (int nt = 0; nt < MT; ++nt) {
                            const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
                            if (m0 < M) {
                                atomicAdd(row + gid * MP + m0, ysum[nt][0]);
                                atomicAdd(row + (gid + 8) * MP + m0, ysum[nt][2]);
                            }
                            if (m1 < M) {
                                atomicAdd(row + gid * MP + m1, ysum[nt][1]);
                                atomicAdd(row + (gid + 8) * MP + m1, ysum[nt][3]);
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) ysum[nt][q] = 0.0f;
                        }
                    }
                    if (++gl == gs) { gl = 0; ++tile; }
                }
            }
        }
        __syncthreads();

        // ---- write this chunk: y directly (one slice), or partials + fix-up ----
        const int nvals = R * 16 * M;
        if (S == 1) {
            for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
                const int m = i / (R * 16), rr = i - m * (R * 16);
                const int r = chunk_lo * 16 + rr;
                if (r < N) a.y[(size_t)m * N + r] = accs[(size_t)rr * MP + m];
            }
        } else {
            float* P = a.partial + ((size_t)sigma * T + chunk_lo) * 16 * M;
            for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
                const int tl = i / (16 * M), rem = i - tl * 16 * M;
                const int m = rem / 16, r = rem - m * 16;
                P[i] = accs[((size_t)tl * 16 + r) * MP + m];   // [tile][m][16]
            }
            __threadfence();
            __syncthreads();
            for (int i = threadIdx.x; i < R; i += blockDim.x)
                fin[i] = (atomicAdd(a.counter + chunk_lo + i, 1u) == (unsigned)(S - 1));
            __syncthreads();
            __threadfence();
            for (int i = threadIdx.x; i < nvals; i += blockDim.x) {
                const int tl = i / (16 * M);
                if (!fin[tl]) continue;
                const int rem = i - tl * 16 * M;
                const int m = rem / 16, r = rem - m * 16;
                const int tile_g = chunk_lo + tl;
                const size_t off = (size_t)tile_g * 16 * M + rem;
                float sum = 0.0f;
                for (int sg = 0; sg < S; ++sg) sum += __ldcg(a.partial + (size_t)sg * T * 16 * M + off);
                const int row = tile_g * 16 + r;
                if (row < N) a.y[(size_t)m * N + row] = sum;
            }
            for (int i = threadIdx.x; i < R; i += blockDim.x)
                if (fin[i]) a.counter[chunk_lo + i] = 0u;
        }

        // ---- next chunk of this CTA's tile range ----
        chunk_lo += R;
        if (chunk_lo >= tile_hi) break;
        __syncthreads();
        R = min(kMaxTiles, tile_hi - chunk_lo);
        U = R * gs;
        u0 = U * warp / kWarps;
        u1 = U * (warp + 1) / kWarps;
        start_chunk_prefetch();
    }
}

// Rotation prologue for the fused path: y_ws (fp32 [M][K]) = H_4096 (s (.) x) / 64,
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
struct Plan {
    int G, T, S, ks, cps, ctas;
    size_t off_xr, off_partial, off_counter, bytes;
};

Plan make_plan(int M, int N, int K, bool rot, int sms) {
    Plan p{};
    p.G = K / kGroup;
    p.T = (N + 15) / 16;
    p.ks = p.G < kSliceGroups ? p.G : kSliceGroups;
    p.S = (p.G + p.ks - 1) / p.ks;
    const int MT = (M + 7) / 8;
    const int cmax = sms * (MT == 1 ? GemvCfg<1>::kCtasPerSm : GemvCfg<2>::kCtasPerSm);
    p.cps = p.S >= cmax ? 1 : cmax / p.S;
    if (p.cps > p.T) p.cps = p.T;
    p.ctas = p.S * p.cps;
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

template <int MT, bool XF32>
cudaError_t launch_gemv(const GemvArgs& args, int ctas, cudaStream_t stream) {
    constexpr size_t smem = gemv_smem_bytes<MT>();
    static bool attr_set[64] = {};   // the attribute is per function and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(gemv_kernel<MT, XF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_pdl(gemv_kernel<MT, XF32>, dim3(ctas), dim3(kWarps * 32), smem, stream, true, args);
}

tern_status run(const void* x, const int8_t* signs, const uint32_t* codes, const void* scales, float* y, int M,
                int N, int K, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const Plan p = make_plan(M, N, K, signs != nullptr, sms);
    if (p.bytes > 256 || signs) {
        if (!workspace || workspace_bytes < p.bytes) return TERN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
    }
    char* ws = reinterpret_cast<char*>(workspace);
    GemvArgs args;
    args.x = x;
    args.codes = codes;
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
    args.ks = p.ks;
    args.cps = p.cps;
    int launches = 1;
    cudaError_t e;
    if (signs) {
        float* xr = reinterpret_cast<float*>(ws + p.off_xr);
        e = launch_pdl(rotate_f32_kernel, dim3(K / kFwhtN, M), dim3(kFwhtThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), signs, xr, K);
        if (e != cudaSuccess) return TERN_ERR_CUDA;
        args.x = xr;
        launches = 2;
        e = M <= 8 ? launch_gemv<1, true>(args, p.ctas, stream) : launch_gemv<2, true>(args, p.ctas, stream);
    } else {
        e = M <= 8 ? launch_gemv<1, false>(args, p.ctas, stream) : launch_gemv<2, false>(args, p.ctas, stream);
    }
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(launches);
    return TERN_OK;
}

size_t workspace_bytes(int M, int N, int K, bool rot) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return 0;
    // sized for the largest plan any supported device could pick (one slice
    // per CTA bound does not change S, only the CTA count), so a size queried
    // on one GB300 fits every other
    const Plan p = make_plan(M, N, K, rot, 1 << 20);
    return p.bytes;
}

}  // namespace
}  // namespace tern

using namespace tern;

extern "C" size_t tern_gemv_workspace_bytes(int M, int N, int K) {
    // covers both the plain and the rotation-fused call of the same shape
    return workspace_bytes(M, N, K, (K % kFwhtN) == 0);
}

extern "C" tern_status tern_gemv(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                 int N, int K, void* workspace, size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (tern::workspace_bytes(M, N, K, false) > 256 && (!workspace || workspace_bytes < tern::workspace_bytes(M, N, K, false)))
        return TERN_ERR_WORKSPACE;
    return run(x, nullptr, codes, scales, y, M, N, K, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" tern_status tern_fwht_gemm(const void* x, const int8_t* signs, const uint32_t* codes,
                                      const void* scales, float* y, int M, int N, int K, void* workspace,
                                      size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    if (K % kFwhtN != 0) return TERN_ERR_SHAPE;
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (!signs) return TERN_ERR_NULL;
    if (!aligned16(signs)) return TERN_ERR_ALIGN;
    if (!workspace || workspace_bytes < tern::workspace_bytes(M, N, K, true)) return TERN_ERR_WORKSPACE;
    return run(x, signs, codes, scales, y, M, N, K, workspace, workspace_bytes, (cudaStream_t)stream);
}
