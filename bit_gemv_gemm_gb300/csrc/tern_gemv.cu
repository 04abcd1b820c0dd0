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
// and a contiguous range of 16-row tiles, and warp w of the CTA owns group w of
// the slice for the whole range: it stages that group's activation once, into
// registers, and streams its own 32-byte column of every tile (16 rows x 32 B =
// one 16-byte cp.async per lane) through a private shared-memory ring, kDepth
// tiles ahead; the first kDepth go out before the programmatic-dependent-launch
// wait.  Two tiles per step run as two independent MMA chains.  Row partial
// sums go to shared memory (private per warp for M <= 4, shared atomics
// beyond).  With one slice the CTA writes y; with several, each CTA stores its
// partial tile sums to the workspace and the last CTA to finish a tile (an
// arrival counter) adds the slices in slice order and writes y.  y is written
// exactly once per element: no pre-zeroing, no global float atomics.
#include "tern_fwht.cuh"

namespace tern {
namespace {

constexpr int kGroup = 128;            // weights per scale
constexpr int kSliceGroups = 8;        // groups per K-slice = warps per CTA
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 12;             // tiles in flight per warp (even)
constexpr int kEarly = 4;              // of which issued before the activation is staged
constexpr int kSlotBytes = 16 * 32;    // one warp's share of a tile: 16 rows x 32 B
constexpr int kMaxTiles = 32;          // tiles per CTA (bounds the shared partials and scales)
constexpr int kPrivateMaxM = 4;        // private per-warp partials up to this many tokens
constexpr size_t kSmemPerSm = 228 * 1024;   // shared memory of one SM
constexpr size_t kCtaSmemReserve = 1024;    // taken by the system from each resident CTA

template <int MT> struct GemvCfg;
template <> struct GemvCfg<1> { static constexpr int kCtasPerSm = 3; };
template <> struct GemvCfg<2> { static constexpr int kCtasPerSm = 2; };

struct GemvArgs {
    const void* x;              // bf16 [M][K], or fp32 [M][K] when the rotation prologue ran
    const uint32_t* codes;      // [N][K/16]
    const __half* scales;       // [N][K/128]
    float* y;                   // [M][N]
    float* partial;             // [S][T][M][16]
    unsigned* counter;          // [T]
    int M, N, K, G, T, S, cps, rmax;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// dynamic shared memory: [code rings | scales [row][8] | row partials | finalize flags]
__host__ __device__ inline size_t smem_sc() { return (size_t)kWarps * kDepth * kSlotBytes; }
__host__ __device__ inline size_t smem_part(int rmax) {
    return smem_sc() + align_up((size_t)kWarps * rmax * 16 * 2, 16);
}
// private: [8 warps][rmax][16][M]; shared: [rmax][16][MP]
__host__ __device__ inline size_t part_floats(int rmax, int M, int MP) {
    return M <= kPrivateMaxM ? (size_t)kWarps * rmax * 16 * M : (size_t)rmax * 16 * MP;
}
__host__ __device__ inline size_t smem_fin(int rmax, int M, int MP) {
    return smem_part(rmax) + part_floats(rmax, M, MP) * 4;
}
__host__ __device__ inline size_t smem_total(int rmax, int M, int MP) { return smem_fin(rmax, M, MP) + (size_t)rmax * 4; }

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

// The chain of one (16-row, 128-weight) unit for one token tile.
__device__ __forceinline__ void mma_chain1(float (&acc)[4], const uint32_t (&w)[4], const uint32_t (&b)[16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[4];
        slot_regs(j, w[0], w[1], w[2], w[3], r);
        mma16816(acc, r[0], r[1], r[2], r[3], b[2 * j], b[2 * j + 1], j > 0);
    }
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

// ---- per-warp asynchronous copies (cp.async, 16 bytes per lane) ----
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int MT, bool XF32>
__global__ void __launch_bounds__(kThreads, GemvCfg<MT>::kCtasPerSm)
gemv_kernel(const GemvArgs a) {
    constexpr int MP = 8 * MT;
    extern __shared__ __align__(16) unsigned char smem[];
    const int rmax = a.rmax;
    const int M = a.M;
    unsigned short* scs = reinterpret_cast<unsigned short*>(smem + smem_sc());   // [rmax * 16][8]
    float* part = reinterpret_cast<float*>(smem + smem_part(rmax));
    int* fin = reinterpret_cast<int*>(smem + smem_fin(rmax, M, MP));           // [rmax]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int N = a.N, G = a.G, T = a.T, S = a.S;
    const int W = a.K / 16;
    const int sigma = blockIdx.x / a.cps, cslot = blockIdx.x - sigma * a.cps;
    const int g0 = sigma * kSliceGroups;
    const int gs = min(kSliceGroups, G - g0);
    const int tile_lo = (int)((long long)T * cslot / a.cps);
    const int tile_hi = (int)((long long)T * (cslot + 1) / a.cps);
    const int R = tile_hi - tile_lo;
    const bool active = warp < gs;
    const int g = g0 + (active ? warp : 0);

    // this warp's ring; lane l copies row l/2, 16-byte half l%2 of its group's 32 bytes
    unsigned char* ring = smem + (size_t)warp * kDepth * kSlotBytes;
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const int crow0 = tile_lo * 16 + (lane >> 1);
    const uint32_t* csrc = a.codes + (size_t)crow0 * W + g * 8 + (lane & 1) * 4;
    const size_t cstep = (size_t)16 * W;   // words per tile
    // tile i into ring slot `slot` (= i mod kDepth)
    auto issue = [&](int i, int slot) {
        if (active && i < R) {
            const bool ok = crow0 + 16 * i < N;
            cp_async16(ring_s + (uint32_t)(slot * kSlotBytes + lane * 16), ok ? csrc + (size_t)i * cstep : a.codes,
                       ok);
        }
        cp_async_commit();   // one group per tile, empty past the end, so the waits count uniformly
    };

    pdl_launch_dependents();
    // codes and scales are never the previous kernel's output: start streaming
    // both before the PDL wait.  The scales of the whole range come first, as
    // one commit group: a row's 8 slice scales are one 16-byte chunk when G is
    // a multiple of 8 (one copy per row), else they are gathered one by one.
    if (G % kSliceGroups == 0) {
        const uint32_t scs_s = static_cast<uint32_t>(__cvta_generic_to_shared(scs));
        for (int i = threadIdx.x; i < R * 16; i += kThreads) {
            const int row = tile_lo * 16 + i;
            const bool ok = row < N;
            cp_async16(scs_s + (uint32_t)i * 16u, a.scales + (size_t)(ok ? row : 0) * G + g0, ok);
        }
    } else {
        for (int i = threadIdx.x; i < R * 16 * kSliceGroups; i += kThreads) {
            const int row = tile_lo * 16 + (i >> 3), gg = i & 7;
            scs[i] = (row < N && gg < gs) ? __half_as_ushort(a.scales[(size_t)row * G + g0 + gg])
                                          : (unsigned short)0;
        }
    }
    cp_async_commit();
#pragma unroll
    for (int i = 0; i < kEarly; ++i) issue(i, i);
    pdl_wait();
    if (M > kPrivateMaxM)   // shared partials take atomics; private ones are written once each
        for (int i = threadIdx.x; i < (int)part_floats(rmax, M, MP); i += kThreads) part[i] = 0.0f;

    // stage this warp's group: lane (gid, t) holds token nt*8+gid, k = 32t .. 32t+31
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
        // E with mx * 2^(E + 10) < 2^15: mx < 2^ex for ex = biased exponent - 126
        const int be = (int)(__float_as_uint(mx) >> 23);   // mx >= 0
        int E = 0;
        if (mx > 0.0f && be < 255) E = max(-100, min(5 - (max(be, 1) - 126), 110));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // exact power of two 2^(E + 10 - 2j'), exponent within [-100, 120]
            const float c = __uint_as_float((uint32_t)(E + 10 - 2 * (j < 6 ? j : j - 6) + 127) << 23);
            const __half2 lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);       // k = 32t+j, +8
            const __half2 hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c); // k = 32t+16+j, +24
            b[nt][2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
            b[nt][2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
        }
        // the -1 correction: the same chain on the all-ones pattern; every row of
        // the result is the same, lane (gid, t) holds tokens 2t, 2t+1
        float acc1[4];
        const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
        mma_chain1(acc1, ones, b[nt]);
        const float F = (m < M) ? __uint_as_float((uint32_t)(14 - E + 127) << 23) : 0.0f;   // 2^(14-E)
        const float F0 = __shfl_sync(0xffffffffu, F, (2 * t) * 4);
        const float F1 = __shfl_sync(0xffffffffu, F, (2 * t + 1) * 4);
        f[nt] = make_float4(F0, F0 * acc1[0], F1, F1 * acc1[1]);
    }
#pragma unroll
    for (int i = kEarly; i < kDepth; ++i) issue(i, i);
    // this thread's scale copies (the oldest group) have landed; after the
    // barrier every thread's have, and the zeroed partials are visible
    cp_async_wait<kDepth>();
    __syncthreads();

    const unsigned short* sc_w = scs + warp;   // row r of the range: sc_w[8 r]
    auto epilogue = [&](int i, const float (&acc)[MT][4]) {
        const float s0 = __half2float(__ushort_as_half(sc_w[(i * 16 + gid) * 8]));
        const float s1 = __half2float(__ushort_as_half(sc_w[(i * 16 + gid + 8) * 8]));
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
            const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
            const float v0 = s0 * fmaf(f[nt].x, acc[nt][0], -f[nt].y);   // row gid,     token m0
            const float v1 = s0 * fmaf(f[nt].z, acc[nt][1], -f[nt].w);   // row gid,     token m1
            const float v2 = s1 * fmaf(f[nt].x, acc[nt][2], -f[nt].y);   // row gid + 8, token m0
            const float v3 = s1 * fmaf(f[nt].z, acc[nt][3], -f[nt].w);   // row gid + 8, token m1
            if (M <= kPrivateMaxM) {
                // [warp][tile][row][M]: each element written once, by its warp
                float* pw = part + (((size_t)warp * rmax + i) * 16) * M;
                if (m0 < M) {
                    pw[gid * M + m0] = v0;
                    pw[(gid + 8) * M + m0] = v2;
                }
                if (m1 < M) {
                    pw[gid * M + m1] = v1;
                    pw[(gid + 8) * M + m1] = v3;
                }
            } else {
                float* row = part + (size_t)i * 16 * MP;   // [tile][row][MP], shared by the warps
                if (m0 < M) {
                    atomicAdd(row + gid * MP + m0, v0);
                    atomicAdd(row + (gid + 8) * MP + m0, v2);
                }
                if (m1 < M) {
                    atomicAdd(row + gid * MP + m1, v1);
                    atomicAdd(row + (gid + 8) * MP + m1, v3);
                }
            }
        }
    };

    if (active) {
        int slot = 0;   // ring slot of tile i (kDepth is even: tile i + 1 sits in slot + 1)
        for (int i = 0; i < R; i += 2) {
            const bool two = i + 1 < R;
            // tiles i and i + 1 have landed (at most kDepth - 2 newer groups pending)
            cp_async_wait<kDepth - 2>();
            __syncwarp();
            uint32_t w[2][4];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const unsigned char* sp = ring + (slot + q) * kSlotBytes;
                const uint2 v0 = *reinterpret_cast<const uint2*>(sp + gid * 32 + 8 * t);
                const uint2 v1 = *reinterpret_cast<const uint2*>(sp + (gid + 8) * 32 + 8 * t);
                w[q][0] = v0.x;   // row gid,     word 2t      (MMA rows 0-7,  k-slots 2t, 2t+1)
                w[q][1] = v1.x;   // row gid + 8, word 2t      (MMA rows 8-15)
                w[q][2] = v0.y;   // row gid,     word 2t + 1  (k-slots 2t+8, 2t+9)
                w[q][3] = v1.y;   // row gid + 8, word 2t + 1
            }
            float acc[2][MT][4];
            pair_mmas<MT>(acc, w, b);
            // both slots fully read by every lane: refill them kDepth tiles ahead
            __syncwarp();
            issue(i + kDepth, slot);
            issue(i + 1 + kDepth, slot + 1);
            epilogue(i, acc[0]);
            if (two) epilogue(i + 1, acc[1]);
            slot = slot + 2 == kDepth ? 0 : slot + 2;
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- reduce the warps' partials into rows ----
    const int nvals = R * 16 * M;
    auto row_value = [&](int tl, int r, int m) -> float {
        if (M <= kPrivateMaxM) {
            float s = 0.0f;
            for (int w2 = 0; w2 < gs; ++w2) s += part[(((size_t)w2 * rmax + tl) * 16 + r) * M + m];
            return s;
        }
        return part[((size_t)tl * 16 + r) * MP + m];
    };
    if (S == 1) {
        for (int i = threadIdx.x; i < nvals; i += kThreads) {
            const int m = i / (R * 16), rr = i - m * (R * 16);
            const int r = tile_lo * 16 + rr;
            if (r < N) a.y[(size_t)m * N + r] = row_value(rr >> 4, rr & 15, m);
        }
        return;
    }
    float* P = a.partial + ((size_t)sigma * T + tile_lo) * 16 * M;
    for (int i = threadIdx.x; i < nvals; i += kThreads) {
        const int tl = i / (16 * M), rem = i - tl * 16 * M;
        const int m = rem / 16, r = rem - m * 16;
        P[i] = row_value(tl, r, m);   // [tile][m][16]
    }
    __threadfence();
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += kThreads)
        fin[i] = (atomicAdd(a.counter + tile_lo + i, 1u) == (unsigned)(S - 1));
    __syncthreads();
    __threadfence();
    for (int i = threadIdx.x; i < nvals; i += kThreads) {
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
    for (int i = threadIdx.x; i < R; i += kThreads)
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
struct Plan {
    int G, T, S, cps, ctas, rmax, MT;
    size_t smem;
    size_t off_xr, off_partial, off_counter, bytes;
};

Plan make_plan(int M, int N, int K, bool rot, int sms) {
    Plan p{};
    p.G = K / kGroup;
    p.T = (N + 15) / 16;
    p.S = (p.G + kSliceGroups - 1) / kSliceGroups;
    p.MT = (M + 7) / 8;
    // one wave: as many CTAs as fit on every SM at once, by registers (the
    // launch bound) and by shared memory (which grows with the range length)
    const int need = (p.T + kMaxTiles - 1) / kMaxTiles;   // ranges short enough for the shared partials
    for (int per_sm = p.MT == 1 ? GemvCfg<1>::kCtasPerSm : GemvCfg<2>::kCtasPerSm; per_sm >= 1; --per_sm) {
        const int cmax = sms * per_sm;
        p.cps = p.S >= cmax ? 1 : cmax / p.S;
        if (p.cps > p.T) p.cps = p.T;
        if (p.cps < need) p.cps = need;
        p.rmax = (p.T + p.cps - 1) / p.cps;
        p.smem = smem_total(p.rmax, M, 8 * p.MT);
        if ((size_t)per_sm * (p.smem + kCtaSmemReserve) <= kSmemPerSm) break;
    }
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

size_t workspace_bytes(int M, int N, int K, bool rot) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return 0;
    // partials and counters depend on (S, T) only, never on the device
    return make_plan(M, N, K, rot, 1 << 20).bytes;
}

template <int MT, bool XF32>
cudaError_t launch_gemv(const GemvArgs& args, const Plan& p, cudaStream_t stream) {
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
    return launch_pdl(gemv_kernel<MT, XF32>, dim3(p.ctas), dim3(kThreads), p.smem, stream, true, args);
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
    args.cps = p.cps;
    args.rmax = p.rmax;
    int launches = 1;
    cudaError_t e;
    if (signs) {
        float* xr = reinterpret_cast<float*>(ws + p.off_xr);
        e = launch_pdl(rotate_f32_kernel, dim3(K / kFwhtN, M), dim3(kFwhtThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), signs, xr, K);
        if (e != cudaSuccess) return TERN_ERR_CUDA;
        args.x = xr;
        launches = 2;
        e = p.MT == 1 ? launch_gemv<1, true>(args, p, stream) : launch_gemv<2, true>(args, p, stream);
    } else {
        e = p.MT == 1 ? launch_gemv<1, false>(args, p, stream) : launch_gemv<2, false>(args, p, stream);
    }
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(launches);
    return TERN_OK;
}

}  // namespace

// The decode product's kernels wait on nothing outside their own CTA, so they
// never raise a device error word; the reader reports a clean state.
cudaError_t read_gemv_device_error(int* code) {
    *code = 0;
    return cudaSuccess;
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

// ---------------------------------------------------------------------------
// Decode product with no allocation anywhere.
//
// Some callers cannot allocate device memory for a workspace: code that runs
// where an allocation may not happen (inside a custom allocator's own callback,
// a caching allocator that must not recurse, an embedded runtime that owns all
// device memory up front).  For them the product's scratch -- the per-slice
// partial row sums and the per-tile arrival counters -- lives in one fixed
// array in the library's own device memory.  Every GPU that loads the library
// holds this array (TERN_NOALLOC_SCRATCH_BYTES) until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace tern {
namespace {

constexpr size_t kNoAllocScratchBytes = TERN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};   // device address of the array, per device

// The device address of the array on the current device.  In host code the
// array's name is only a stand-in for the symbol, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace tern

extern "C" tern_status tern_gemv_noalloc(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                         int N, int K, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (tern::workspace_bytes(M, N, K, false) > kNoAllocScratchBytes) return TERN_ERR_WORKSPACE;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return TERN_ERR_CUDA;
    // the array keeps the previous call's contents: the arrival counters must
    // start at zero, so clear them on the stream first (no allocation involved)
    const Plan p = make_plan(M, N, K, false, sms);
    if (p.S > 1 &&
        cudaMemsetAsync(static_cast<char*>(scratch) + p.off_counter, 0, (size_t)p.T * 4, (cudaStream_t)stream) !=
            cudaSuccess)
        return TERN_ERR_CUDA;
    return run(x, nullptr, codes, scales, y, M, N, K, scratch, kNoAllocScratchBytes, (cudaStream_t)stream);
}
