// tern_fwht.cuh -- 4096-point Walsh-Hadamard transform of one block in shared
// memory by one 256-thread CTA (internal).
//
// The rotation is the normalized Sylvester-Walsh-Hadamard transform of block
// 4096 along the activation's last dimension with an explicit +-1 sign pattern
// ("Ternary-Bonsai-2-9B-2bit" article, section 3): x' = H_4096 (s (.) x) / 64,
// H[i][j] = (-1)^popcount(i & j) (natural order).
//
// Because H_4096 = H_16 (x) H_16 (x) H_16 in natural order, the transform is
// three passes of 16-point transforms, one per 4-bit digit of the index.  Each
// thread owns 16 elements per pass (registers); the passes exchange through a
// padded fp32 shared buffer (one pad word per 16 keeps every pass's accesses
// on distinct banks).
#pragma once

#include "tern_common.cuh"

namespace tern {

constexpr int kFwhtN = 4096;
constexpr int kFwhtThreads = 256;
constexpr int kFwhtSmemFloats = kFwhtN + kFwhtN / 16;

__device__ __forceinline__ int fwht_pos(int idx) { return idx + (idx >> 4); }

// In-register 16-point transform, natural order.
__device__ __forceinline__ void fwht16(float (&v)[16]) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                const float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
        }
    }
}

// Rotates one 4096 block: x (bf16, 16-byte aligned), signs (int8, 16-byte
// aligned), result (scaled by 1/64) left in `sm` at fwht_pos(idx).  Must be
// called by all 256 threads; ends with a __syncthreads().
__device__ __forceinline__ void fwht4096_block(const __nv_bfloat16* __restrict__ x,
                                               const int8_t* __restrict__ signs,
                                               float* __restrict__ sm) {
    const int i = threadIdx.x;
    float v[16];
    // pass 1: index digit 0 (bits 0..3); thread i owns [16 i, 16 i + 16)
    {
        const int4* xp = reinterpret_cast<const int4*>(x + 16 * i);
        const int4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
        const int4 sg = __ldg(reinterpret_cast<const int4*>(signs + 16 * i));
        const uint32_t xw[8] = {(uint32_t)x0.x, (uint32_t)x0.y, (uint32_t)x0.z, (uint32_t)x0.w,
                                (uint32_t)x1.x, (uint32_t)x1.y, (uint32_t)x1.z, (uint32_t)x1.w};
        const uint32_t sw[4] = {(uint32_t)sg.x, (uint32_t)sg.y, (uint32_t)sg.z, (uint32_t)sg.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t bits = (xw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
            const float xv = __uint_as_float(bits << 16);
            const int s = (int)(int8_t)((sw[e >> 2] >> (8 * (e & 3))) & 0xFFu);
            v[e] = s < 0 ? -xv : xv;
        }
        fwht16(v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sm[fwht_pos(16 * i + e)] = v[e];
    }
    __syncthreads();
    // pass 2: digit 1 (bits 4..7)
    {
        const int base = (i & 15) | ((i >> 4) << 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = sm[fwht_pos(base | (e << 4))];
        fwht16(v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sm[fwht_pos(base | (e << 4))] = v[e];
    }
    __syncthreads();
    // pass 3: digit 2 (bits 8..11), then the 1/sqrt(4096) normalization
    {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = sm[fwht_pos(i | (e << 8))];
        fwht16(v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sm[fwht_pos(i | (e << 8))] = v[e] * (1.0f / 64.0f);
    }
    __syncthreads();
}

// The 4-point transform in natural order, in registers.
__device__ __forceinline__ void fwht4(float (&v)[4]) {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
}

constexpr int kFwhtSliceN = 1024;                                   // a quarter of a block
constexpr int kFwhtSliceSmemFloats = kFwhtSliceN + kFwhtSliceN / 8;

// Where value j of a slice sits in its shared buffer: a pad of four floats
// per 32 keeps each phase below on distinct banks, and a reader of 32
// consecutive values (one lane quarter of a group) gets them 16-byte aligned.
__device__ __forceinline__ int fwht_slice_pos(int j) { return j + 4 * (j >> 5); }

// Slice a (0..3) of one 4096 block of H_4096 (s (.) x) / 64, with H_4096 =
// H_4 (x) H_1024 in natural order: the slice is H_1024 u / 64, u[j] =
// sum_{a'} (-1)^popcount(a & a') z[1024 a' + j], z = s (.) x over the block.
// Thread i sums u for j = 4 i .. 4 i + 3 (a sign is a flip of the bf16 sign
// bit: its sign byte's bit 7, and row a of H_4 for the whole part), then
// H_1024 = H_8 (x) H_128 runs as the index's bits 0-1 in registers, bits 2-6
// across the lanes of the warp that holds those 128 values (j = 128 w + ...),
// and bits 7-9 across the warps through shared memory: two barriers.  x and
// signs point at the block (8- and 4-byte aligned); the result is left in
// `sm` at fwht_slice_pos(j).  Must be called by all 256 threads; ends with a
// __syncthreads().
__device__ __forceinline__ void fwht1024_slice(const __nv_bfloat16* __restrict__ x,
                                               const int8_t* __restrict__ signs, int a,
                                               float* __restrict__ sm) {
    const int i = threadIdx.x, lane = i & 31;
    float u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ap = 0; ap < 4; ++ap) {
        const int k0 = kFwhtSliceN * ap + 4 * i;
        const uint2 xw = *reinterpret_cast<const uint2*>(x + k0);
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(signs + k0);
        const uint32_t neg = (__popc(a & ap) & 1) ? 0x80008000u : 0u;
        // sign bytes 0 and 1 (2 and 3) to bytes 1 and 3: their bit 7 onto
        // the sign bits of the two bf16 values of a word
        const uint32_t lo = xw.x ^ ((__byte_perm(sw, 0u, 0x1404u) & 0x80008000u) ^ neg);
        const uint32_t hi = xw.y ^ ((__byte_perm(sw, 0u, 0x3424u) & 0x80008000u) ^ neg);
        u[0] += __uint_as_float(lo << 16);
        u[1] += __uint_as_float(lo & 0xFFFF0000u);
        u[2] += __uint_as_float(hi << 16);
        u[3] += __uint_as_float(hi & 0xFFFF0000u);
    }
    fwht4(u);   // index bits 0-1
#pragma unroll
    for (int b = 0; b < 5; ++b) {   // index bits 2-6: lane bit b
        const float sg = ((lane >> b) & 1) ? -1.0f : 1.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = fmaf(u[e], sg, __shfl_xor_sync(0xffffffffu, u[e], 1 << b));
    }
    *reinterpret_cast<float4*>(sm + fwht_slice_pos(4 * i)) = make_float4(u[0], u[1], u[2], u[3]);
    __syncthreads();
    if (i < 128) {   // index bits 7-9: thread i takes value i of each of the eight 128-wide parts
        float v[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) v[g] = sm[fwht_slice_pos(128 * g + i)];
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if ((g & h) == 0) {
                    const float p = v[g], q = v[g + h];
                    v[g] = p + q;
                    v[g + h] = p - q;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) sm[fwht_slice_pos(128 * g + i)] = v[g] * (1.0f / 64.0f);
    }
    __syncthreads();
}

}  // namespace tern
