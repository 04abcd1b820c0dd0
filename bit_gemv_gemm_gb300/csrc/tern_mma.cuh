// tern_mma.cuh -- device helpers shared by the decode products: the f16
// `mma.sync` of the exact-adder unpack, the activation staging's exponents,
// asynchronous copies and the range-flag count.  Internal.
#pragma once

#include "tern_common.cuh"

namespace tern {

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

// Activation staging: a token's 128 values of one group become fp16
// x 2^(E + 10 - 2j'), j' the code's position within its 16-bit half (j for
// slots 0-5, j - 6 for 6 and 7, which are read after a shift by 12; with Q3,
// all four codes valid: j for 0-4, j - 5 for 5-7 after a shift by 10), with E
// such that the largest |x| times 2^(E + 10) stays below 2^15.
__device__ __forceinline__ int stage_exponent(float mx) {
    // mx < 2^ex for ex = biased exponent - 126
    const int be = (int)(__float_as_uint(mx) >> 23);   // mx >= 0
    return (mx > 0.0f && be < 255) ? max(-100, min(5 - (max(be, 1) - 126), 110)) : 0;
}
// the exact power of two 2^(E + 10 - 2j') for slot j, exponent within [-100, 120]
template <bool Q3 = false>
__device__ __forceinline__ float stage_multiplier(int E, int j) {
    constexpr int kSplit = Q3 ? 5 : 6;
    return __uint_as_float((uint32_t)(E + 10 - 2 * (j < kSplit ? j : j - kSplit) + 127) << 23);
}

// Slot j's A registers from the four code words by one AND (codes 6, 7, 14, 15
// after a shift by 12; with Q3, codes 5-7 and 13-15 after a shift by 10).
template <bool Q3>
__device__ __forceinline__ void slot_regs(int j, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                          uint32_t (&r)[4]) {
    constexpr int kSplit = Q3 ? 5 : 6, kShift = 2 * kSplit;
    if (j < kSplit) {
        const uint32_t mk = 0x00030003u << (2 * j);
        r[0] = w0 & mk;
        r[1] = w1 & mk;
        r[2] = w2 & mk;
        r[3] = w3 & mk;
    } else {
        const uint32_t mk = 0x00030003u << (2 * (j - kSplit));
        r[0] = (w0 >> kShift) & mk;
        r[1] = (w1 >> kShift) & mk;
        r[2] = (w2 >> kShift) & mk;
        r[3] = (w3 >> kShift) & mk;
    }
}

// One unit's chain (16 rows x 128 weights, one token tile): slot j's MMA after
// slot j - 1's in one accumulator.
__device__ __forceinline__ void unit_chain(float (&acc)[4], const uint32_t (&w)[4], const uint32_t (&b)[16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[4];
        slot_regs<false>(j, w[0], w[1], w[2], w[3], r);
        mma16816(acc, r[0], r[1], r[2], r[3], b[2 * j], b[2 * j + 1], j > 0);
    }
}

// ---- asynchronous copies (cp.async) ----
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- the per-range flag word ----
constexpr uint64_t kFlagWaitNs = 1000000000ull;   // 1 s: far beyond any real wait
// Counts into a range flag modulo `wrap + 1` without waiting for the old value.
__device__ __forceinline__ void red_inc(unsigned* p, unsigned wrap) {
    asm volatile("red.relaxed.gpu.global.inc.u32 [%0], %1;" ::"l"(p), "r"(wrap) : "memory");
}

}  // namespace tern
