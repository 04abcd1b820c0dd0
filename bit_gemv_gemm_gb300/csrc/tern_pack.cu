// tern_pack.cu -- device packers: int8 trits -> 2-bit codes, 16 per uint32,
// and int8 +-1 -> bits, 32 per uint32 (the 1-bit sibling format).
//
// Code q = t + 1 in a 2-bit slot ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model
// card, "Memory requirement"); slot k%16 of word k/16, lowest k in the lowest
// bits.  An input outside {-1, 0, +1} becomes the invalid code 3 and is counted.
#include "tern_common.cuh"

namespace tern {
namespace {

constexpr int kPackThreads = 256;

// One thread per output word: a 16-byte load of 16 trits, a 4-byte store.
__global__ void __launch_bounds__(kPackThreads)
pack_kernel(const int4* __restrict__ t, uint32_t* __restrict__ codes, long long words,
            int* __restrict__ bad_count) {
    int bad = 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < words; w += stride) {
        const int4 v = __ldg(t + w);
        const uint32_t in[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t byte = (in[j] >> (8 * b)) & 0xFFu;
                // 0xFF (-1) -> 0, 0 -> 1, 1 -> 2: (byte + 1) & 0xFF for the valid three
                const uint32_t plus1 = (byte + 1u) & 0xFFu;
                const bool ok = plus1 <= 2u;
                bad += ok ? 0 : 1;
                word |= (ok ? plus1 : 3u) << (2 * (4 * j + b));
            }
        }
        codes[w] = word;
    }
    if (bad_count) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(bad_count, bad);
    }
}

// The 1-bit sibling: one thread per output word, two 16-byte loads of 32
// values, bit i of the word set for value i = +1.  Anything but +-1 is
// counted and stored as -1.
__global__ void __launch_bounds__(kPackThreads)
bin_pack_kernel(const int4* __restrict__ t, uint32_t* __restrict__ words_out, long long words,
                int* __restrict__ bad_count) {
    int bad = 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < words; w += stride) {
        const int4 v0 = __ldg(t + 2 * w), v1 = __ldg(t + 2 * w + 1);
        const uint32_t in[8] = {(uint32_t)v0.x, (uint32_t)v0.y, (uint32_t)v0.z, (uint32_t)v0.w,
                                (uint32_t)v1.x, (uint32_t)v1.y, (uint32_t)v1.z, (uint32_t)v1.w};
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t byte = (in[j] >> (8 * b)) & 0xFFu;
                bad += (byte == 1u || byte == 0xFFu) ? 0 : 1;
                word |= (byte == 1u ? 1u : 0u) << (4 * j + b);
            }
        }
        words_out[w] = word;
    }
    if (bad_count) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(bad_count, bad);
    }
}

// The group-size-64 pack's scales: group g of a row is the pair (2g, 2g + 1),
// which the pack repeats; one thread per output scale keeps the first and
// counts pairs that differ bit for bit.
__global__ void __launch_bounds__(kPackThreads)
scales_g64_kernel(const unsigned short* __restrict__ s64, unsigned short* __restrict__ s128, long long groups,
                  int* __restrict__ mismatch) {
    int bad = 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < groups; i += stride) {
        const unsigned int pair = reinterpret_cast<const unsigned int*>(s64)[i];   // (s[2g], s[2g+1])
        const unsigned short lo = (unsigned short)(pair & 0xFFFFu), hi = (unsigned short)(pair >> 16);
        bad += lo != hi;
        s128[i] = lo;
    }
    if (mismatch) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatch, bad);
    }
}

}  // namespace
}  // namespace tern

using namespace tern;

extern "C" tern_status tern_scales_from_g64(const void* s64, int N, int K, void* s128, int* mismatch,
                                            tern_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || K < 0 || K % 128 != 0) return TERN_ERR_SHAPE;
    const long long groups = (long long)N * (K / 128);
    if (groups == 0) return TERN_OK;
    if (!s64 || !s128) return TERN_ERR_NULL;
    if (!aligned16(s64) || !aligned16(s128)) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    long long blocks = (groups + kPackThreads - 1) / kPackThreads;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    scales_g64_kernel<<<(unsigned)blocks, kPackThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const unsigned short*>(s64), reinterpret_cast<unsigned short*>(s128), groups, mismatch);
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}

extern "C" tern_status tern_bin_pack(const int8_t* t, int N, int K, uint32_t* words, int* bad_count,
                                     tern_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || K < 0 || K % 32 != 0) return TERN_ERR_SHAPE;
    const long long nwords = (long long)N * (K / 32);
    if (nwords == 0) return TERN_OK;
    if (!t || !words) return TERN_ERR_NULL;
    if (!aligned16(t) || !aligned16(words)) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    long long blocks = (nwords + kPackThreads - 1) / kPackThreads;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    bin_pack_kernel<<<(unsigned)blocks, kPackThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const int4*>(t), words, nwords, bad_count);
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}

extern "C" tern_status tern_pack(const int8_t* t, int N, int K, uint32_t* codes, int* bad_count,
                                 tern_stream_t stream) {
    set_launch_count(0);
    if (N < 0 || K < 0 || K % 16 != 0) return TERN_ERR_SHAPE;
    const long long words = (long long)N * (K / 16);
    if (words == 0) return TERN_OK;
    if (!t || !codes) return TERN_ERR_NULL;
    if (!aligned16(t) || !aligned16(codes)) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    long long blocks = (words + kPackThreads - 1) / kPackThreads;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    pack_kernel<<<(unsigned)blocks, kPackThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const int4*>(t), codes, words, bad_count);
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}
