// tern_fwht.cu -- standalone rotation: y = H_4096 (s (.) x) / 64 per block,
// bf16 in, fp32 in shared memory, bf16 out (round to nearest even).
// ("Ternary-Bonsai-2-9B-2bit" article, section 3: normalized
// Sylvester-Walsh-Hadamard, block 4096, last dimension, explicit signs.)
#include "tern_fwht.cuh"

namespace tern {
namespace {

// One CTA per (4096-block, row).  Bandwidth: 8 KB read + 8 KB written per
// block, 4 KB of signs from L2; 12 * 4096 add/sub.
__global__ void __launch_bounds__(kFwhtThreads)
fwht_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs,
            __nv_bfloat16* __restrict__ y, int K) {
    __shared__ float sm[kFwhtSmemFloats];
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x, m = blockIdx.y;
    const size_t off = (size_t)m * K + (size_t)b * kFwhtN;
    fwht4096_block(x + off, signs + (size_t)b * kFwhtN, sm);
    // thread i writes pairs (2i, 2i+1) + 512 e: 4-byte stores, fully coalesced
    const int i = threadIdx.x;
    __nv_bfloat162* yo = reinterpret_cast<__nv_bfloat162*>(y + off);
#pragma unroll
    for (int e = 0; e < kFwhtN / 512; ++e) {
        const int idx = 2 * i + 512 * e;
        yo[idx >> 1] = __floats2bfloat162_rn(sm[fwht_pos(idx)], sm[fwht_pos(idx + 1)]);
    }
}

// One CTA per (1024-wide slice, row): four times the CTAs of fwht_kernel and
// a quarter of its serial work per thread, for calls too small to fill the
// GPU with blocks (each slice reads its whole block: 4x the input reads).
__global__ void __launch_bounds__(kFwhtThreads)
fwht_slice_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs,
                  __nv_bfloat16* __restrict__ y, int K) {
    __shared__ __align__(16) float sm[kFwhtSliceSmemFloats];
    pdl_launch_dependents();
    pdl_wait();
    const int sigma = blockIdx.x, m = blockIdx.y, b = sigma >> 2;
    const size_t off = (size_t)m * K + (size_t)b * kFwhtN;
    fwht1024_slice(x + off, signs + (size_t)b * kFwhtN, sigma & 3, sm);
    // thread i writes values 4 i .. 4 i + 3 of the slice: 8-byte stores, coalesced
    const int i = threadIdx.x;
    const float4 q = *reinterpret_cast<const float4*>(sm + fwht_slice_pos(4 * i));
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(q.x, q.y);
    const __nv_bfloat162 p1 = __floats2bfloat162_rn(q.z, q.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&p0);
    o.y = *reinterpret_cast<const uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(y + off + (size_t)kFwhtSliceN * (sigma & 3) + 4 * i) = o;
}

}  // namespace
}  // namespace tern

using namespace tern;

extern "C" tern_status tern_fwht(const void* x, const int8_t* signs, void* y, int M, int K,
                                 tern_stream_t stream) {
    set_launch_count(0);
    if (M < 1 || K < kFwhtN || K % kFwhtN != 0 || M > 65535) return TERN_ERR_SHAPE;
    if (!x || !signs || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(signs) || !aligned16(y)) return TERN_ERR_ALIGN;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    // fewer blocks than SMs: one CTA per 1024-wide slice instead (latency-bound sizes)
    const bool slices = (long long)(K / kFwhtN) * M < sms;
    const dim3 grid(slices ? K / kFwhtSliceN : K / kFwhtN, M);
    cudaError_t e = launch_pdl(slices ? fwht_slice_kernel : fwht_kernel, grid, dim3(kFwhtThreads), 0,
                               (cudaStream_t)stream, true, reinterpret_cast<const __nv_bfloat16*>(x), signs,
                               reinterpret_cast<__nv_bfloat16*>(y), K);
    if (e != cudaSuccess) return TERN_ERR_CUDA;
    set_launch_count(1);
    return TERN_OK;
}
