// tern_common.cuh -- shared device/host helpers of libtern (internal).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/tern.h"

namespace tern {

// ----------------------------------------------------------------------------
// Device-side error word (sticky; read and cleared by tern_device_error()).
// ----------------------------------------------------------------------------
enum DeviceError : int {
    kDevErrNone = 0,
    kDevErrGemmProducerWait = TERN_DEVERR_GEMM_PRODUCER_WAIT,
    kDevErrGemmUnpackWait = TERN_DEVERR_GEMM_UNPACK_WAIT,
    kDevErrGemmMmaWait = TERN_DEVERR_GEMM_MMA_WAIT,
    kDevErrGemmEpilogueWait = TERN_DEVERR_GEMM_EPILOGUE_WAIT,
    kDevErrGemmTeardownWait = TERN_DEVERR_GEMM_TEARDOWN_WAIT,
    kDevErrGemvConsumerWait = TERN_DEVERR_GEMV_RANGE_FLAG_WAIT,
    kDevErrGemvActivationRange = TERN_DEVERR_GEMV_ACTIVATION_RANGE,
};

// Each translation unit whose kernels wait on barriers (the prefill and the
// decode products) defines its own word, so no relocatable device code is
// needed, and exports a host reader that reads and clears it.
__device__ __forceinline__ void report_device_error(int* word, int code) {
    atomicCAS(word, 0, code);
}
cudaError_t read_gemm_device_error(int* code);
cudaError_t read_gemv_device_error(int* code);
cudaError_t read_f3_device_error(int* code);
// One-CTA kernels that run a bounded wait nothing completes (tern_wait_selftest).
cudaError_t launch_flag_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_mbar_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Bounded waits.  No kernel of the library spins without a time limit: a wait
// that runs out returns false, and its caller reports a code into its sticky
// word and returns, so the context stays usable.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Waits until the word at p is non-zero, for at most limit_ns.
__device__ __forceinline__ bool wait_flag_nonzero(const unsigned* p, uint64_t limit_ns) {
    if (ld_acquire_gpu(p) != 0u) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire_gpu(p) != 0u) return true;
        if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch (PDL).
// ----------------------------------------------------------------------------
// Wait until the preceding kernel on the stream has completed and its memory
// is visible.  A no-op when the kernel was not launched with PDL.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next PDL-launched kernel on the stream to be scheduled.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Host helpers.
// ----------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks that the current device is an sm_103 part; caches per device.
tern_status check_device(int* sm_count);

// Launch bookkeeping (tern_last_launch_count).
void set_launch_count(int n);

// cudaLaunchKernelEx with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace tern
