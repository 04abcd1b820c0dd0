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
    kDevErrGemmProducerWait = 0x101,   // TMA producer gave up waiting for a free stage
    kDevErrGemmUnpackWait = 0x102,     // unpack warps gave up waiting for raw tiles / free slots
    kDevErrGemmMmaWait = 0x103,        // MMA issuer gave up waiting for operands / TMEM
    kDevErrGemmEpilogueWait = 0x104,   // epilogue gave up waiting for an accumulator
    kDevErrGemmTeardownWait = 0x105,   // teardown gave up waiting for in-flight work
    kDevErrGemvProducerWait = 0x201,   // decode producer gave up waiting for a free ring slot
    kDevErrGemvConsumerWait = 0x202,   // decode warps gave up waiting for a code tile
};

// Each translation unit whose kernels wait on barriers (the prefill and the
// decode products) defines its own word, so no relocatable device code is
// needed, and exports a host reader that reads and clears it.
__device__ __forceinline__ void report_device_error(int* word, int code) {
    atomicCAS(word, 0, code);
}
cudaError_t read_gemm_device_error(int* code);
cudaError_t read_gemv_device_error(int* code);

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
