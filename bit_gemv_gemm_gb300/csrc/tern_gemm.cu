// tern_gemm.cu -- prefill product on the tcgen05 tensor cores (in progress).
#include "tern_common.cuh"

namespace tern {
namespace {
__device__ int g_gemm_error;
}  // namespace

cudaError_t read_gemm_device_error(int* code) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemm_error, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
}
}  // namespace tern

using namespace tern;

extern "C" size_t tern_gemm_workspace_bytes(int M, int N, int K) {
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return 0;
    return 256;
}

extern "C" tern_status tern_gemm(const void* x, const uint32_t* codes, const void* scales, void* y,
                                 int y_is_bf16, int M, int N, int K, void* workspace,
                                 size_t workspace_bytes, tern_stream_t stream) {
    set_launch_count(0);
    (void)x; (void)codes; (void)scales; (void)y; (void)y_is_bf16; (void)M; (void)N; (void)K;
    (void)workspace; (void)workspace_bytes; (void)stream;
    return TERN_ERR_SHAPE;
}
