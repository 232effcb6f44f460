// gemm_tc.cu -- prefill path of the W4A16 linear layer on the tcgen05 tensor
// cores (placeholder until the kernel lands: reports "not supported").
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

// Per-device word that kernels set when a bounded wait gives up.
__device__ uint32_t g_status_word = 0;

cudaError_t launch_gemm(const void*, const GemvMat&, int64_t, int64_t, int64_t, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t read_and_clear_status(uint32_t* word) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_status_word, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(uint32_t));
}

}  // namespace w4a16
