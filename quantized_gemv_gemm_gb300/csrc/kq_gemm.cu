// kq_gemm.cu - tensor-core prefill GEMM (tcgen05).  Placeholder until the
// tcgen05 kernel lands: every shape reports cudaErrorNotSupported and the
// C-ABI layer runs the CUDA-core token-group kernel instead.
#include "kq_internal.h"

namespace kq {

__device__ int g_status = 0;

size_t gemm_workspace_bytes(int, int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_gemm_tc(int, const void *, int64_t, int64_t, Q8K, int64_t, const int32_t *, int64_t,
                           uint64_t, float *, void *, size_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

int read_and_clear_status(cudaStream_t s, int *status) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    *status = v;
    return 0;
}

}  // namespace kq
