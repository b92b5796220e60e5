// kq_noalloc.cu - kq_gemm_noalloc: the prefill GEMM with its scratch in a
// fixed device array of the library, for callers that cannot allocate
// device memory or pass a workspace (include/kq.h says who and why).  The
// source pages have no counterpart of this entry point.
#include "kq_internal.h"

#include <atomic>

namespace {

// The scratch: reserved on every GPU that loads the library, until exit.
// Every call on a device shares it; calls that overlap on the GPU race.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KQ_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol's name is only a host-side handle,
// not a device address).  Host threads making their first call on a device
// at the same time may both look it up; they store the same address.
constexpr int MAX_DEVICES = 64;
std::atomic<void *> g_scratch_ptr[MAX_DEVICES];

int scratch_of_current_device(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KQ_ERR_DEVICE;
    void *p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KQ_ERR_LAUNCH;
        }
        g_scratch_ptr[dev].store(p, std::memory_order_relaxed);
    }
    *ptr = p;
    return KQ_OK;
}

}  // namespace

extern "C" int kq_gemm_noalloc(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M,
                               float *y, cudaStream_t s) {
    if (f != KQ_Q4_K && f != KQ_Q5_K && f != KQ_Q6_K) return KQ_ERR_FORMAT;
    if (N < 0 || M < 0 || K <= 0 || K % kq::QK != 0) return KQ_ERR_ARG;
    // the activation image must fit; the split-tile room is used when it fits too
    const size_t need = kq::gemm_workspace_min_bytes(f, M, N, K);
    if (need > KQ_NOALLOC_SCRATCH_BYTES) return KQ_ERR_TOO_LARGE;
    void *ws = nullptr;
    if (need > 0 && M > 0 && N > 0) {
        if (int r = scratch_of_current_device(&ws)) return r;
    }
    return kq::gemm_common(f, packed, 1, nullptr, N, K, a, M, y, ws, need ? KQ_NOALLOC_SCRATCH_BYTES : 0, s);
}
