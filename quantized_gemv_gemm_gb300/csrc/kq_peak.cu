// kq_peak.cu - measurement hook: the int8 tensor-core rate of the legacy
// warp-level MMA (mma.sync m16n8k32 s8 x s8 -> s32), the integer MMA that
// sm_103a offers (it has no integer tcgen05.mma).  The prefill GEMM runs its
// exact-integer contraction on the fp16 tcgen05 pipe instead; this kernel
// gives the int8 rate that path is compared against.
#include "kq_internal.h"

namespace kq {

// Every warp issues `iters` rounds of 8 independent MMAs (8 accumulator sets,
// so the tensor pipe never waits on one result).  A and B are all ones, so
// each accumulator element ends at 32 * iters and each thread's checksum at
// 8 * 4 * 32 * iters, which the caller can check.
__global__ void __launch_bounds__(256) mma_s8_rate_kernel(int64_t iters, int32_t *out) {
    const uint32_t a0 = 0x01010101u, a1 = a0, a2 = a0, a3 = a0, b0 = a0, b1 = a0;
    int32_t c[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
    int32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

cudaError_t launch_mma_s8_rate(int64_t blocks, int64_t iters, int32_t *out, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    mma_s8_rate_kernel<<<(unsigned)blocks, 256, 0, s>>>(iters, out);
    return cudaGetLastError();
}

}  // namespace kq
