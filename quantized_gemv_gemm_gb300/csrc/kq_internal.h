// kq_internal.h - host-side launchers shared between the translation units of
// libkq.  Arguments are validated by the C-ABI layer (kq_api.cu) before any
// of these run; they only shape grids and enqueue kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kq_device.cuh"
#include "../../include/kq.h"

namespace kq {

// Library-wide launch options (kq_set_launch_flags).
constexpr unsigned LAUNCH_PDL = 1u;
constexpr unsigned LAUNCH_GEMV_SPLIT = 2u;
constexpr unsigned LAUNCH_GEMM_SPLIT = 4u;
unsigned launch_flags();

struct Q8K {
    const float *d;
    const int8_t *qs;
    const int16_t *bsums;
};

// Q8_K quantization of x [M][K].
cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, float *d, int8_t *qs,
                            int16_t *bsums, cudaStream_t s);

// The Q8_0 rail (kq_q8_0.cu): image size, repack, Q8_0-form activations, GEMV.
uint64_t q8_0_image_bytes(int64_t N, int64_t K);
cudaError_t launch_repack_q8_0(const uint8_t *disk, int64_t N, int64_t K, uint8_t *packed, cudaStream_t s);
cudaError_t launch_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *qs, cudaStream_t s);
// (x != nullptr: the fp32 row, quantized in the kernel; d, qs unused)
cudaError_t launch_gemv_q8_0(const void *packed, int64_t N, int64_t K, const float *d, const int8_t *qs,
                             const float *x, float *y, cudaStream_t s);

// Q8_0 prefill GEMM (kq_q8_0_gemm.cu): y [M][N] from the image and M
// Q8_0-form activation rows.
cudaError_t launch_gemm_q8_0(const void *packed, int64_t N, int64_t K, const float *d_a, const int8_t *q_a, int64_t M,
                             float *y, cudaStream_t s);

// Disk superblocks -> packed image.
cudaError_t launch_repack(int f, const uint8_t *disk, int64_t N, int64_t K, uint8_t *packed,
                          cudaStream_t s);

// CUDA-core matrix-vector family: M tokens (grouped by expert when
// row_offsets != nullptr), each weight superblock unpacked once per pass
// over a group of up to 8 tokens.
cudaError_t launch_mv(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                      const int32_t *row_offsets, int64_t E, uint64_t expert_bytes, float *y,
                      cudaStream_t s);

// Decode GEMV over nmat (<= 4) matrices sharing one input row: either the
// fp32 row x (quantized inside the kernel) or, when x is null, Q8_K planes a.
// ws: null, or a zero-filled workspace of GEMV_WORKSPACE_BYTES: one 64-bit
// word per row of a row group cut between two blocks, [GEMV_MAX_BLOCKS][16].
constexpr int GEMV_MAX_MATRICES = 16;  // kernel tables (kq_gemv_fused takes at most GEMV_FUSED_MAX)
constexpr int GEMV_FUSED_MAX = 4;
constexpr int64_t GEMV_MAX_K = 40960;
constexpr int64_t GEMV_MAX_BLOCKS = 512;
constexpr size_t GEMV_WORKSPACE_BYTES = KQ_GEMV_WORKSPACE_BYTES;
static_assert(GEMV_MAX_BLOCKS * 16 * 8 <= (int64_t)KQ_GEMV_WORKSPACE_BYTES, "GEMV workspace layout");
cudaError_t launch_gemv(int f, int nmat, const void *const *packed, const int64_t *N, int64_t K, const float *x,
                        Q8K a, float *const *y, void *ws, size_t ws_bytes, cudaStream_t s);

// Small batches (M < GEMM_TC_MIN_M token rows) on the decode GEMV's stream:
// passes of up to 8 tokens that read each weight item once.
constexpr int64_t GEMM_TC_MIN_M = 16;
cudaError_t launch_gemv_batch(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, float *y,
                              cudaStream_t s);

// Fused quantize + GEMV of a small batch: M fp32 rows, up to GEMV_FUSED_MAX
// matrices sharing them, y[m] [M][N[m]].
cudaError_t launch_gemv_fused_batch(int f, int nmat, const void *const *packed, const int64_t *N, int64_t K,
                                    const float *x, int64_t M, float *const *y, void *ws, size_t ws_bytes,
                                    cudaStream_t s);

// Grouped rows (MoE decode): M token rows grouped by expert (device offsets
// [E+1]), one GEMV launch over every row's expert in each of `sets` weight
// sets sharing the rows (sets * M <= GEMV_MAX_MATRICES); the rows come as
// Q8_K planes (x == nullptr) or as fp32 x [M][K] quantized in the kernel.
bool gemv_grouped_fits(int64_t M, int64_t K, int sets);
cudaError_t launch_gemv_grouped(int f, int sets, const void *const *packed, const int64_t *N, int64_t E,
                                const int32_t *offsets, uint64_t const *expert_bytes, int64_t K, Q8K a,
                                const float *x, int64_t M, float *const *y, cudaStream_t s);

cudaError_t launch_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                            int32_t *isum, int32_t *msum, cudaStream_t s);
// the same from the small-batch passes' integer-MMA fold (Q4_K, Q6_K; M <= 8)
cudaError_t launch_mma_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, int32_t *isum,
                                int32_t *msum, cudaStream_t s);

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_mma_s8_rate(int64_t blocks, int64_t iters, int32_t *out, cudaStream_t s);
cudaError_t launch_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s);
cudaError_t launch_debug_decode(int f, const void *packed, int64_t N, int64_t K, int32_t *q,
                                int32_t *sc, int32_t *mn, float *d, float *dmin, cudaStream_t s);

// Tensor-core GEMM (tcgen05).  Returns cudaErrorNotSupported when the shape
// or device is not handled, so the caller can fall back to launch_mv.
// gemm_workspace_bytes: the workspace with room for the dense split-tile
// schedule (what kq_gemm_workspace_bytes reports); gemm_workspace_min_bytes:
// the least a launch accepts (the activation image alone; the dense GEMM then
// runs a block per tile).
size_t gemm_workspace_bytes(int f, int64_t M, int64_t N, int64_t K);
size_t gemm_workspace_min_bytes(int f, int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_tc(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                           const int32_t *row_offsets, int64_t E, uint64_t expert_bytes, float *y,
                           void *workspace, size_t workspace_bytes, cudaStream_t s);

// The same kernel with the debug epilogue: per (row, weight row, superblock)
// the int32 sums isum / msum [M][N][K/256] (zero-filled here, then
// accumulated) instead of y.
cudaError_t launch_gemm_tc_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                                    const int32_t *row_offsets, int64_t E, uint64_t expert_bytes, int32_t *isum,
                                    int32_t *msum, void *workspace, size_t workspace_bytes, cudaStream_t s);

// The C-ABI body of the three GEMM entry points (kq_api.cu).
int gemm_common(kq_format f, const void *packed, int64_t E, const int32_t *offsets, int64_t N, int64_t K,
                kq_q8k_const a, int64_t M, float *y, void *ws, size_t ws_bytes, cudaStream_t s);

// Device status words of the bounded waits (tensor-core GEMM; decode GEMV).
int read_and_clear_status(cudaStream_t s, int *status);
int read_and_clear_gemv_status(cudaStream_t s, int *status);

}  // namespace kq
