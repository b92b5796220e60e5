// kq_api.cu - the C ABI of libkq (declared in include/kq.h): argument
// checks on the host, then the launchers.  Nothing here allocates memory or
// synchronises, except kq_device_status().
#include "../../include/kq.h"
#include "kq_internal.h"

#include <atomic>

using namespace kq;

namespace kq {
static std::atomic<unsigned> g_launch_flags{0};
unsigned launch_flags() { return g_launch_flags.load(std::memory_order_relaxed); }
}  // namespace kq

namespace {

bool fmt_ok(int f) { return f == KQ_Q4_K || f == KQ_Q5_K || f == KQ_Q6_K; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(int64_t N, int64_t K) {
    if (N < 0 || K <= 0 || K % QK != 0) return KQ_ERR_ARG;
    return KQ_OK;
}

int check_q8k(const float *d, const int8_t *qs, const int16_t *bs) {
    if (!d || !qs || !bs) return KQ_ERR_ARG;
    if (!aligned(d, 4) || !aligned(qs, 16) || !aligned(bs, 16)) return KQ_ERR_ALIGN;
    return KQ_OK;
}

int launch_status(cudaError_t e) {
    if (e == cudaSuccess) return KQ_OK;
    cudaGetLastError();  // clear a non-sticky launch error
    return KQ_ERR_LAUNCH;
}

}  // namespace

namespace kq {
// Shared body of kq_gemm, kq_gemm_grouped and kq_gemm_noalloc: argument
// checks, then the tensor-core GEMM (or the small-M kernel below its token
// threshold).
int gemm_common(kq_format f, const void *packed, int64_t E, const int32_t *offsets, int64_t N, int64_t K,
                kq_q8k_const a, int64_t M, float *y, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (M < 0 || E < 1) return KQ_ERR_ARG;
    if (M == 0 || N == 0) return KQ_OK;
    if (!packed || !y) return KQ_ERR_ARG;
    if (int r = check_q8k(a.d, a.qs, a.bsums)) return r;
    if (!aligned(packed, 256) || !aligned(y, 4)) return KQ_ERR_ALIGN;
    const size_t need = gemm_workspace_min_bytes(f, M, N, K);
    if (need && (!ws || ws_bytes < need)) return KQ_ERR_WORKSPACE;
    if (ws && !aligned(ws, 256)) return KQ_ERR_ALIGN;
    const Q8K q{a.d, a.qs, a.bsums};
    const uint64_t expert_bytes = kq_repack_bytes(f, N, K);
    // a few token rows: the decode GEMV's weight stream, each item read once
    // for up to 8 tokens
    if (!offsets && M < GEMM_TC_MIN_M && K <= GEMV_MAX_K) return launch_status(launch_gemv_batch(f, packed, N, K, q, M, y, s));
    // a few grouped rows (MoE decode): one GEMV over every row's expert
    if (offsets && M < GEMM_TC_MIN_M && K <= GEMV_MAX_K && gemv_grouped_fits(M, K, 1))
        return launch_status(launch_gemv_grouped(f, 1, &packed, &N, E, offsets, &expert_bytes, K, q, nullptr, M, &y, s));
    cudaError_t e = launch_gemm_tc(f, packed, N, K, q, M, offsets, E, expert_bytes, y, ws, ws_bytes, s);
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        e = launch_mv(f, packed, N, K, q, M, offsets, E, expert_bytes, y, s);
    }
    return launch_status(e);
}
}  // namespace kq

extern "C" {

const char *kq_strerror(int code) {
    switch (code) {
    case KQ_OK: return "ok";
    case KQ_ERR_ARG: return "invalid argument (null pointer, negative size or K not a multiple of 256)";
    case KQ_ERR_ALIGN: return "misaligned pointer (16 bytes; 256 bytes for packed images and workspaces)";
    case KQ_ERR_FORMAT: return "unknown K-quant format";
    case KQ_ERR_LAUNCH: return "CUDA kernel launch failed";
    case KQ_ERR_TIMEOUT: return "a device-side bounded wait timed out";
    case KQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KQ_ERR_DEVICE: return "unsupported device";
    case KQ_ERR_TOO_LARGE: return "problem needs more scratch than the fixed array of kq_gemm_noalloc";
    default: return "unknown kq status";
    }
}

size_t kq_block_bytes(kq_format f) {
    if (f == KQ_Q8_0) return 34;
    return fmt_ok(f) ? (size_t)block_bytes(f) : 0;
}

int kq_quantize_q8k(const float *x, int64_t M, int64_t K, kq_q8k out, cudaStream_t s) {
    if (M < 0 || K <= 0 || K % QK != 0) return KQ_ERR_ARG;
    if (M == 0) return KQ_OK;
    if (!x) return KQ_ERR_ARG;
    if (int r = check_q8k(out.d, out.qs, out.bsums)) return r;
    if (!aligned(x, 16)) return KQ_ERR_ALIGN;
    return launch_status(launch_quantize(x, M, K, out.d, out.qs, out.bsums, s));
}

size_t kq_repack_bytes(kq_format f, int64_t N, int64_t K) {
    if (f == KQ_Q8_0) return check_shape(N, K) ? 0 : (size_t)q8_0_image_bytes(N, K);
    if (!fmt_ok(f) || check_shape(N, K)) return 0;
    uint64_t off[6];
    plane_offsets(f, N, K / QK, off);
    return (size_t)off[5];
}

int kq_repack(kq_format f, const void *disk, int64_t N, int64_t K, void *packed, cudaStream_t s) {
    if (!fmt_ok(f) && f != KQ_Q8_0) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (N == 0) return KQ_OK;
    if (!disk || !packed) return KQ_ERR_ARG;
    if (!aligned(disk, 16) || !aligned(packed, 256)) return KQ_ERR_ALIGN;
    if (f == KQ_Q8_0)
        return launch_status(launch_repack_q8_0(static_cast<const uint8_t *>(disk), N, K, static_cast<uint8_t *>(packed), s));
    return launch_status(launch_repack(f, static_cast<const uint8_t *>(disk), N, K, static_cast<uint8_t *>(packed), s));
}

int kq_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *qs, cudaStream_t s) {
    if (M < 0 || K <= 0 || K % 32 != 0) return KQ_ERR_ARG;
    if (M == 0) return KQ_OK;
    if (!x || !d || !qs) return KQ_ERR_ARG;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(d, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_quantize_q8_0(x, M, K, d, qs, s));
}

int kq_gemm_q8_0(const void *packed, int64_t N, int64_t K, const float *d, const int8_t *qs, int64_t M, float *y,
                 cudaStream_t s) {
    if (N < 0 || M < 0 || K <= 0 || K % QK != 0) return KQ_ERR_ARG;
    if (M == 0 || N == 0) return KQ_OK;
    if (!packed || !d || !qs || !y) return KQ_ERR_ARG;
    if (!aligned(packed, 256) || !aligned(d, 16) || !aligned(qs, 16) || !aligned(y, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_gemm_q8_0(packed, N, K, d, qs, M, y, s));
}

int kq_gemv_q8_0(const void *packed, int64_t N, int64_t K, const float *d, const int8_t *qs, float *y,
                 cudaStream_t s) {
    if (int r = check_shape(N, K)) return r;
    if (K > GEMV_MAX_K) return KQ_ERR_ARG;
    if (N == 0) return KQ_OK;
    if (!packed || !d || !qs || !y) return KQ_ERR_ARG;
    if (!aligned(packed, 256) || !aligned(qs, 16) || !aligned(d, 4) || !aligned(y, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_gemv_q8_0(packed, N, K, d, qs, nullptr, y, s));
}

int kq_gemv_q8_0_fused(const void *packed, int64_t N, int64_t K, const float *x, float *y, cudaStream_t s) {
    if (int r = check_shape(N, K)) return r;
    if (K > GEMV_MAX_K) return KQ_ERR_ARG;
    if (N == 0) return KQ_OK;
    if (!packed || !x || !y) return KQ_ERR_ARG;
    if (!aligned(packed, 256) || !aligned(x, 16) || !aligned(y, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_gemv_q8_0(packed, N, K, nullptr, nullptr, x, y, s));
}

size_t kq_gemv_workspace_bytes(void) { return GEMV_WORKSPACE_BYTES; }

// a GEMV workspace: none, or at least GEMV_WORKSPACE_BYTES, 16-byte aligned
static int check_gemv_ws(const void *ws, size_t bytes) {
    if (!ws) return KQ_OK;
    if (bytes < GEMV_WORKSPACE_BYTES) return KQ_ERR_WORKSPACE;
    return aligned(ws, 16) ? KQ_OK : KQ_ERR_ALIGN;
}

int kq_gemv(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, float *y, void *workspace,
            size_t workspace_bytes, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (N == 0) return KQ_OK;
    if (!packed || !y) return KQ_ERR_ARG;
    if (int r = check_q8k(a.d, a.qs, a.bsums)) return r;
    if (!aligned(packed, 256) || !aligned(y, 4)) return KQ_ERR_ALIGN;
    if (int r = check_gemv_ws(workspace, workspace_bytes)) return r;
    const Q8K q{a.d, a.qs, a.bsums};
    if (K <= GEMV_MAX_K)
        return launch_status(launch_gemv(f, 1, &packed, &N, K, nullptr, q, &y, workspace, workspace_bytes, s));
    return launch_status(launch_mv(f, packed, N, K, q, 1, nullptr, 1, 0, y, s));
}

// The body of kq_gemv_fused (M = 1) and kq_gemv_fused_batch.
static int gemv_fused_common(kq_format f, int n_mats, const void *const *packed, const int64_t *N, int64_t K,
                             const float *x, int64_t M, float *const *y, void *workspace, size_t workspace_bytes,
                             cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (M < 0) return KQ_ERR_ARG;
    if (n_mats < 1 || n_mats > GEMV_FUSED_MAX || !packed || !N || !y) return KQ_ERR_ARG;
    if (K <= 0 || K % QK != 0 || K > GEMV_MAX_K) return KQ_ERR_ARG;
    if (int r = check_gemv_ws(workspace, workspace_bytes)) return r;
    int64_t total = 0;
    for (int m = 0; m < n_mats; ++m) {
        if (N[m] < 0) return KQ_ERR_ARG;
        total += N[m];
        if (N[m] == 0) continue;
        if (!packed[m] || !y[m]) return KQ_ERR_ARG;
        if (!aligned(packed[m], 256) || !aligned(y[m], 4)) return KQ_ERR_ALIGN;
    }
    if (total == 0 || M == 0) return KQ_OK;
    if (!x) return KQ_ERR_ARG;
    if (!aligned(x, 16)) return KQ_ERR_ALIGN;
    // matrices with N = 0 are dropped
    const void *pk[GEMV_MAX_MATRICES];
    int64_t nn[GEMV_MAX_MATRICES];
    float *yy[GEMV_MAX_MATRICES];
    int k = 0;
    for (int m = 0; m < n_mats; ++m)
        if (N[m] > 0) { pk[k] = packed[m]; nn[k] = N[m]; yy[k] = y[m]; ++k; }
    if (M == 1)
        return launch_status(
            launch_gemv(f, k, pk, nn, K, x, Q8K{nullptr, nullptr, nullptr}, yy, workspace, workspace_bytes, s));
    return launch_status(launch_gemv_fused_batch(f, k, pk, nn, K, x, M, yy, workspace, workspace_bytes, s));
}

int kq_gemv_fused(kq_format f, int n_mats, const void *const *packed, const int64_t *N, int64_t K, const float *x,
                  float *const *y, void *workspace, size_t workspace_bytes, cudaStream_t s) {
    return gemv_fused_common(f, n_mats, packed, N, K, x, 1, y, workspace, workspace_bytes, s);
}

int kq_gemv_fused_batch(kq_format f, int n_mats, const void *const *packed, const int64_t *N, int64_t K,
                        const float *x, int64_t M, float *const *y, void *workspace, size_t workspace_bytes,
                        cudaStream_t s) {
    return gemv_fused_common(f, n_mats, packed, N, K, x, M, y, workspace, workspace_bytes, s);
}

size_t kq_gemm_workspace_bytes(kq_format f, int64_t M, int64_t N, int64_t K) {
    if (!fmt_ok(f) || M < 0 || check_shape(N, K)) return 0;
    return gemm_workspace_bytes(f, M, N, K);
}

size_t kq_gemm_min_workspace_bytes(kq_format f, int64_t M, int64_t N, int64_t K) {
    if (!fmt_ok(f) || M < 0 || check_shape(N, K)) return 0;
    return gemm_workspace_min_bytes(f, M, N, K);
}

int kq_gemm(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M, float *y,
            void *workspace, size_t workspace_bytes, cudaStream_t s) {
    return gemm_common(f, packed, 1, nullptr, N, K, a, M, y, workspace, workspace_bytes, s);
}

int kq_gemv_grouped_fused(kq_format f, int n_sets, const void *const *packed, const int64_t *N, int64_t K, int64_t E,
                          const int32_t *row_offsets, const float *x, int64_t M, float *const *y, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (M < 0 || E < 1 || n_sets < 1 || n_sets > GEMV_FUSED_MAX || !packed || !N || !y) return KQ_ERR_ARG;
    if (K <= 0 || K % QK != 0 || K > GEMV_MAX_K) return KQ_ERR_ARG;
    if (M == 0) return KQ_OK;
    if (!gemv_grouped_fits(M, K, n_sets)) return KQ_ERR_ARG;
    if (!x || !row_offsets) return KQ_ERR_ARG;
    if (!aligned(x, 16) || !aligned(row_offsets, 4)) return KQ_ERR_ALIGN;
    uint64_t eb[GEMV_FUSED_MAX];
    for (int st = 0; st < n_sets; ++st) {
        if (N[st] < 1 || !packed[st] || !y[st]) return KQ_ERR_ARG;
        if (!aligned(packed[st], 256) || !aligned(y[st], 4)) return KQ_ERR_ALIGN;
        eb[st] = kq_repack_bytes(f, N[st], K);
    }
    return launch_status(launch_gemv_grouped(f, n_sets, packed, N, E, row_offsets, eb, K, Q8K{nullptr, nullptr, nullptr},
                                             x, M, y, s));
}

int kq_gemm_grouped(kq_format f, const void *packed, int64_t E, const int32_t *row_offsets, int64_t N, int64_t K,
                    kq_q8k_const a, int64_t M_total, float *y, void *workspace, size_t workspace_bytes,
                    cudaStream_t s) {
    if (!row_offsets && M_total > 0) return KQ_ERR_ARG;
    if (row_offsets && !aligned(row_offsets, 4)) return KQ_ERR_ALIGN;
    return gemm_common(f, packed, E, row_offsets, N, K, a, M_total, y, workspace, workspace_bytes, s);
}

int kq_debug_partials(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M,
                      int32_t *isum, int32_t *msum, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (M < 0) return KQ_ERR_ARG;
    if (M == 0 || N == 0) return KQ_OK;
    if (!packed || !isum || !msum) return KQ_ERR_ARG;
    if (int r = check_q8k(a.d, a.qs, a.bsums)) return r;
    if (!aligned(packed, 256) || !aligned(isum, 4) || !aligned(msum, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_partials(f, packed, N, K, Q8K{a.d, a.qs, a.bsums}, M, isum, msum, s));
}

int kq_debug_batch_partials(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M,
                            int32_t *isum, int32_t *msum, cudaStream_t s) {
    if (f != KQ_Q4_K && f != KQ_Q6_K) return fmt_ok(f) ? KQ_ERR_ARG : KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (M < 0 || M > 8) return KQ_ERR_ARG;
    if (M == 0 || N == 0) return KQ_OK;
    if (!packed || !isum || !msum) return KQ_ERR_ARG;
    if (int r = check_q8k(a.d, a.qs, a.bsums)) return r;
    if (!aligned(packed, 256) || !aligned(isum, 4) || !aligned(msum, 4)) return KQ_ERR_ALIGN;
    return launch_status(launch_mma_partials(f, packed, N, K, Q8K{a.d, a.qs, a.bsums}, M, isum, msum, s));
}

int kq_debug_gemm_partials(kq_format f, const void *packed, int64_t E, const int32_t *row_offsets, int64_t N,
                           int64_t K, kq_q8k_const a, int64_t M, int32_t *isum, int32_t *msum, void *workspace,
                           size_t workspace_bytes, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (M < GEMM_TC_MIN_M || E < 1 || (E > 1 && !row_offsets)) return KQ_ERR_ARG;
    if (N == 0) return KQ_OK;
    if (!packed || !isum || !msum) return KQ_ERR_ARG;
    if (int r = check_q8k(a.d, a.qs, a.bsums)) return r;
    if (!aligned(packed, 256) || !aligned(isum, 4) || !aligned(msum, 4)) return KQ_ERR_ALIGN;
    const size_t need = gemm_workspace_min_bytes(f, M, N, K);
    if (!workspace || workspace_bytes < need) return KQ_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return KQ_ERR_ALIGN;
    const uint64_t expert_bytes = kq_repack_bytes(f, N, K);
    cudaError_t e = launch_gemm_tc_partials(f, packed, N, K, Q8K{a.d, a.qs, a.bsums}, M, row_offsets, E, expert_bytes,
                                            isum, msum, workspace, workspace_bytes, s);
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        return KQ_ERR_ARG;
    }
    return launch_status(e);
}

int kq_debug_decode(kq_format f, const void *packed, int64_t N, int64_t K, int32_t *q, int32_t *sc, int32_t *mn,
                    float *d, float *dmin, cudaStream_t s) {
    if (!fmt_ok(f)) return KQ_ERR_FORMAT;
    if (int r = check_shape(N, K)) return r;
    if (N == 0) return KQ_OK;
    if (!packed || !q || !sc || !mn || !d || !dmin) return KQ_ERR_ARG;
    if (!aligned(packed, 256)) return KQ_ERR_ALIGN;
    return launch_status(launch_debug_decode(f, packed, N, K, q, sc, mn, d, dmin, s));
}

int kq_debug_wait_timeout(uint64_t limit_ns, cudaStream_t s) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return KQ_ERR_ARG;
    return launch_status(launch_wait_timeout(limit_ns, s));
}

int kq_measure_mma_s8(int64_t blocks, int64_t iters, int32_t *out, cudaStream_t s) {
    if (blocks < 0 || iters < 0 || blocks > (int64_t)INT32_MAX) return KQ_ERR_ARG;
    if (blocks == 0) return KQ_OK;
    if (!out) return KQ_ERR_ARG;
    return launch_status(launch_mma_s8_rate(blocks, iters, out, s));
}

int kq_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s) {
    if (bytes % 16 != 0 || bytes > ((size_t)1 << 40)) return KQ_ERR_ARG;
    if (bytes == 0) return KQ_OK;
    if (!src || !dst) return KQ_ERR_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16)) return KQ_ERR_ALIGN;
    return launch_status(launch_copy_in(src, dst, bytes, s));
}

unsigned kq_set_launch_flags(unsigned flags) {
    return g_launch_flags.exchange(flags & (KQ_LAUNCH_PDL | KQ_LAUNCH_GEMV_SPLIT | KQ_LAUNCH_GEMM_SPLIT),
                                   std::memory_order_relaxed);
}

unsigned kq_get_launch_flags(void) { return launch_flags(); }

int kq_device_status(cudaStream_t s) {
    int st = 0, sg = 0;
    if (read_and_clear_status(s, &st) || read_and_clear_gemv_status(s, &sg)) return KQ_ERR_LAUNCH;
    return (st || sg) ? KQ_ERR_TIMEOUT : KQ_OK;
}

}  // extern "C"
