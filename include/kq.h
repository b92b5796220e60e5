/*
 * kq.h - C ABI of libkq: K-quant (Q4_K / Q5_K / Q6_K) x Q8_K matrix products
 * on GB300 (sm_103a).
 *
 * Method source, cited as [kq-arc] below: the page "dasLLAMA: K-quant
 * kernel arc - kq v2 integer folds, kq v3 panel-scratch tiles, chain
 * regrain, parity gates" (daScript pull request #3450), its section
 * "The pieces" (the kq v2 and kq v3 bullets) and two of its commit
 * messages: the k4 kq-v2 commit (Q8_K activations and integer folds for
 * Q4_K) and the k5/k6 kq-v2 commit (the same scheme for Q5_K and Q6_K).
 *
 * Conventions for every entry point
 *   - Pointers named as device pointers must be device (or managed) memory
 *     of the current CUDA device; the library never allocates, frees or
 *     synchronises.  All work is enqueued on the caller's stream `s`
 *     (0 = legacy default stream) and the call returns before it finishes.
 *   - The caller owns every buffer.  Inputs are read-only.
 *   - Sizes are int64_t; K must be a positive multiple of 256.
 *   - Return value: KQ_OK (0) or a negative kq_status.  Argument errors are
 *     detected on the host before anything is enqueued; KQ_ERR_LAUNCH
 *     reports a CUDA launch failure (cudaGetLastError after the launch).
 *     kq_strerror() names a code.
 *   - Nothing here reads the status of earlier launches except
 *     kq_device_status(), which synchronises the given stream.
 *
 * Block formats (256 weights per superblock, GGUF byte order, little
 * endian; the pages name the fields, the bit layout is the public GGUF one):
 *   Q4_K, 144 B: d f16 | dmin f16 | scales[12] (8 six-bit sub-scales and 8
 *                six-bit sub-mins, one per 32 weights) | qs[128] (4-bit)
 *   Q5_K, 176 B: d f16 | dmin f16 | scales[12] | qh[32] (5th bits) | qs[128]
 *   Q6_K, 210 B: ql[128] (low 4 bits) | qh[64] (high 2 bits) |
 *                scales[16] (signed int8, one per 16 weights) | d f16
 *   Q8_K activations ([kq-arc], k4 kq-v2 commit: a single fp32 scale for
 *   each 256-element block and a sum for each 16 elements) are held as
 *   three row-major planes:
 *     d     float  [M][K/256]   block scale d8
 *     qs    int8   [M][K]       quants in -127..127
 *     bsums int16  [M][K/16]    sum of each 16 consecutive quants
 *
 * Output of every product: y float32 row-major [M][N] (M tokens, N weight
 * rows), y[m][n] = sum over superblocks sb of
 *     Q4_K/Q5_K: d*d8*isum - dmin*d8*msum
 *                isum = sum_j sc_j * dot32_j(q, a8), msum = sum_j m_j*(bs_2j + bs_2j+1)
 *     Q6_K:      d*d8*(iacc - 32*bacc)
 *                iacc = sum_i sc_i * dot16_i(q, a8), bacc = sum_i sc_i * bs_i
 * with isum, msum, iacc, bacc formed exactly in int32 and one float fold per
 * superblock ([kq-arc], "The pieces", kq v2 bullet).
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KQ_Q8_0: Q8_0 weights (blocks of 32 values: fp16 d, 32 int8 q), accepted
 * only by kq_block_bytes, kq_repack_bytes, kq_repack and kq_gemv_q8_0; every
 * K-quant entry point returns KQ_ERR_FORMAT for it. */
typedef enum { KQ_Q4_K = 1, KQ_Q5_K = 2, KQ_Q6_K = 3, KQ_Q8_0 = 4 } kq_format;

typedef enum {
    KQ_OK = 0,
    KQ_ERR_ARG = -1,       /* null pointer, K % 256 != 0, negative size, ... */
    KQ_ERR_ALIGN = -2,     /* a pointer is not 16-byte aligned (256 for packed) */
    KQ_ERR_FORMAT = -3,    /* unknown kq_format */
    KQ_ERR_LAUNCH = -4,    /* CUDA reported an error at launch */
    KQ_ERR_TIMEOUT = -5,   /* a device-side bounded wait gave up (see kq_device_status) */
    KQ_ERR_WORKSPACE = -6, /* workspace missing or smaller than required */
    KQ_ERR_DEVICE = -7,    /* the current device is not sm_103 / cannot run the kernel */
    KQ_ERR_TOO_LARGE = -8  /* the problem needs more scratch than kq_gemm_noalloc's fixed array */
} kq_status;

/* Q8_K planes (device pointers), see the format note above. */
typedef struct { const float *d; const int8_t *qs; const int16_t *bsums; } kq_q8k_const;
typedef struct { float *d; int8_t *qs; int16_t *bsums; } kq_q8k;

/* Human-readable name of a kq_status. */
const char *kq_strerror(int code);

/* Bytes of one disk block of format f: a 256-weight superblock for the
 * K-quants (144 / 176 / 210), a 32-weight block for KQ_Q8_0 (34); 0 if
 * unknown. */
size_t kq_block_bytes(kq_format f);

/*
 * Activation quantization to Q8_K ([kq-arc], k4 kq-v2 commit, which names
 * quantize_q8_k_into: one fp32 scale per 256 activations plus per-16 sums).
 * Per 256-block of each
 * row of x: amax = max|x|; if amax == 0 then d8 = 0 and q = 0; otherwise
 * iscale = 127/amax and q = clamp(round_half_even(x*iscale), -127, 127), both
 * steps in IEEE fp32, and d8 = amax/127.  bsums[i] sums q over 16i..16i+15.
 *   x   device float32 [M][K] row-major, 16-byte aligned, finite values
 *   out device planes as described above (qs 16-byte aligned)
 * Errors: KQ_ERR_ARG (null, M < 0, K % 256), KQ_ERR_ALIGN, KQ_ERR_LAUNCH.
 * M == 0 is a no-op.
 */
int kq_quantize_q8k(const float *x, int64_t M, int64_t K, kq_q8k out, cudaStream_t s);

/*
 * Size in bytes of the repacked (device) image of an [N][K] weight matrix.
 * Always a multiple of 256, so experts stacked back to back stay aligned.
 * Returns 0 for an unknown format, N < 0 or K not a positive multiple of 256.
 *
 * Packed image ([kq-arc], k4 kq-v2 commit: the scale block is stored as it
 * is on disk and the rows are repacked into interleaved groups; kq v3
 * commit: the planes in DRAM stay bit-packed, never byte-expanded).  Rows
 * are taken in groups of 16 (the last group padded with zero rows).  Each
 * plane holds, for every (row group g, superblock sb) in the order
 * g * K/256 + sb, one contiguous chunk with that plane's bytes of the 16
 * rows' superblock sb; planes start on 256-byte boundaries:
 *   Q4_K: qs  (2048 B chunks) | hdr (256 B: d, dmin, scales[12] per row)
 *   Q5_K: qs  (2048) | qh (512) | hdr (256)
 *   Q6_K: ql  (2048) | qh (1024) | sc (256) | d (32, fp16 per row)
 * Inside a chunk, row r's 16-byte piece i (disk bytes 16i .. 16i+15 of that
 * field) sits at: qs/ql 512*(i%4) + 16*(r + 16*(i/4)); Q6_K qh
 * 512*(i%2) + 16*(r + 16*(i/2)); Q5_K qh 256*i + 16*r; hdr/sc 16*r; d 2*r.
 * Every byte of the disk superblock is kept once.  A last plane holds data
 * derived at repack time for the tensor-core GEMM: per (row group,
 * superblock), two uint32, for each half of the superblock the largest
 * over the group's rows of W1 = sum |w'| (w' = sub-scale * q, Q6_K
 * q - 32), which bounds every partial sum of the half's integer dot
 * (|a8| <= 128) and so tells the GEMM how long its fp32 accumulators may
 * run exactly.  The image is the disk size of the rows padded to a multiple
 * of 16, plus 8 bytes per (row group, superblock), plus at most 4 x 255
 * bytes of plane padding.
 */
size_t kq_repack_bytes(kq_format f, int64_t N, int64_t K);
/*
 * KQ_Q8_0 images (K a positive multiple of 256): rows in groups of 16 as
 * above, two planes: qs (4096-byte chunks; row r's 16 quants of columns
 * 16k..16k+15 of the superblock at 256*k + 16*r) | d (256-byte chunks; row
 * r's 8 fp16 block scales at 16*r).  1.0625 bytes per weight, as on disk.
 */

/*
 * One-time repack of disk superblocks into the packed image ([kq-arc], k4
 * kq-v2 commit: the weights are transcoded and repacked once at load, and
 * the repacked planes dequantize bit-identically to the file).
 *   disk   device uint8 [N][K/256][block_bytes] (GGUF order; KQ_Q8_0:
 *          [N][K/32][34]), 16-byte aligned
 *   packed device, kq_repack_bytes(f, N, K) bytes, 256-byte aligned
 * Errors: KQ_ERR_ARG, KQ_ERR_FORMAT, KQ_ERR_ALIGN, KQ_ERR_LAUNCH.
 */
int kq_repack(kq_format f, const void *disk, int64_t N, int64_t K, void *packed, cudaStream_t s);

/*
 * Workspace of the decode GEMV (kq_gemv, kq_gemv_fused): KQ_GEMV_WORKSPACE_BYTES
 * (64 KiB) of device memory, 16-byte aligned, zero-filled once before its
 * first use; every call leaves it zero-filled again.  With it the GEMV gives
 * every SM an even share of the superblocks, cutting a row group between two
 * blocks where needed and finishing that row group through the workspace;
 * without it (NULL) each block takes whole row groups, which leaves SMs idle
 * when the row groups do not divide evenly among them.  Either way the
 * result does not depend on timing (every sum has a fixed order; the two
 * ways differ only in float rounding).  Calls on one stream may share a workspace (each reads it only
 * after the previous kernels in the stream have completed); calls that may
 * run at the same time on different streams need one each.  The source
 * pages have no counterpart of this buffer (their decode kernels run one
 * row per work-group, on hardware where that fills the device).
 * kq_gemv_workspace_bytes() returns the same number, for bindings.
 */
#define KQ_GEMV_WORKSPACE_BYTES ((size_t)64 << 10)
size_t kq_gemv_workspace_bytes(void);

/*
 * Decode GEMV, M = 1 ([kq-arc], "The pieces", kq v2: the GEMV unpacks the
 * packed planes in the kernel; kq v3 bullet: decode is bound by DRAM
 * traffic, so every byte of the weight planes costs decode time).  y[n]
 * for n < N, as in the header note.
 *   packed     device image from kq_repack (256-byte aligned)
 *   a          device Q8_K planes of one row of K
 *   y          device float32 [N]
 *   workspace  NULL, or KQ_GEMV_WORKSPACE_BYTES as described above
 * Errors: KQ_ERR_ARG, KQ_ERR_FORMAT, KQ_ERR_ALIGN, KQ_ERR_WORKSPACE
 * (workspace_bytes too small), KQ_ERR_LAUNCH.
 */
int kq_gemv(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a,
            float *y, void *workspace, size_t workspace_bytes, cudaStream_t s);

/*
 * Fused decode GEMV: quantize + GEMV in one launch, over up to four matrices
 * that share one input row (q/k/v projections, gate/up).  The fp32 row x is
 * quantized to Q8_K inside the kernel, bit-identically to kq_quantize_q8k,
 * and y_m = W_m x for each matrix m, as kq_gemv computes it.  This is the
 * kernel-level form of the page's chain regrain ([kq-arc], "The pieces":
 * the decode chains quantize the activation image where it is consumed, in
 * whole superblocks).
 *   n_mats  1..4
 *   packed  host array of n_mats device pointers to packed images of format
 *           f (256-byte aligned); N host array of their row counts (>= 0;
 *           a matrix with N = 0 is skipped)
 *   K       shared inner dimension: a multiple of 256, at most 40960
 *   x       device float32 [K], 16-byte aligned, finite values
 *   y       host array of n_mats pointers, y[m] float32 [N[m]] in device
 *           memory or in mapped pinned host memory (see kq_copy_in)
 *   workspace  NULL, or KQ_GEMV_WORKSPACE_BYTES as for kq_gemv
 * The host arrays are read during the call only.
 * Errors: KQ_ERR_FORMAT, KQ_ERR_ARG (n_mats out of range, null, K), KQ_ERR_ALIGN,
 * KQ_ERR_WORKSPACE, KQ_ERR_LAUNCH.
 */
int kq_gemv_fused(kq_format f, int n_mats, const void *const *packed, const int64_t *N, int64_t K,
                  const float *x, float *const *y, void *workspace, size_t workspace_bytes,
                  cudaStream_t s);

/*
 * Fused quantize + GEMV of a small batch: as kq_gemv_fused for M token rows
 * at once (batched decode).  Each weight item is read once per pass of up to
 * 8 rows (4 when K > 8192, fewer for longer K), and every row is quantized
 * inside the kernel bit-identically to kq_quantize_q8k.  M = 1 is
 * kq_gemv_fused.  There is no counterpart of a batched entry point in the
 * source pages; it is the decode chain's fused quantize ([kq-arc], "The
 * pieces") for several sequences decoding together.
 *   x          device float32 [M][K] (row-major, 16-byte aligned), finite
 *   y          host array of n_mats device pointers, y[m] float32 [M][N[m]]
 *   workspace  as for kq_gemv (used by the single-row passes)
 * Errors: as kq_gemv_fused; KQ_ERR_ARG also for M < 0.  M == 0 is a no-op.
 */
int kq_gemv_fused_batch(kq_format f, int n_mats, const void *const *packed, const int64_t *N, int64_t K,
                        const float *x, int64_t M, float *const *y, void *workspace,
                        size_t workspace_bytes, cudaStream_t s);

/*
 * Size of the device workspace kq_gemm / kq_gemm_grouped use for M token
 * rows of K and N weight rows: an fp16 image of the activation quants and
 * bsums with the transposed scales, then room for the dense GEMM's split-
 * tile schedule (two fp32 128 x 128 partial tiles per SM and a counter per
 * 128 x 128 output tile).  With it, kq_gemm runs one block per SM, each an
 * even share of the tiles x superblocks steps, so no wave of tiles runs
 * part-empty; a tile cut between blocks is added up, in block order, by the
 * last of them.  0 means no workspace is needed for this shape.
 */
size_t kq_gemm_workspace_bytes(kq_format f, int64_t M, int64_t N, int64_t K);

/*
 * The least workspace kq_gemm / kq_gemm_grouped accept for this shape: the
 * activation image alone (about 2.14 bytes per activation).  With less than
 * kq_gemm_workspace_bytes, kq_gemm runs one block per output tile instead
 * of the split-tile schedule (same results up to float rounding order).
 */
size_t kq_gemm_min_workspace_bytes(kq_format f, int64_t M, int64_t N, int64_t K);

/*
 * Prefill GEMM ([kq-arc], "The pieces", kq v3: each weight panel is unpacked
 * once per block of tokens, so the unpack cost is shared by the whole token
 * block): y [M][N] = the fold above for every
 * token row m of a.
 *   a          device Q8_K planes of M rows
 *   y          device float32 [M][N]
 *   workspace  device, >= kq_gemm_min_workspace_bytes(f, M, N, K) bytes
 *              (kq_gemm_workspace_bytes for the split-tile schedule),
 *              256-byte aligned (may be NULL when that size is 0)
 * Calls that share a workspace must not overlap on the GPU.
 * Errors: KQ_ERR_ARG, KQ_ERR_FORMAT, KQ_ERR_ALIGN, KQ_ERR_WORKSPACE,
 * KQ_ERR_LAUNCH.  M == 0 is a no-op.
 */
int kq_gemm(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a,
            int64_t M, float *y, void *workspace, size_t workspace_bytes, cudaStream_t s);

/*
 * Grouped (MoE) GEMM ([kq-arc], k4 and k5/k6 kq-v2 commits: the grouped MoE
 * prefill, ffn_moe_prefill_grouped, reads its expert rows from one Q8_K
 * image of the token batch): rows of a are grouped by
 * expert; rows row_offsets[e] .. row_offsets[e+1]-1 use expert e's weights.
 *   packed       device, E expert images back to back, each
 *                kq_repack_bytes(f, N, K) bytes (expert e at
 *                packed + e * kq_repack_bytes(f, N, K))
 *   row_offsets  device int32 [E+1], non-decreasing, row_offsets[0] = 0,
 *                row_offsets[E] = M_total (not checked on the host: the
 *                kernels clamp every range to [0, M_total])
 *   a            device Q8_K planes of M_total rows
 *   y            device float32 [M_total][N]
 *   workspace    as for kq_gemm with M = M_total
 * Errors as kq_gemm.
 */
int kq_gemm_grouped(kq_format f, const void *packed, int64_t E, const int32_t *row_offsets,
                    int64_t N, int64_t K, kq_q8k_const a, int64_t M_total, float *y,
                    void *workspace, size_t workspace_bytes, cudaStream_t s);

/*
 * MoE decode, fused: M token rows routed to experts (rows grouped by expert),
 * quantized to Q8_K inside the kernel (bit-identical to kq_quantize_q8k) and
 * multiplied by their experts' matrices of n_sets weight sets that share the
 * rows (gate and up, say) in one launch: the decode GEMV over every row's
 * expert, its weights streamed once.  It is the page's fused decode chain
 * ([kq-arc], "The pieces": chain regrain) for the grouped MoE form; there is
 * no counterpart of the multi-set call in the pages.
 *   packed[s]    device: the E expert images of set s back to back, expert e
 *                at packed[s] + e * kq_repack_bytes(f, N[s], K), 256-byte aligned
 *   N[s]         rows of set s's expert matrices (>= 1)
 *   row_offsets  device int32 [E+1], as for kq_gemm_grouped (clamped to [0, M])
 *   x            device float32 [M][K] row-major, 16-byte aligned, finite
 *   y[s]         device float32 [M][N[s]]; a row that no expert range holds is
 *                left as it was
 * Limits: 1 <= n_sets <= 4, 1 <= n_sets * M <= 16, K % 256 == 0, K <= 40960
 * and the M staged rows within the kernel's shared memory (M * (K + K/8 +
 * K/64) plus two 16-row items per warp at most 212 KB).
 * Errors: KQ_ERR_FORMAT, KQ_ERR_ARG (outside the limits, null), KQ_ERR_ALIGN,
 * KQ_ERR_LAUNCH.  M == 0 is a no-op.
 */
int kq_gemv_grouped_fused(kq_format f, int n_sets, const void *const *packed, const int64_t *N, int64_t K, int64_t E,
                          const int32_t *row_offsets, const float *x, int64_t M, float *const *y, cudaStream_t s);

/*
 * Test hook: the int32 partials of the fold, per (token, row, superblock),
 * computed by the same device code the GEMV runs.
 *   isum, msum  device int32 [M][N][K/256]; for Q6_K isum = iacc - 32*bacc
 *               and msum = 0 ([kq-arc], k5/k6 kq-v2 commit).
 */
int kq_debug_partials(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a,
                      int64_t M, int32_t *isum, int32_t *msum, cudaStream_t s);

/*
 * Test hook: the same int32 partials from the small-batch passes' integer
 * warp-MMA fold (the 8-token passes of kq_gemm / kq_gemv_fused_batch for
 * Q4_K and Q6_K; the other passes fold with the GEMV's dp4a code above),
 * run by the same device functions on M <= 8 token rows ([kq-arc], kq v3
 * panel-scratch commit: every tile form must equal the GEMV bit for bit).
 *   f           KQ_Q4_K or KQ_Q6_K (KQ_Q5_K: KQ_ERR_ARG, it has no such fold)
 *   isum, msum  device int32 [M][N][K/256], as kq_debug_partials
 * Errors: KQ_ERR_FORMAT, KQ_ERR_ARG (M > 8, null), KQ_ERR_ALIGN, KQ_ERR_LAUNCH.
 */
int kq_debug_batch_partials(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M,
                            int32_t *isum, int32_t *msum, cudaStream_t s);

/*
 * Test hook: the same int32 partials from the tensor-core GEMM ([kq-arc],
 * kq v3 panel-scratch commit: the tile must equal the GEMV bit for bit,
 * unpack included).  It runs the kq_gemm / kq_gemm_grouped kernel with its
 * epilogue switched from the float fold to integers: each fp32 accumulator
 * unit the tensor pipe produced (an exact integer below 2^24) is converted
 * to int32 and the units of a superblock are added, so isum and msum are
 * what the GEMM's contraction computed, bit for bit.
 *   E, row_offsets  1 and NULL for the dense GEMM; else as kq_gemm_grouped
 *   M           token rows, >= 16 (the tensor-core path)
 *   isum, msum  device int32 [M][N][K/256]; for Q6_K isum = iacc - 32*bacc,
 *               msum = 0; rows outside every expert range are left 0
 *   workspace   as kq_gemm (kq_gemm_workspace_bytes(f, M, N, K) bytes)
 * Errors: KQ_ERR_FORMAT, KQ_ERR_ARG (M < 16, null, E > 1 without offsets, a
 * grouped shape the tensor-core kernel does not take), KQ_ERR_ALIGN,
 * KQ_ERR_WORKSPACE, KQ_ERR_LAUNCH.
 */
int kq_debug_gemm_partials(kq_format f, const void *packed, int64_t E, const int32_t *row_offsets, int64_t N,
                           int64_t K, kq_q8k_const a, int64_t M, int32_t *isum, int32_t *msum, void *workspace,
                           size_t workspace_bytes, cudaStream_t s);

/*
 * Test hook: decode the packed image back to stored quants and scales with
 * the device unpack helpers, to check the repack round trip.
 *   q     device int32 [N][K]        stored quant (Q6_K: 0..63, before -32)
 *   sc    device int32 [N][K/256][16] sub-scales (8 used for Q4_K/Q5_K)
 *   mn    device int32 [N][K/256][8]  sub-mins (0 for Q6_K)
 *   d     device float [N][K/256], dmin device float [N][K/256] (0 for Q6_K)
 */
int kq_debug_decode(kq_format f, const void *packed, int64_t N, int64_t K, int32_t *q,
                    int32_t *sc, int32_t *mn, float *d, float *dmin, cudaStream_t s);

/*
 * The Q8_0 rail ([kq-arc], chain-regrain commit: one activation image per
 * consumed form, the Q8_0 projections reading a Q8_0-form image; grouped-
 * prefill fix: the Q8_0 weights' fp16 scale plane).  Q8_0-form activations:
 * per 32 values of each row of x, amax = max|x|; amax == 0 gives d = 0 and
 * q = 0, else q = clamp(round_half_even(x * (127/amax)), -127, 127) in IEEE
 * fp32 and d = amax/127 (the Q8_K arithmetic, per 32).
 *   x   device float32 [M][K] row-major (K % 32 == 0), 16-byte aligned, finite
 *   d   device float32 [M][K/32], 4-byte aligned
 *   qs  device int8 [M][K], 16-byte aligned
 * Errors: KQ_ERR_ARG (null, M < 0, K % 32), KQ_ERR_ALIGN, KQ_ERR_LAUNCH.
 * M == 0 is a no-op.
 */
int kq_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *qs, cudaStream_t s);

/*
 * Q8_0 GEMM (prefill, any M >= 1): y[m][n] = sum over the 32-blocks b of
 * d_w(n, b) * d(m, b) * isum(m, n, b), isum the int32 dot of the block's
 * weight quants and token m's activation quants, one float fold per block
 * ([kq-arc], MoE prefill fix: the Q8_0 GEMMs read the Q8_0-form batch
 * image).  Each block's dot is one warp-level integer MMA, exact in int32.
 *   packed  device KQ_Q8_0 image from kq_repack (256-byte aligned)
 *   d       device float32 [M][K/32] from kq_quantize_q8_0, 16-byte aligned
 *   qs      device int8 [M][K], 16-byte aligned
 *   y       device float32 [M][N] row-major
 *   K       a positive multiple of 256
 * The result is independent of scheduling (fixed summation order).
 * Errors: KQ_ERR_ARG, KQ_ERR_ALIGN, KQ_ERR_LAUNCH.  M == 0 or N == 0 is a no-op.
 */
int kq_gemm_q8_0(const void *packed, int64_t N, int64_t K, const float *d, const int8_t *qs, int64_t M, float *y,
                 cudaStream_t s);

/*
 * Q8_0 GEMV (M = 1): y[n] = sum over the 32-blocks b of row n of
 * d_w(n, b) * d(b) * isum_b, isum_b the int32 dot of the block's weight and
 * activation quants (one float fold per block).  Reads every packed byte once.
 *   packed  device KQ_Q8_0 image from kq_repack (256-byte aligned)
 *   d, qs   one activation row from kq_quantize_q8_0 (K/32 floats, K int8;
 *           qs 16-byte aligned)
 *   y       device float32 [N]
 *   K       a positive multiple of 256, at most 40960
 * The result is independent of scheduling (fixed summation order).
 * Errors: KQ_ERR_ARG, KQ_ERR_ALIGN, KQ_ERR_LAUNCH.  N == 0 is a no-op.
 */
int kq_gemv_q8_0(const void *packed, int64_t N, int64_t K, const float *d, const int8_t *qs, float *y,
                 cudaStream_t s);

/*
 * kq_gemv_q8_0 with the quantize fused in ([kq-arc], "The pieces": the chain
 * regrain applied to the q8 rail): every block quantizes the fp32 row into its
 * shared memory bit-identically to kq_quantize_q8_0, so the result equals
 * kq_quantize_q8_0 + kq_gemv_q8_0 bit for bit, in one launch.
 *   x   device float32 [K], 16-byte aligned, finite
 * Other arguments, limits and errors as kq_gemv_q8_0.
 */
int kq_gemv_q8_0_fused(const void *packed, int64_t N, int64_t K, const float *x, float *y, cudaStream_t s);

/*
 * Test hook for failure detection: launches one block whose single bounded
 * mbarrier wait is never satisfied; after limit_ns nanoseconds the wait gives
 * up and records KQ_ERR_TIMEOUT in the device status word, as a stuck stage
 * of the GEMM or GEMV would, without any fault or hang.  kq_device_status
 * then returns KQ_ERR_TIMEOUT once (and clears it).
 * Errors: KQ_ERR_ARG for limit_ns == 0 or > 1e9 (one second); KQ_ERR_LAUNCH.
 */
int kq_debug_wait_timeout(uint64_t limit_ns, cudaStream_t s);

/*
 * Measurement hook: the int8 rate of the warp-level integer MMA
 * (mma.sync m16n8k32, s8 x s8 -> s32), the only integer tensor-core MMA on
 * sm_103a.  Launches `blocks` blocks of 8 warps; every warp issues iters x 8
 * independent MMAs of 16 x 8 x 32, i.e. blocks * 8 * iters * 8 * 8192 int8
 * operations (multiply and add counted separately).  Time it with events on
 * `s`.  All operands are ones, so every thread writes the checksum
 * 1024 * iters to out[block * 256 + thread].
 *   out   device int32 [blocks * 256]
 * Errors: KQ_ERR_ARG for blocks < 0, iters < 0 or a null out; KQ_ERR_LAUNCH.
 */
int kq_measure_mma_s8(int64_t blocks, int64_t iters, int32_t *out, cudaStream_t s);

/*
 * Transport, not part of the method: copy a step's input rows from pinned
 * host memory into device memory with a kernel in the stream's launch chain,
 * so that under KQ_LAUNCH_PDL the copy needs no copy engine and no
 * cross-stream event (either breaks the chain's early launch).  The kernel
 * reads src BEFORE its dependency wait and writes dst after it: src must
 * not be written by earlier kernels in the stream (host-produced data,
 * ready when the call is made), while dst may still be read by them.
 *   src    pinned host memory mapped into the device address space (page-
 *          locked by cudaHostAlloc or cudaHostRegister on a system with
 *          unified addressing), or device memory; 16-byte aligned
 *   dst    device memory, 16-byte aligned, not overlapping src
 *   bytes  a multiple of 16 (at most 2^40)
 * The outputs of the GEMV entry points may likewise be pinned host memory:
 * the kernels store the results there directly.
 * Errors: KQ_ERR_ARG (bytes, null), KQ_ERR_ALIGN, KQ_ERR_LAUNCH.
 */
int kq_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s);

/*
 * Launch options, process-wide (a plain atomic word; the new value applies
 * to launches enqueued after the call).  Returns the previous flags.
 *
 * KQ_LAUNCH_PDL: launch the kernels of kq_quantize_q8k, kq_gemv,
 *   kq_gemv_fused, kq_gemm, kq_gemm_grouped and kq_gemm_noalloc with
 *   programmatic dependent launch, so that each may start while the previous
 *   kernel in the stream is still running.  They wait (griddepcontrol.wait)
 *   for the previous kernels to complete before reading activations, scales
 *   or expert offsets and before writing any output, except that the GEMV
 *   and GEMM kernels read the packed weight image BEFORE that wait, to
 *   overlap their weight stream (GEMM: the first weight unpack) with the
 *   previous kernel.  With the flag set, a packed image must not be written
 *   by work that may still be running on the stream when one of them is
 *   enqueued (synchronise, or wait on an event recorded after kq_repack,
 *   before the first use).  Default: off.
 */
#define KQ_LAUNCH_PDL 1u
/*
 * KQ_LAUNCH_GEMV_SPLIT: a decode GEMV given a workspace always gives every SM
 * an even share of the superblocks, cutting row groups between blocks
 * wherever the shares fall.  Default (off): it cuts only where taking whole
 * row groups would leave the busiest warp three or more superblocks above an
 * even share, since the exchange at a cut costs about as much as folding a
 * few superblocks.  The results differ between the two only in float
 * rounding.
 */
#define KQ_LAUNCH_GEMV_SPLIT 2u
/*
 * KQ_LAUNCH_GEMM_SPLIT: a dense kq_gemm given kq_gemm_workspace_bytes always
 * runs the split-tile schedule (one block per SM, an even share of the
 * tiles x superblocks steps each, tiles cut between blocks finished from
 * their partial tiles in block order).  Without it the schedule is chosen
 * by shape: where a block per tile would leave the last wave of tiles
 * mostly empty and every block still gets 16 superblock steps or more.
 * Results of the two schedules differ only in float rounding order.
 */
#define KQ_LAUNCH_GEMM_SPLIT 4u
unsigned kq_set_launch_flags(unsigned flags);
unsigned kq_get_launch_flags(void);

/*
 * Prefill GEMM without any allocation by anyone: kq_gemm with its scratch
 * (the fp16 activation image and the transposed scales) held in a fixed
 * array that the library reserves in device memory on every GPU that loads
 * it, KQ_NOALLOC_SCRATCH_BYTES (32 MiB), kept until the process exits.  The
 * source pages have no counterpart of this entry point.
 *
 * It is for callers that cannot call cudaMalloc or hand the library a
 * workspace: for example a serving runtime that plans its whole device
 * memory budget at start-up and forbids allocation on the request path, a
 * latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation, or plain C host code that only receives device pointers
 * for its inputs and outputs and has no allocator of its own.  The caller
 * still passes the inputs and the output, as for kq_gemm.
 *
 *   arguments  as kq_gemm, without workspace / workspace_bytes
 * Limits and behaviour:
 *   - The scratch needed, kq_gemm_min_workspace_bytes(f, M, N, K), must
 *     not exceed KQ_NOALLOC_SCRATCH_BYTES; larger problems return
 *     KQ_ERR_TOO_LARGE before anything is enqueued.  The scratch is about
 *     2.14 bytes per activation, so M*K up to about 15.6 million
 *     activations fit (e.g. 512 tokens x K = 30464; K = 30720 is refused).
 *     When kq_gemm_workspace_bytes(f, M, N, K) fits as well, the call runs
 *     the split-tile schedule, else one block per output tile.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after a cudaDeviceReset the next call would reuse the old
 *     one, so do not call it on a device that has been reset.
 *   - Every call on a device shares the one array, and the array keeps what
 *     the last call wrote; each call rewrites every scratch byte it reads,
 *     so nothing needs clearing.  Calls whose work may overlap on the GPU
 *     (different streams, no ordering between them) race on the array and
 *     must not be issued; calls on one stream are ordered and safe.
 *   - Errors as kq_gemm, plus KQ_ERR_TOO_LARGE; KQ_ERR_LAUNCH if the address
 *     lookup fails.
 */
#define KQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int kq_gemm_noalloc(kq_format f, const void *packed, int64_t N, int64_t K, kq_q8k_const a, int64_t M,
                    float *y, cudaStream_t s);

/*
 * Synchronise stream s and return the device status word of the library's
 * bounded waits on the current device (KQ_OK, or KQ_ERR_TIMEOUT if a kernel
 * gave up waiting), then clear it.  Returns KQ_ERR_LAUNCH if the
 * synchronisation itself failed.
 */
int kq_device_status(cudaStream_t s);

#ifdef __cplusplus
}
#endif
#endif /* KQ_H */
