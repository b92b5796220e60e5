/*
 * kq_oracle.h - plain scalar CPU oracle for the K-quant x Q8_K products.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the correctness reference for
 * the CUDA path; it shares no code, header, table or constant with it.  Only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  The product path never calls it and has no CPU fallback.
 *
 * Source of the method, cited as [kq-arc]: the page "dasLLAMA: K-quant
 * kernel arc - kq v2 integer folds, kq v3 panel-scratch tiles, chain
 * regrain, parity gates" (daScript pull request #3450): its section
 * "The pieces" (kq v2 bullet) and its k4 and k5/k6 kq-v2 commit messages.
 *
 * Formats.  The page names the blocks (Q4_K, Q5_K, Q6_K, Q8_K) and their
 * 256-weight superblocks; it says the Q4_K/Q5_K scale block is an fp16 d
 * and dmin followed by 12 bytes of packed 6-bit sub-scales and sub-mins,
 * that Q6_K carries signed 8-bit sub-scales (one per 16 weights) and an
 * fp16 d, and that a Q8_K activation block has one fp32 scale per 256
 * values plus a sum per 16.  It prints no bit layout; this oracle reads
 * the layouts as the public GGUF block formats (byte order given in
 * kq_oracle.c beside each decoder).
 *
 * All pointers are host pointers.  Sizes are 64-bit.
 */
#ifndef KQ_ORACLE_H
#define KQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { KO_Q4_K = 1, KO_Q5_K = 2, KO_Q6_K = 3 };

/* Bytes of one 256-weight superblock on disk: 144, 176, 210 (0 if unknown). */
int ko_block_bytes(int fmt);

/* Decode one disk superblock.
 *   d, dmin : super-scales as doubles (dmin = 0 for Q6_K)
 *   sc      : sub-scales, 8 (Q4_K/Q5_K, one per 32 weights) or 16 (Q6_K,
 *             signed, one per 16 weights)
 *   mn      : 8 sub-mins (Q4_K/Q5_K; zeros for Q6_K)
 *   q       : 256 stored quant values (Q4_K 0..15, Q5_K 0..31, Q6_K 0..63;
 *             the Q6_K weight uses q - 32)
 * Returns the number of sub-scales (8 or 16), or -1 for an unknown format. */
int ko_decode(int fmt, const uint8_t *blk, double *d, double *dmin,
              int32_t *sc, int32_t *mn, int32_t *q);

/* Dequantize one superblock to 256 doubles: d*sc*q - dmin*m (Q4_K/Q5_K),
 * d*sc*(q-32) (Q6_K).  Returns 0, or -1 for an unknown format. */
int ko_dequant(int fmt, const uint8_t *blk, double *w);

/* Q8_K quantization of M rows of K floats (K % 256 == 0), row-major.
 * Per 256-block: d8 (one float), q (256 int8), bsums (16 int16).
 * Output planes are row-major [M][K/256], [M][K], [M][K/16]. */
void ko_quantize_q8k(const float *x, int64_t M, int64_t K,
                     float *d8, int8_t *q, int16_t *bsums);

/* Integer partials of one (weight superblock, activation superblock) pair.
 * Q4_K/Q5_K: isum = sum_j sc_j * dot32_j(q, a8), msum = sum_j m_j * (bs_2j + bs_2j+1)
 * Q6_K     : isum = iacc - 32*bacc with iacc = sum_i sc_i * dot16_i(q, a8),
 *            bacc = sum_i sc_i * bs_i; msum = 0. */
void ko_partials_block(int fmt, const uint8_t *blk, const int8_t *a8,
                       const int16_t *bs, int32_t *isum, int32_t *msum);

/* Partials for a whole problem: isum/msum are [M][N][K/256] row-major. */
int ko_partials(int fmt, const uint8_t *disk, int64_t N, int64_t K,
                const int8_t *a8, const int16_t *bs, int64_t M,
                int32_t *isum, int32_t *msum);

/* One output Y[m, n] = sum_sb d*d8*isum - dmin*d8*msum, evaluated in double.
 * row points at the N-row's K/256 consecutive disk superblocks; d8/a8/bs
 * point at the token's activation planes. */
double ko_dot(int fmt, const uint8_t *row, int64_t nsb, const float *d8,
              const int8_t *a8, const int16_t *bs);

/* Y[i][j] = ko_dot(weight row n_idx[j], token tok_idx[i]) for the selected
 * tokens and rows (both index lists may be NULL, meaning "all").
 * Y is [ntok][nn] row-major.  Parallel over rows with OpenMP when built
 * with it.  Returns 0, or -1 on a bad argument. */
int ko_gemm(int fmt, const uint8_t *disk, int64_t N, int64_t K,
            const float *d8, const int8_t *a8, const int16_t *bs, int64_t M,
            const int64_t *tok_idx, int64_t ntok,
            const int64_t *n_idx, int64_t nn, double *Y);

/* Brute force: dequantize the weight row and the activation (d8*q8) to
 * double and take the plain dot product.  Independent of the fold. */
double ko_bruteforce_dot(int fmt, const uint8_t *row, int64_t nsb,
                         const float *d8, const int8_t *a8);

/* ---- Q8_0 (the pages' "q8 rail": Q8_0 weights read with Q8_0-form
 * activations, one activation image per consumed form; [kq-arc], the
 * chain-regrain commit and the grouped-prefill fix of the MoE page).
 * A block holds 32 values: on disk an fp16 d then 32 int8 q (34 bytes,
 * the public GGUF block), weight = d * q.  The activation form has one
 * fp32 scale per 32 values, quantized like Q8_K but per 32:
 * d = amax / 127, q = clamp(round_half_even(x * (127 / amax)), -127, 127),
 * amax == 0 giving d = 0 and q = 0. */
enum { KO_Q8_0_BLOCK = 34, KO_QK8_0 = 32 };

/* Q8_0 activations of M rows of K floats (K % 32 == 0): d [M][K/32],
 * q [M][K], row-major. */
void ko_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *q);

/* Y[m][n] = sum over the K/32 blocks b of d_w(n,b) * d_a(m,b) * isum, with
 * isum = sum_k q_w * q_a in int32 and the sum over blocks in double.
 * disk is [N][K/32][34]; d_a / q_a are the activation planes of M rows.
 * Returns 0, or -1 on a bad argument. */
int ko_gemv_q8_0(const uint8_t *disk, int64_t N, int64_t K, const float *d_a,
                 const int8_t *q_a, int64_t M, double *Y);

/* Brute force for one row and one activation row: both dequantized to
 * double (d * q), plain dot product.  Independent of the fold. */
/* Per-block int32 dots of Q8_0 weights [N][K/32] and M activation rows:
 * isum [M][N][K/32].  Returns 0, or -1 for bad sizes. */
int ko_partials_q8_0(const uint8_t *disk, int64_t N, int64_t K, const int8_t *q_a, int64_t M, int32_t *isum);
double ko_bruteforce_q8_0(const uint8_t *row, int64_t nblk, const float *d_a,
                          const int8_t *q_a);

/* Threads the OpenMP loops use (1 without OpenMP). */
int ko_num_threads(void);
void ko_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
