/*
 * kq_oracle.c - plain scalar CPU oracle for the K-quant x Q8_K products.
 *
 * TEST INFRASTRUCTURE ONLY (see kq_oracle.h): loaded by the tests, the smoke
 * check and the benchmark's CPU-baseline leg, never by the product path.
 *
 * [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
 * kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
 *
 * Written for the reader, not for speed: one superblock at a time, every
 * element decoded into a plain int array first, then the sums of the fold
 * in the order the page states them.  Build with -ffp-contract=off and no
 * fast-math so that the Q8_K quantizer's fp32 steps are the IEEE operations
 * written here.
 */
#include "kq_oracle.h"

#include <math.h>
#include <fenv.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256

int ko_block_bytes(int fmt) {
    switch (fmt) {
    case KO_Q4_K: return 144; /* 2+2+12 scale block + 128 B of 4-bit quants */
    case KO_Q5_K: return 176; /* same scale block + 32 B high bits + 128 B    */
    case KO_Q6_K: return 210; /* 128 B low nibbles + 64 B 2-bit highs + 16 + 2 */
    default: return 0;
    }
}

/* IEEE binary16 -> double, from the definition of the encoding:
 * sign bit, 5-bit exponent with bias 15, 10-bit fraction. */
static double half_bits_to_double(uint16_t h) {
    int sign = h >> 15;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);              /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), expo - 25); /* 1.frac * 2^(expo-15) */
    return sign ? -v : v;
}

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* The 12-byte 6-bit scale/min packing of Q4_K and Q5_K ([kq-arc], k4 kq-v2
 * commit: fp16 d and dmin, then 12 bytes of 6-bit fields; the k5/k6 commit
 * says Q5_K uses the very same scale block).  Reading (GGUF): bytes 0..3 hold the low
 * 6 bits of scales 0..3, bytes 4..7 the low 6 bits of mins 0..3; bytes 8..11
 * hold scales 4..7 (low nibble) and mins 4..7 (high nibble) as their low 4
 * bits, whose top 2 bits sit in bits 6..7 of bytes 0..3 (scales) and 4..7
 * (mins). */
static void unpack_scale_min_12(const uint8_t *s, int32_t *sc, int32_t *mn) {
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        mn[j] = s[j + 4] & 63;
    }
    for (int j = 4; j < 8; ++j) {
        sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

int ko_decode(int fmt, const uint8_t *b, double *d, double *dmin,
              int32_t *sc, int32_t *mn, int32_t *q) {
    if (fmt == KO_Q4_K || fmt == KO_Q5_K) {
        /* Q4_K: d f16 | dmin f16 | scales[12] | qs[128]
         * Q5_K: d f16 | dmin f16 | scales[12] | qh[32] | qs[128]
         * Element 64c+l (c < 4, l < 32) is the low nibble of qs[32c+l] and
         * belongs to sub-block 2c; element 64c+32+l is its high nibble, in
         * sub-block 2c+1.  Q5_K adds bit 2c (resp. 2c+1) of qh[l] as value 16
         * (k5/k6 commit: Q5_K differs from Q4_K only by OR-ing in that high
         * bit while walking the quants). */
        *d = half_bits_to_double(le16(b));
        *dmin = half_bits_to_double(le16(b + 2));
        unpack_scale_min_12(b + 4, sc, mn);
        const uint8_t *qh = b + 16;
        const uint8_t *qs = (fmt == KO_Q4_K) ? b + 16 : b + 48;
        for (int c = 0; c < 4; ++c) {
            for (int l = 0; l < 32; ++l) {
                int lo = qs[32 * c + l] & 15;
                int hi = qs[32 * c + l] >> 4;
                if (fmt == KO_Q5_K) {
                    lo |= ((qh[l] >> (2 * c)) & 1) << 4;
                    hi |= ((qh[l] >> (2 * c + 1)) & 1) << 4;
                }
                q[64 * c + l] = lo;
                q[64 * c + 32 + l] = hi;
            }
        }
        return 8;
    }
    if (fmt == KO_Q6_K) {
        /* Q6_K: ql[128] | qh[64] | scales[16] int8 | d f16.
         * Half h in {0,1} owns elements 128h..128h+127 and uses ql+64h,
         * qh+32h.  For l < 32:
         *   128h+l    : low nibble of ql[l]    | bits 0..1 of qh[l] << 4
         *   128h+32+l : low nibble of ql[l+32] | bits 2..3 of qh[l] << 4
         *   128h+64+l : high nibble of ql[l]   | bits 4..5 of qh[l] << 4
         *   128h+96+l : high nibble of ql[l+32]| bits 6..7 of qh[l] << 4
         * Element e is scaled by the signed sub-scale scales[e/16]
         * (k5/k6 commit: one signed sub-scale per 16 weights); its weight
         * is q-32. */
        const uint8_t *ql = b;
        const uint8_t *qh = b + 128;
        const int8_t *s = (const int8_t *)(b + 192);
        *d = half_bits_to_double(le16(b + 208));
        *dmin = 0.0;
        for (int i = 0; i < 16; ++i) sc[i] = s[i];
        for (int j = 0; j < 8; ++j) mn[j] = 0;
        for (int h = 0; h < 2; ++h) {
            const uint8_t *L = ql + 64 * h;
            const uint8_t *H = qh + 32 * h;
            for (int l = 0; l < 32; ++l) {
                q[128 * h + l]      = (L[l] & 15)      | (((H[l] >> 0) & 3) << 4);
                q[128 * h + 32 + l] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);
                q[128 * h + 64 + l] = (L[l] >> 4)      | (((H[l] >> 4) & 3) << 4);
                q[128 * h + 96 + l] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
            }
        }
        return 16;
    }
    return -1;
}

int ko_dequant(int fmt, const uint8_t *blk, double *w) {
    double d, dmin;
    int32_t sc[16], mn[8], q[QK];
    int nsub = ko_decode(fmt, blk, &d, &dmin, sc, mn, q);
    if (nsub < 0) return -1;
    int width = QK / nsub;
    for (int e = 0; e < QK; ++e) {
        int j = e / width;
        if (fmt == KO_Q6_K)
            w[e] = d * sc[j] * (q[e] - 32);
        else
            w[e] = d * sc[j] * q[e] - dmin * mn[j];
    }
    return 0;
}

/* Q8_K quantization ([kq-arc], k4 kq-v2 commit: a single fp32 scale for each
 * 256-value block plus the sum of every 16 quants).  The page gives no
 * formula; the reading:
 *   amax = max |x| over the block
 *   amax == 0  ->  d8 = 0, every q = 0
 *   otherwise  ->  iscale = 127/amax (fp32 division),
 *                  q = clamp(round_half_even(x * iscale), -127, 127),
 *                  d8 = amax/127 (fp32 division)
 *   bsums[i] = sum of q over elements 16i..16i+15.
 * Inputs are assumed finite. */
void ko_quantize_q8k(const float *x, int64_t M, int64_t K,
                     float *d8, int8_t *q, int16_t *bsums) {
    const int64_t nsb = K / QK;
    const int saved_round = fegetround();
    fesetround(FE_TONEAREST);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t s = 0; s < nsb; ++s) {
            const float *xb = x + m * K + s * QK;
            int8_t *qb = q + m * K + s * QK;
            int16_t *bb = bsums + (m * nsb + s) * 16;
            float amax = 0.0f;
            for (int j = 0; j < QK; ++j) {
                float ax = fabsf(xb[j]);
                if (ax > amax) amax = ax;
            }
            if (amax == 0.0f) {
                d8[m * nsb + s] = 0.0f;
                memset(qb, 0, QK);
                memset(bb, 0, 16 * sizeof(int16_t));
                continue;
            }
            volatile float iscale = 127.0f / amax;
            for (int j = 0; j < QK; ++j) {
                volatile float t = xb[j] * iscale;
                long v = lrintf(t);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
                qb[j] = (int8_t)v;
            }
            d8[m * nsb + s] = amax / 127.0f;
            for (int i = 0; i < 16; ++i) {
                int sum = 0;
                for (int k = 0; k < 16; ++k) sum += qb[16 * i + k];
                bb[i] = (int16_t)sum;
            }
        }
    }
    fesetround(saved_round);
}

/* The integer fold of one superblock ([kq-arc], k4 kq-v2 commit: per
 * superblock, the integer sub-scales multiply int32 dot products and the
 * sub-mins multiply the activation bsums, both accumulated in int32;
 * k5/k6 commit for Q6_K: each signed sub-scale multiplies both the int32
 * dot of its 16 stored quants and the bsum of the same 16 activations,
 * giving iacc and bacc, and the superblock closes as float(iacc - 32*bacc)
 * times d*d8).  All sums are int32; the page bounds |iacc| and |32*bacc|
 * below 2^28. */
void ko_partials_block(int fmt, const uint8_t *blk, const int8_t *a8,
                       const int16_t *bs, int32_t *isum, int32_t *msum) {
    double d, dmin;
    int32_t sc[16], mn[8], q[QK];
    int nsub = ko_decode(fmt, blk, &d, &dmin, sc, mn, q);
    if (nsub == 8) {
        int32_t is = 0, ms = 0;
        for (int j = 0; j < 8; ++j) {
            int32_t dot = 0;
            for (int k = 0; k < 32; ++k) dot += q[32 * j + k] * (int32_t)a8[32 * j + k];
            is += sc[j] * dot;
            ms += mn[j] * ((int32_t)bs[2 * j] + (int32_t)bs[2 * j + 1]);
        }
        *isum = is;
        *msum = ms;
    } else if (nsub == 16) {
        int32_t iacc = 0, bacc = 0;
        for (int i = 0; i < 16; ++i) {
            int32_t dot = 0;
            for (int k = 0; k < 16; ++k) dot += q[16 * i + k] * (int32_t)a8[16 * i + k];
            iacc += sc[i] * dot;
            bacc += sc[i] * (int32_t)bs[i];
        }
        *isum = iacc - 32 * bacc;
        *msum = 0;
    } else {
        *isum = 0;
        *msum = 0;
    }
}

int ko_partials(int fmt, const uint8_t *disk, int64_t N, int64_t K,
                const int8_t *a8, const int16_t *bs, int64_t M,
                int32_t *isum, int32_t *msum) {
    const int bb = ko_block_bytes(fmt);
    if (!bb || K % QK || N < 0 || M < 0) return -1;
    const int64_t nsb = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t s = 0; s < nsb; ++s) {
                int64_t o = (m * N + n) * nsb + s;
                ko_partials_block(fmt, disk + (n * nsb + s) * bb, a8 + m * K + s * QK,
                                  bs + (m * nsb + s) * 16, &isum[o], &msum[o]);
            }
    return 0;
}

/* One output: the fold closed once per superblock ([kq-arc], "The pieces",
 * kq v2 bullet: a single float fold per superblock), d*d8*isum -
 * dmin*d8*msum, summed over
 * the superblocks of the row.  Evaluated in double: d (fp16) times d8 (fp32)
 * is exact in double, so this is the quantized product to ~1e-16. */
double ko_dot(int fmt, const uint8_t *row, int64_t nsb, const float *d8,
              const int8_t *a8, const int16_t *bs) {
    const int bb = ko_block_bytes(fmt);
    double acc = 0.0;
    for (int64_t s = 0; s < nsb; ++s) {
        const uint8_t *blk = row + s * bb;
        double d, dmin;
        int32_t sc[16], mn[8], q[QK];
        ko_decode(fmt, blk, &d, &dmin, sc, mn, q);
        int32_t isum, msum;
        ko_partials_block(fmt, blk, a8 + s * QK, bs + s * 16, &isum, &msum);
        acc += d * (double)d8[s] * (double)isum - dmin * (double)d8[s] * (double)msum;
    }
    return acc;
}

int ko_gemm(int fmt, const uint8_t *disk, int64_t N, int64_t K,
            const float *d8, const int8_t *a8, const int16_t *bs, int64_t M,
            const int64_t *tok_idx, int64_t ntok,
            const int64_t *n_idx, int64_t nn, double *Y) {
    const int bb = ko_block_bytes(fmt);
    if (!bb || K % QK || N < 0 || M < 0) return -1;
    const int64_t nsb = K / QK;
    if (!tok_idx) ntok = M;
    if (!n_idx) nn = N;
    for (int64_t i = 0; i < ntok; ++i) {
        int64_t t = tok_idx ? tok_idx[i] : i;
        if (t < 0 || t >= M) return -1;
    }
    for (int64_t j = 0; j < nn; ++j) {
        int64_t n = n_idx ? n_idx[j] : j;
        if (n < 0 || n >= N) return -1;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t j = 0; j < nn; ++j) {
        int64_t n = n_idx ? n_idx[j] : j;
        for (int64_t i = 0; i < ntok; ++i) {
            int64_t t = tok_idx ? tok_idx[i] : i;
            Y[i * nn + j] = ko_dot(fmt, disk + n * nsb * bb, nsb, d8 + t * nsb,
                                   a8 + t * K, bs + t * nsb * 16);
        }
    }
    return 0;
}

double ko_bruteforce_dot(int fmt, const uint8_t *row, int64_t nsb,
                         const float *d8, const int8_t *a8) {
    const int bb = ko_block_bytes(fmt);
    double w[QK];
    double acc = 0.0;
    for (int64_t s = 0; s < nsb; ++s) {
        ko_dequant(fmt, row + s * bb, w);
        for (int e = 0; e < QK; ++e)
            acc += w[e] * ((double)d8[s] * (double)a8[s * QK + e]);
    }
    return acc;
}

/* ---- Q8_0 ---------------------------------------------------------------- */

void ko_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *q) {
    const int64_t nb = K / KO_QK8_0;
    const int saved_round = fegetround();
    fesetround(FE_TONEAREST);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + m * K + b * KO_QK8_0;
            int8_t *qb = q + m * K + b * KO_QK8_0;
            float amax = 0.0f;
            for (int j = 0; j < KO_QK8_0; ++j) {
                float ax = fabsf(xb[j]);
                if (ax > amax) amax = ax;
            }
            if (amax == 0.0f) {
                d[m * nb + b] = 0.0f;
                memset(qb, 0, KO_QK8_0);
                continue;
            }
            volatile float iscale = 127.0f / amax;
            for (int j = 0; j < KO_QK8_0; ++j) {
                volatile float t = xb[j] * iscale;
                long v = lrintf(t);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
                qb[j] = (int8_t)v;
            }
            d[m * nb + b] = amax / 127.0f;
        }
    }
    fesetround(saved_round);
}

/* One output: the integer dot of each 32-block, closed by one float fold
 * per block (d_w * d_a * isum), summed over the row in double.  d_w (fp16)
 * times d_a (fp32) is exact in double. */
static double q8_0_dot(const uint8_t *row, int64_t nb, const float *d_a, const int8_t *q_a) {
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row + b * KO_Q8_0_BLOCK;
        const double dw = half_bits_to_double(le16(blk));
        int32_t isum = 0;
        for (int k = 0; k < KO_QK8_0; ++k) isum += (int32_t)(int8_t)blk[2 + k] * (int32_t)q_a[b * KO_QK8_0 + k];
        acc += dw * (double)d_a[b] * (double)isum;
    }
    return acc;
}

int ko_gemv_q8_0(const uint8_t *disk, int64_t N, int64_t K, const float *d_a,
                 const int8_t *q_a, int64_t M, double *Y) {
    if (K % KO_QK8_0 || N < 0 || M < 0) return -1;
    const int64_t nb = K / KO_QK8_0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            Y[m * N + n] = q8_0_dot(disk + n * nb * KO_Q8_0_BLOCK, nb, d_a + m * nb, q_a + m * K);
    return 0;
}

/* The integer dot of every 32-block, per (activation row m, weight row n,
 * block b): isum[(m * N + n) * nb + b] = sum_k q_w * q_a over the block. */
int ko_partials_q8_0(const uint8_t *disk, int64_t N, int64_t K, const int8_t *q_a, int64_t M, int32_t *isum) {
    if (K % KO_QK8_0 || N < 0 || M < 0) return -1;
    const int64_t nb = K / KO_QK8_0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = disk + (n * nb + b) * KO_Q8_0_BLOCK;
                int32_t acc = 0;
                for (int k = 0; k < KO_QK8_0; ++k) acc += (int32_t)(int8_t)blk[2 + k] * (int32_t)q_a[m * K + b * KO_QK8_0 + k];
                isum[(m * N + n) * nb + b] = acc;
            }
    return 0;
}

double ko_bruteforce_q8_0(const uint8_t *row, int64_t nblk, const float *d_a, const int8_t *q_a) {
    double acc = 0.0;
    for (int64_t b = 0; b < nblk; ++b) {
        const uint8_t *blk = row + b * KO_Q8_0_BLOCK;
        const double dw = half_bits_to_double(le16(blk));
        for (int k = 0; k < KO_QK8_0; ++k) {
            const double w = dw * (double)(int8_t)blk[2 + k];
            const double a = (double)d_a[b] * (double)q_a[b * KO_QK8_0 + k];
            acc += w * a;
        }
    }
    return acc;
}

int ko_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ko_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
