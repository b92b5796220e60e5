// kq_mv.cu - the CUDA-core small-token-count product (a group of up to 8
// tokens per pass over each weight superblock) and its MoE grouped form,
// used below the tensor-core GEMM's token threshold and for K beyond the
// decode GEMV's shared-memory row; plus the packed-decode test hook.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
//
// Work split: a 256-thread block = 8 warps = WR row groups x WK superblock
// slices (WR * WK = 8).  A warp owns 8 rows
// (one per quad, see kq_device.cuh) and walks its slice of superblocks,
// loading the next superblock's weights before folding the current one.
// Per superblock the quad's lanes add their int32 partials with two xor
// shuffles and fold once in fp32: acc += d*d8*isum - dmin*d8*msum (Q6_K:
// acc += d*d8*(iacc - 32*bacc)) ([kq-arc], "The pieces": a single float fold
// per superblock).  Slices of one row are summed through shared memory.
#include "kq_internal.h"

#include <algorithm>

namespace kq {

struct MvParams {
    const uint8_t *packed;   // expert 0 (or the only matrix)
    uint64_t expert_bytes;   // stride between experts' images
    int64_t N, nsb, K;
    const float *d8;
    const int8_t *qs;
    const int16_t *bs;
    int64_t M;                // token rows (total)
    const int32_t *offsets;   // [E+1] for grouped, nullptr for dense
    float *y;
    int wk;                   // superblock slices per row group (1, 2, 4, 8)
};

template <int F, int TOK>
__global__ void __launch_bounds__(256) mv_kernel(const MvParams p) {
    __shared__ float red[8][TOK][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wk = p.wk;
    const int kw = warp % wk, rg = warp / wk;
    const int rows_per_block = 8 * (8 / wk);
    const int r8 = lane >> 2, c = lane & 3;
    const int64_t n = (int64_t)blockIdx.x * rows_per_block + rg * 8 + r8;
    const int64_t nc = n < p.N ? n : p.N - 1;

    // expert and its token range
    const int e = blockIdx.z;
    int64_t t_begin = 0, t_end = p.M;
    if (p.offsets) {
        const int64_t o0 = p.offsets[e], o1 = p.offsets[e + 1];
        t_begin = o0 < 0 ? 0 : (o0 > p.M ? p.M : o0);
        t_end = o1 < t_begin ? t_begin : (o1 > p.M ? p.M : o1);
    }
    const Planes P = make_planes(F, p.packed + (uint64_t)e * p.expert_bytes, p.N, p.nsb);

    const int64_t s_begin = kw * p.nsb / wk, s_end = (kw + 1) * p.nsb / wk;
    using W = typename WRegs<F>::T;

    for (int64_t t0 = t_begin + (int64_t)blockIdx.y * TOK; t0 < t_end; t0 += (int64_t)gridDim.y * TOK) {
        const int ntok = (t_end - t0) < TOK ? (int)(t_end - t0) : TOK;
        float acc[TOK];
#pragma unroll
        for (int t = 0; t < TOK; ++t) acc[t] = 0.0f;

        W cur, nxt;
        if (s_begin < s_end) load_w(cur, P, nc, s_begin, p.nsb, c);
        for (int64_t sb = s_begin; sb < s_end; ++sb) {
            if (sb + 1 < s_end) load_w(nxt, P, nc, sb + 1, p.nsb, c);
            LaneQ L;
            decode_lane(cur, c, L);
#pragma unroll
            for (int t = 0; t < TOK; ++t) {
                if (t < ntok) {
                    const int64_t tok = t0 + t;
                    int isum, msum;
                    lane_partials<F>(L, p.qs + tok * p.K + sb * QK, p.bs + (tok * p.nsb + sb) * 16, c, isum,
                                     msum);
                    isum = quad_sum(isum);
                    const float d8 = __ldg(p.d8 + tok * p.nsb + sb);
                    if constexpr (F == FMT_Q6_K) {
                        acc[t] = fmaf(L.d * d8, static_cast<float>(isum), acc[t]);
                    } else {
                        msum = quad_sum(msum);
                        acc[t] = fmaf(L.d * d8, static_cast<float>(isum), acc[t]);
                        acc[t] = fmaf(-(L.dmin * d8), static_cast<float>(msum), acc[t]);
                    }
                }
            }
            cur = nxt;
        }

        if (wk == 1) {
            if (c == 0 && n < p.N) {
#pragma unroll
                for (int t = 0; t < TOK; ++t)
                    if (t < ntok) p.y[(t0 + t) * p.N + n] = acc[t];
            }
        } else {
            if (c == 0) {
#pragma unroll
                for (int t = 0; t < TOK; ++t) red[warp][t][r8] = acc[t];
            }
            __syncthreads();
            if (kw == 0 && c == 0 && n < p.N) {
#pragma unroll
                for (int t = 0; t < TOK; ++t) {
                    if (t < ntok) {
                        float v = red[warp][t][r8];
                        for (int k = 1; k < wk; ++k) v += red[warp + k][t][r8];
                        p.y[(t0 + t) * p.N + n] = v;
                    }
                }
            }
            __syncthreads();
        }
    }
}

static int pick_wk(int64_t N, int64_t nsb, int64_t token_groups) {
    // enough warps in flight for HBM (about 13 per SM on 152 SMs), without
    // slicing a row finer than one superblock per warp
    const int64_t target_warps = 2048;
    int wk = 1;
    while (wk < 8 && wk * 2 <= nsb) {
        const int64_t blocks = (N + (64 / wk) - 1) / (64 / wk);
        if (blocks * 8 * token_groups >= target_warps) break;
        wk *= 2;
    }
    return wk;
}

template <int F, int TOK>
static cudaError_t launch_mv_s(const MvParams &p0, int64_t E, int64_t tg, cudaStream_t s) {
    MvParams p = p0;
    p.wk = pick_wk(p.N, p.nsb, tg * E);
    const int rows_per_block = 8 * (8 / p.wk);
    dim3 grid((unsigned)((p.N + rows_per_block - 1) / rows_per_block), (unsigned)tg, (unsigned)E);
    mv_kernel<F, TOK><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <int F>
static cudaError_t launch_mv_f(const MvParams &p, int64_t E, cudaStream_t s) {
    if (!p.offsets && p.M == 1) return launch_mv_s<F, 1>(p, 1, 1, s);
    // token groups of 8; enough groups in parallel to fill the GPU, each
    // block walking further groups with the same weights hot in L1/L2
    const int64_t per_expert = p.offsets ? (p.M + E - 1) / E : p.M;
    int64_t tg = (per_expert + 7) / 8;
    const int64_t row_blocks = (p.N + 63) / 64;
    const int64_t want = 4 * 152;
    const int64_t cap = (want + row_blocks * E - 1) / (row_blocks * E);
    if (tg > cap) tg = cap;
    if (tg < 1) tg = 1;
    if (p.M <= 2 && !p.offsets) return launch_mv_s<F, 2>(p, 1, 1, s);
    if (p.M <= 4 && !p.offsets) return launch_mv_s<F, 4>(p, 1, 1, s);
    return launch_mv_s<F, 8>(p, E, tg, s);
}

cudaError_t launch_mv(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                      const int32_t *row_offsets, int64_t E, uint64_t expert_bytes, float *y,
                      cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    MvParams p{};
    p.packed = static_cast<const uint8_t *>(packed);
    p.expert_bytes = expert_bytes;
    p.N = N;
    p.K = K;
    p.nsb = K / QK;
    p.d8 = a.d;
    p.qs = a.qs;
    p.bs = a.bsums;
    p.M = M;
    p.offsets = row_offsets;
    p.y = y;
    if (!row_offsets) E = 1;
    if (f == FMT_Q4_K) return launch_mv_f<FMT_Q4_K>(p, E, s);
    if (f == FMT_Q5_K) return launch_mv_f<FMT_Q5_K>(p, E, s);
    return launch_mv_f<FMT_Q6_K>(p, E, s);
}

// ---------------------------------------------------------------------------
// Test hook: decode the packed image with the GEMV's unpack helpers.
template <int F>
__global__ void __launch_bounds__(256) debug_decode_kernel(const uint8_t *packed, int64_t N, int64_t nsb,
                                                           int32_t *q, int32_t *sc, int32_t *mn, float *d,
                                                           float *dmin) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r8 = lane >> 2, c = lane & 3;
    const int64_t n = ((int64_t)blockIdx.x * 8 + warp) * 8 + r8;
    const int64_t sb = blockIdx.y;
    if (n >= N) return;
    const Planes P = make_planes(F, packed, N, nsb);
    typename WRegs<F>::T w;
    load_w(w, P, n, sb, nsb, c);
    LaneQ L;
    decode_lane(w, c, L);
    int32_t *qrow = q + (n * nsb + sb) * QK;
    const int width = (F == FMT_Q6_K) ? 16 : 32;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t wv[4] = {L.g[g].x, L.g[g].y, L.g[g].z, L.g[g].w};
        for (int i = 0; i < 16; ++i) qrow[L.aoff[g] + i] = (wv[i >> 2] >> (8 * (i & 3))) & 0xFF;
        sc[(n * nsb + sb) * 16 + L.aoff[g] / width] = L.sc[g];
    }
    if (F != FMT_Q6_K) {
        mn[(n * nsb + sb) * 8 + 2 * c] = L.m0;
        mn[(n * nsb + sb) * 8 + 2 * c + 1] = L.m1;
    } else {
        mn[(n * nsb + sb) * 8 + 2 * c] = 0;
        mn[(n * nsb + sb) * 8 + 2 * c + 1] = 0;
    }
    if (c == 0) {
        d[n * nsb + sb] = L.d;
        dmin[n * nsb + sb] = L.dmin;
    }
}

cudaError_t launch_debug_decode(int f, const void *packed, int64_t N, int64_t K, int32_t *q,
                                int32_t *sc, int32_t *mn, float *d, float *dmin, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    dim3 grid((unsigned)((N + 63) / 64), (unsigned)nsb);
    const uint8_t *pk = static_cast<const uint8_t *>(packed);
    if (f == FMT_Q4_K) debug_decode_kernel<FMT_Q4_K><<<grid, 256, 0, s>>>(pk, N, nsb, q, sc, mn, d, dmin);
    else if (f == FMT_Q5_K) debug_decode_kernel<FMT_Q5_K><<<grid, 256, 0, s>>>(pk, N, nsb, q, sc, mn, d, dmin);
    else debug_decode_kernel<FMT_Q6_K><<<grid, 256, 0, s>>>(pk, N, nsb, q, sc, mn, d, dmin);
    return cudaGetLastError();
}

}  // namespace kq
