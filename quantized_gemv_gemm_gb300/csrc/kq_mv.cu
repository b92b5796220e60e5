// kq_mv.cu - the CUDA-core matrix-vector family: decode GEMV (M = 1), the
// small-token-count product (a group of up to 8 tokens per pass) and its MoE
// grouped form, plus the two test hooks (int32 partials, packed decode).
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
//
// The GEMV streams the packed planes once from HBM ([kq-arc], kq v3 commit:
// decode time is set by DRAM traffic, so the planes stay bit-packed and no
// byte-expanded copy of them exists in DRAM).  Work split: a 256-thread block = 8 warps =
// WR row groups x WK superblock slices (WR * WK = 8).  A warp owns 8 rows
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
        if (s_begin < s_end) load_w(cur, P, (uint64_t)nc * p.nsb + s_begin, c);
        for (int64_t sb = s_begin; sb < s_end; ++sb) {
            if (sb + 1 < s_end) load_w(nxt, P, (uint64_t)nc * p.nsb + sb + 1, c);
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

// ---------------------------------------------------------------------------
// Decode GEMV (M = 1), over up to four matrices of one format that share one
// input row, optionally quantizing that row itself (fp32 in).
//
// Work split.  Rows are taken in groups of 8 (one per quad of a warp) across
// all the matrices; G groups in total.  A task is R = 8/S row groups x S
// superblock slices, one (group, slice) per warp of a 256-thread block; the
// S partial sums of a row are added in shared memory in a fixed order (the
// result does not depend on timing).  S is the smallest of 1, 2, 4, 8 that
// gives at least one task per block slot; every block gets the same number
// of consecutive tasks (tpc), so there is no partial second wave.
// Pipelining.  Each warp walks the flattened sequence (task, superblock of
// its slice) with a D-deep ring of weight registers: the loads for item i+D
// are issued as soon as item i is decoded, across task boundaries.  Slices
// are padded to a common length so every warp reaches each task's
// reduction barrier at the same item.  The first D items are loaded before
// griddep_wait() (weights are read-only on this path), overlapping the
// previous kernel under programmatic dependent launch; then the block stages
// the Q8_K row in shared memory (copied, or quantized from the fp32 row by
// quantize_block_warp, bit-identical to kq_quantize_q8k).

struct GemvParams {
    int nmat;
    const uint8_t *packed[GEMV_MAX_MATRICES];
    int64_t N[GEMV_MAX_MATRICES];
    float *y[GEMV_MAX_MATRICES];
    int64_t gpre[GEMV_MAX_MATRICES + 1];  // prefix sums of row groups
    int64_t K, nsb;
    int S;                                 // slices per row group (1, 2, 4, 8)
    int64_t tasks, tpc;                    // task count, tasks per block
    const float *x;                        // fp32 row (fused quantize), or nullptr
    const float *d8;                       // else: the Q8_K planes of the row
    const int8_t *qs;
    const int16_t *bs;
};

template <int F> constexpr int gemv_depth() { return F == FMT_Q4_K ? 4 : 3; }
constexpr int64_t GEMV_PREFETCH_TASKS = 3;

__host__ __device__ inline size_t gemv_smem_bytes(int64_t K) { return (size_t)(K + K / 8 + K / 64); }

template <int F, int D>
__global__ void __launch_bounds__(256, 2) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ Planes s_planes[GEMV_MAX_MATRICES];
    __shared__ float red[2][8][8];
    const int64_t K = p.K, nsb = p.nsb;
    int8_t *s_qs = reinterpret_cast<int8_t *>(smem);
    int16_t *s_bs = reinterpret_cast<int16_t *>(smem + K);
    float *s_d8 = reinterpret_cast<float *>(smem + K + K / 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r8 = lane >> 2, c = lane & 3;
    const int S = p.S, R = 8 / S;
    const int rg = warp / S, slice = warp % S;
    const int64_t s0 = slice * nsb / S, s1 = (slice + 1) * nsb / S, len = s1 - s0;
    const int64_t t_begin = (int64_t)blockIdx.x * p.tpc;
    const int64_t left = p.tasks - t_begin;
    const int64_t ntask = left <= 0 ? 0 : (left < p.tpc ? left : p.tpc);
    const int64_t G = p.gpre[p.nmat];
    if (threadIdx.x < p.nmat) s_planes[threadIdx.x] = make_planes(F, p.packed[threadIdx.x], p.N[threadIdx.x], nsb);
    __syncthreads();

    // task tl of this block -> this lane's matrix, row and plane pointers
    auto task_ptr = [&](int64_t tl, int &m, int64_t &n, bool &valid) {
        const int64_t g = (t_begin + tl) * R + rg;
        valid = g < G;
        m = 0;
        while (m + 1 < p.nmat && g >= p.gpre[m + 1]) ++m;
        n = (g - p.gpre[m]) * 8 + r8;
        const int64_t nc = n < p.N[m] ? n : p.N[m] - 1;
        return lane_ptr<F>(s_planes[m], (uint64_t)nc * nsb + s0, c);
    };
    // L2 prefetch of whole tasks (their rows are contiguous in every plane)
    auto prefetch_task = [&](int64_t tl) {
        if (tl >= ntask) return;
        const int64_t g0 = (t_begin + tl) * R, g1 = g0 + R < G ? g0 + R : G;
        int u[4];
        plane_unit_bytes(F, u);
        for (int m = 0; m < p.nmat; ++m) {
            const int64_t a = g0 > p.gpre[m] ? g0 : p.gpre[m], b = g1 < p.gpre[m + 1] ? g1 : p.gpre[m + 1];
            if (a >= b) continue;
            const int64_t r0 = (a - p.gpre[m]) * 8, r1e = (b - p.gpre[m]) * 8, r1 = r1e < p.N[m] ? r1e : p.N[m];
            const uint8_t *base[4] = {s_planes[m].p0, s_planes[m].p1, s_planes[m].p2, s_planes[m].p3};
            for (int q = 0; q < 4; ++q)
                if (u[q]) prefetch_l2_bulk(base[q] + (uint64_t)r0 * nsb * u[q], (uint64_t)(r1 - r0) * nsb * u[q]);
        }
    };
    if (threadIdx.x == 0)
        for (int64_t tl = 0; tl < GEMV_PREFETCH_TASKS; ++tl) prefetch_task(tl);

    using W = typename WRegs<F>::T;
    W buf[D];
    int m = 0;
    int64_t n = 0;
    bool valid = false;
    LanePtr lp{};
    if (ntask > 0) {
        lp = task_ptr(0, m, n, valid);
        if (valid) {
#pragma unroll
            for (int i = 0; i < D; ++i)
                if (i < len) load_at(buf[i], lp, i);
        }
    }

    griddep_wait();
    if (p.x) {
        for (int64_t b = warp; b < nsb; b += 8)
            quantize_block_warp(p.x + b * QK, lane, s_qs + b * QK, s_bs + b * 16, s_d8 + b);
    } else {
        const uint4 *gq = reinterpret_cast<const uint4 *>(p.qs);
        const uint4 *gb = reinterpret_cast<const uint4 *>(p.bs);
        for (int64_t i = threadIdx.x; i < K / 16; i += 256) reinterpret_cast<uint4 *>(s_qs)[i] = gq[i];
        for (int64_t i = threadIdx.x; i < K / 128; i += 256) reinterpret_cast<uint4 *>(s_bs)[i] = gb[i];
        for (int64_t i = threadIdx.x; i < nsb; i += 256) s_d8[i] = p.d8[i];
    }
    __syncthreads();
    griddep_launch_dependents();

    for (int64_t tl = 0; tl < ntask; ++tl) {
        // fold this task's slice: every lane folds its own int32 partials
        // once per superblock; the quad's four lanes are added at the end
        float acc = 0.0f;
        if (valid) {
            for (int64_t j = 0; j < len; j += D) {
#pragma unroll
                for (int i = 0; i < D; ++i) {
                    if (j + i < len) {
                        const int64_t sb = s0 + j + i;
                        LaneQ L;
                        decode_lane(buf[i], c, L);
                        if (j + i + D < len) load_at(buf[i], lp, j + i + D);
                        int isum, msum;
                        lane_partials<F, true>(L, s_qs + sb * QK, s_bs + sb * 16, c, isum, msum);
                        const float d8 = s_d8[sb];
                        acc = fmaf(L.d * d8, static_cast<float>(isum), acc);
                        if constexpr (F != FMT_Q6_K) acc = fmaf(-(L.dmin * d8), static_cast<float>(msum), acc);
                    }
                }
            }
        }
        // the next task's first loads go out before the reduction barrier
        int m2 = 0;
        int64_t n2 = 0;
        bool valid2 = false;
        LanePtr lp2{};
        if (tl + 1 < ntask) {
            lp2 = task_ptr(tl + 1, m2, n2, valid2);
            if (valid2) {
#pragma unroll
                for (int i = 0; i < D; ++i)
                    if (i < len) load_at(buf[i], lp2, i);
            }
        }
        if (threadIdx.x == 0) prefetch_task(tl + GEMV_PREFETCH_TASKS);
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
        if (c == 0) red[tl & 1][warp][r8] = acc;
        __syncthreads();
        if (slice == 0 && c == 0 && valid && n < p.N[m]) {
            float v = 0.0f;
            for (int j = 0; j < S; ++j) v += red[tl & 1][rg * S + j][r8];
            p.y[m][n] = v;
        }
        m = m2;
        n = n2;
        valid = valid2;
        lp = lp2;
    }
}

static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
        cached[dev] = v;
    }
    return cached[dev];
}

template <int F>
static cudaError_t launch_gemv_t(GemvParams p, cudaStream_t s) {
    p.gpre[0] = 0;
    for (int m = 0; m < p.nmat; ++m) p.gpre[m + 1] = p.gpre[m] + (p.N[m] + 7) / 8;
    const int64_t G = p.gpre[p.nmat];
    if (G == 0) return cudaSuccess;
    const int64_t slots = 2 * (int64_t)sm_count();  // two resident blocks per SM
    int S = 1;
    while (S < 8 && 2 * S <= p.nsb && (G * S + 7) / 8 < slots) S *= 2;
    p.S = S;
    const int64_t R = 8 / S;
    p.tasks = (G + R - 1) / R;
    p.tpc = (p.tasks + slots - 1) / slots;
    const int64_t blocks = (p.tasks + p.tpc - 1) / p.tpc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = gemv_smem_bytes(p.K);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<F, gemv_depth<F>()>, p);
}

cudaError_t launch_gemv(int f, int nmat, const void *const *packed, const int64_t *N, int64_t K, const float *x,
                        Q8K a, float *const *y, cudaStream_t s) {
    GemvParams p{};
    p.nmat = nmat;
    for (int m = 0; m < nmat; ++m) {
        p.packed[m] = static_cast<const uint8_t *>(packed[m]);
        p.N[m] = N[m];
        p.y[m] = y[m];
    }
    p.K = K;
    p.nsb = K / QK;
    p.x = x;
    p.d8 = a.d;
    p.qs = a.qs;
    p.bs = a.bsums;
    if (f == FMT_Q4_K) return launch_gemv_t<FMT_Q4_K>(p, s);
    if (f == FMT_Q5_K) return launch_gemv_t<FMT_Q5_K>(p, s);
    return launch_gemv_t<FMT_Q6_K>(p, s);
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
// Test hook: int32 partials per (token, row, superblock), with the GEMV's own
// unpack and lane partials.  One warp = 8 rows x one superblock x one token.
template <int F>
__global__ void __launch_bounds__(256) partials_kernel(const uint8_t *packed, int64_t N, int64_t nsb, int64_t K,
                                                       Q8K a, int64_t M, int32_t *isum_out, int32_t *msum_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r8 = lane >> 2, c = lane & 3;
    const int64_t n = ((int64_t)blockIdx.x * 8 + warp) * 8 + r8;
    const int64_t sb = blockIdx.y;
    const int64_t tok = blockIdx.z;
    const int64_t nc = n < N ? n : N - 1;
    const Planes P = make_planes(F, packed, N, nsb);
    typename WRegs<F>::T w;
    load_w(w, P, (uint64_t)nc * nsb + sb, c);
    LaneQ L;
    decode_lane(w, c, L);
    int isum, msum;
    lane_partials<F>(L, a.qs + tok * K + sb * QK, a.bsums + (tok * nsb + sb) * 16, c, isum, msum);
    isum = quad_sum(isum);
    msum = quad_sum(msum);
    if (c == 0 && n < N) {
        const int64_t o = (tok * N + n) * nsb + sb;
        isum_out[o] = isum;
        msum_out[o] = msum;
    }
}

cudaError_t launch_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                            int32_t *isum, int32_t *msum, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    dim3 grid((unsigned)((N + 63) / 64), (unsigned)nsb, (unsigned)M);
    const uint8_t *pk = static_cast<const uint8_t *>(packed);
    if (f == FMT_Q4_K) partials_kernel<FMT_Q4_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    else if (f == FMT_Q5_K) partials_kernel<FMT_Q5_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    else partials_kernel<FMT_Q6_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    return cudaGetLastError();
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
    load_w(w, P, (uint64_t)n * nsb + sb, c);
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
