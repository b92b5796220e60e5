// kq_q8_0.cu - the Q8_0 rail: Q8_0 weights (blocks of 32: an fp16 scale and
// 32 int8 quants) read with Q8_0-form activations (one fp32 scale per 32).
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
// Its chain-regrain commit keeps one activation image per consumed form: the
// Q8_0 projections read a Q8_0-form image while the K-quant ones read Q8_K;
// its MoE prefill fix names the Q8_0 weights' separate fp16 scale plane.
// Per output: y[n] = sum over 32-blocks b of d_w(n, b) * d_a(b) * isum_b,
// isum_b = sum_k q_w * q_a in int32 (dp4a), one float fold per block.
//
// Packed image (rows in groups of 16, the last group padded with zeros; for
// every (row group g, 256-column superblock sb) in the order g * K/256 + sb
// one chunk per plane; planes on 256-byte boundaries):
//   qs plane: 4096-byte chunks; row r's 16-byte piece k (columns 16k..16k+15
//             of the superblock) at 256*k + 16*r
//   d  plane: 256-byte chunks; row r's 8 fp16 block scales at 16*r
// So a half-warp reading piece k of 16 rows reads 256 consecutive bytes, and
// every disk byte is kept once (1.0625 bytes per weight, as on disk).
#include "kq_internal.h"

namespace kq {

constexpr int QK8_0 = 32;
constexpr int Q8_0_BLOCK = 34;

// Offsets of the two planes of an [N][K] Q8_0 image; off[2] = total bytes.
static void q8_0_planes(int64_t N, int64_t nsb, uint64_t off[3]) {
    const uint64_t chunks = (uint64_t)row_groups(N) * (uint64_t)nsb;
    off[0] = 0;
    off[1] = align256(chunks * 4096);
    off[2] = off[1] + align256(chunks * 256);
}

uint64_t q8_0_image_bytes(int64_t N, int64_t K) {
    uint64_t off[3];
    q8_0_planes(N, K / QK, off);
    return off[2];
}

// ---------------------------------------------------------------------------
// Q8_0 activations: 4 lanes per 32-block (8 values each), so a warp does 8
// blocks at once.  Same arithmetic as Q8_K per block (IEEE fp32 division and
// product, round half to even, clamp to +-127).  Lanes whose block is past
// the end (on == false) take part in the shuffles and store nothing.  The
// load and the arithmetic are separate steps so that a loop can have the
// next values in flight while it quantizes the current ones.
__device__ __forceinline__ void q8_0_load_lanes(const float *x, int64_t blk, bool on, int lane, float (&v)[8]) {
    const int64_t base = (on ? blk : 0) * QK8_0 + 8 * (lane & 3);
    if (on) {
        const float4 a = *reinterpret_cast<const float4 *>(x + base);
        const float4 b = *reinterpret_cast<const float4 *>(x + base + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
}

__device__ __forceinline__ void q8_0_quant_lanes(const float (&v)[8], int64_t blk, bool on, int lane, float *d,
                                                 int8_t *qs) {
    const int64_t base = (on ? blk : 0) * QK8_0 + 8 * (lane & 3);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    if (!on) return;
    uint32_t w[2] = {0u, 0u};
    if (amax > 0.0f) {
        const float iscale = __fdiv_rn(127.0f, amax);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = __float2int_rn(__fmul_rn(v[i], iscale));
            q = q > 127 ? 127 : (q < -127 ? -127 : q);
            w[i >> 2] |= (uint32_t)(q & 0xFF) << (8 * (i & 3));
        }
    }
    *reinterpret_cast<uint2 *>(qs + base) = make_uint2(w[0], w[1]);
    if ((lane & 3) == 0) d[blk] = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
}

// a warp per 8 blocks of the flattened [M][K/32] block list
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float *__restrict__ x, int64_t nblocks,
                                                            float *__restrict__ d, int8_t *__restrict__ qs) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t blk = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 8 + (lane >> 2);
    float v[8];
    q8_0_load_lanes(x, blk, blk < nblocks, lane, v);
    q8_0_quant_lanes(v, blk, blk < nblocks, lane, d, qs);
}

cudaError_t launch_quantize_q8_0(const float *x, int64_t M, int64_t K, float *d, int8_t *qs, cudaStream_t s) {
    const int64_t nblocks = M * (K / QK8_0);
    if (nblocks == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((nblocks + 63) / 64));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel, x, nblocks, d, qs);
}

// ---------------------------------------------------------------------------
// Repack: one thread per (row n of the rows padded to whole groups, 32-block
// b).  The 34-byte disk block is read as 16-bit words (it is only 2-byte
// aligned); no value changes, padding rows are zero.
__global__ void __launch_bounds__(256) repack_q8_0_kernel(const uint8_t *__restrict__ disk, int64_t N, int64_t nb,
                                                          int64_t units, uint8_t *__restrict__ qs_plane,
                                                          uint8_t *__restrict__ d_plane) {
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int64_t n = u / nb, b = u % nb;
    const int64_t nsb = nb / 8, sb = b / 8;
    const int j = (int)(b % 8);                       // 32-block of the superblock
    const int r = (int)(n % GROUP_ROWS);
    const uint64_t ch = (uint64_t)(n / GROUP_ROWS) * (uint64_t)nsb + (uint64_t)sb;
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint16_t dbits = 0;
    if (n < N) {
        const uint16_t *src = reinterpret_cast<const uint16_t *>(disk + u * Q8_0_BLOCK);
        dbits = src[0];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = (uint32_t)src[1 + 2 * i] | ((uint32_t)src[2 + 2 * i] << 16);
    }
    uint8_t *q = qs_plane + ch * 4096 + 16 * r;
    *reinterpret_cast<uint4 *>(q + 256 * (2 * j)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(q + 256 * (2 * j + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
    reinterpret_cast<uint16_t *>(d_plane + ch * 256 + 16 * r)[j] = dbits;
}

cudaError_t launch_repack_q8_0(const uint8_t *disk, int64_t N, int64_t K, uint8_t *packed, cudaStream_t s) {
    const int64_t nb = K / QK8_0;
    const int64_t units = row_groups(N) * GROUP_ROWS * nb;
    if (units == 0) return cudaSuccess;
    uint64_t off[3];
    q8_0_planes(N, K / QK, off);
    repack_q8_0_kernel<<<(unsigned)((units + 255) / 256), 256, 0, s>>>(disk, N, nb, units, packed, packed + off[1]);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// GEMV: one block per 16-row group; its 8 warps take the superblocks
// sb = warp, warp + 8, ...; lane (r = lane % 16, half = lane / 16) folds row
// r's columns 128*half .. +127 of each (8 x 16-byte pieces, 4 blocks of 32).
// The activation row is staged in shared memory once per block.  Each row's
// partial sums are added in a fixed order (lane pair, then warps 0..7), so
// the result does not depend on scheduling.
// PIPE: each warp loads its next superblock while folding the current one
// (two in flight, 96 registers: best for short rows, where a warp has one or
// two superblocks); otherwise one at a time (72 registers, one more block
// per SM: best for long rows).  The first superblock's weights are loaded
// before the dependency wait either way.
// FUSED: the block quantizes the fp32 row x itself (bit-identical to
// kq_quantize_q8_0, the next 8 values of each lane loaded while the current
// ones are quantized) instead of copying the Q8_0 planes d_a, q_a; the grid
// is then at most the resident blocks of all SMs, each block walking the row
// groups g = blockIdx.x, + gridDim.x, ... so that the row is quantized once
// per block rather than once per row group.  The next group's first
// superblock is loaded while the current group's sums are reduced.
template <bool PIPE, bool FUSED>
__global__ void __launch_bounds__(256) gemv_q8_0_kernel(const uint8_t *__restrict__ qs_plane,
                                                        const uint8_t *__restrict__ d_plane, int64_t N, int64_t nsb,
                                                        const float *__restrict__ d_a, const int8_t *__restrict__ q_a,
                                                        const float *__restrict__ x, float *__restrict__ y) {
    extern __shared__ __align__(16) uint8_t sm[];
    __shared__ float part[8][16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane & 15, hf = lane >> 4;
    const int64_t K = nsb * QK;
    const uint64_t groups = (uint64_t)row_groups(N);
    uint64_t g = blockIdx.x;
    griddep_launch_dependents();
    // one superblock's weights of this lane: 8 pieces of 16 quants + 4 scales
    struct W {
        uint4 q[8];
        uint2 d;
    };
    auto load = [&](W &w, int64_t sb) {
        const uint64_t ch = g * (uint64_t)nsb + (uint64_t)sb;
        const uint8_t *qc = qs_plane + ch * 4096 + 16 * r + 256 * 8 * hf;
#pragma unroll
        for (int k = 0; k < 8; ++k) w.q[k] = ld_stream(qc + 256 * k);
        w.d = __ldg(reinterpret_cast<const uint2 *>(d_plane + ch * 256 + 16 * r + 8 * hf));
    };
    // the weights do not depend on earlier kernels: the first superblock is
    // in flight before the dependency wait
    W cur, nxt;
    int64_t sb = warp;
    if (sb < nsb) load(cur, sb);
    griddep_wait();  // the activations are written by the kernels before this one
    float *s_d = reinterpret_cast<float *>(sm + K);
    if constexpr (FUSED) {
        const int64_t nblk = K / QK8_0;
        float v[8], vn[8];
        int64_t blk = (int64_t)warp * 8 + (lane >> 2);
        q8_0_load_lanes(x, blk, blk < nblk, lane, v);
        for (int64_t b0 = (int64_t)warp * 8; b0 < nblk; b0 += 64, blk += 64) {
            q8_0_load_lanes(x, blk + 64, blk + 64 < nblk, lane, vn);
            q8_0_quant_lanes(v, blk, blk < nblk, lane, s_d, reinterpret_cast<int8_t *>(sm));
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = vn[i];
        }
    } else {
        for (int64_t i = threadIdx.x; i < K / 16; i += 256)
            reinterpret_cast<uint4 *>(sm)[i] = __ldg(reinterpret_cast<const uint4 *>(q_a) + i);
        for (int64_t i = threadIdx.x; i < K / QK8_0; i += 256) s_d[i] = __ldg(d_a + i);
    }
    __syncthreads();
    for (;;) {
        float acc = 0.0f;
        for (sb = warp; sb < nsb; sb += 8) {
            if (PIPE && sb + 8 < nsb) load(nxt, sb + 8);
            const uint8_t *ac = sm + sb * QK + 128 * hf;
            const float *dac = s_d + sb * 8 + 4 * hf;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 a0 = *reinterpret_cast<const uint4 *>(ac + 32 * j);
                const uint4 a1 = *reinterpret_cast<const uint4 *>(ac + 32 * j + 16);
                const uint4 w0 = cur.q[2 * j], w1 = cur.q[2 * j + 1];
                int isum = 0;
                isum = __dp4a((int)w0.x, (int)a0.x, isum);
                isum = __dp4a((int)w0.y, (int)a0.y, isum);
                isum = __dp4a((int)w0.z, (int)a0.z, isum);
                isum = __dp4a((int)w0.w, (int)a0.w, isum);
                isum = __dp4a((int)w1.x, (int)a1.x, isum);
                isum = __dp4a((int)w1.y, (int)a1.y, isum);
                isum = __dp4a((int)w1.z, (int)a1.z, isum);
                isum = __dp4a((int)w1.w, (int)a1.w, isum);
                const uint32_t hw = (j < 2 ? cur.d.x : cur.d.y) >> (16 * (j & 1));
                const float dwf = __half2float(__ushort_as_half((unsigned short)(hw & 0xFFFF)));
                acc = fmaf(dwf * dac[j], static_cast<float>(isum), acc);
            }
            if (PIPE) cur = nxt;
            else if (sb + 8 < nsb) load(cur, sb + 8);
        }
        const uint64_t gn = g + gridDim.x;
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
        if (hf == 0) part[warp][r] = acc;
        __syncthreads();
        if (warp == 0 && lane < 16) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) t += part[w][lane];
            const int64_t n = (int64_t)g * GROUP_ROWS + lane;
            if (n < N) y[n] = t;
        }
        if (!FUSED || gn >= groups) break;
        g = gn;
        if (warp < nsb) load(cur, warp);
        __syncthreads();  // part[] is read before the next group writes it
    }
}

cudaError_t launch_gemv_q8_0(const void *packed, int64_t N, int64_t K, const float *d_a, const int8_t *q_a,
                             const float *x, float *y, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    uint64_t off[3];
    q8_0_planes(N, nsb, off);
    const uint8_t *p = static_cast<const uint8_t *>(packed);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)row_groups(N));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = (size_t)K + (size_t)(K / QK8_0) * 4;
    if (x) {
        auto kern = nsb < 16 ? gemv_q8_0_kernel<true, true> : gemv_q8_0_kernel<false, true>;
        int per_sm = 0, dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
        const int64_t resident = (int64_t)std::max(per_sm, 1) * sms;
        cfg.gridDim = dim3((unsigned)std::min<int64_t>(row_groups(N), resident));
    }
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    // rows of fewer than 16 superblocks: two in flight per warp (measured on
    // GB300: K = 2560 rows 3.1 vs 2.4 TB/s; K = 5120 and 17408 rows the other
    // way round, 5.6 vs 5.1 and 5.5 vs 4.5 TB/s)
    if (x) {
        if (nsb < 16) return cudaLaunchKernelEx(&cfg, gemv_q8_0_kernel<true, true>, p, p + off[1], N, nsb, d_a, q_a, x, y);
        return cudaLaunchKernelEx(&cfg, gemv_q8_0_kernel<false, true>, p, p + off[1], N, nsb, d_a, q_a, x, y);
    }
    if (nsb < 16) return cudaLaunchKernelEx(&cfg, gemv_q8_0_kernel<true, false>, p, p + off[1], N, nsb, d_a, q_a, x, y);
    return cudaLaunchKernelEx(&cfg, gemv_q8_0_kernel<false, false>, p, p + off[1], N, nsb, d_a, q_a, x, y);
}

}  // namespace kq
