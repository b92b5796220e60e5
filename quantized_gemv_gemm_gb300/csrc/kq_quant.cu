// kq_quant.cu - Q8_K activation quantization and the one-time weight repack.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
#include "kq_internal.h"

namespace kq {

// ---------------------------------------------------------------------------
// Q8_K quantization of M rows: one warp per 256-block (quantize_block_warp
// in kq_device.cuh holds the arithmetic).
__global__ void __launch_bounds__(256) quantize_q8k_kernel(const float *__restrict__ x, int64_t K,
                                                           int64_t nblocks, float *__restrict__ d,
                                                           int8_t *__restrict__ qs,
                                                           int16_t *__restrict__ bsums) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    // x may be produced, and the Q8_K planes still read, by the previous
    // kernels in the stream
    griddep_wait();
    griddep_launch_dependents();
    if (blk >= nblocks) return;
    const int64_t nsb = K / QK;
    const int64_t m = blk / nsb, sb = blk % nsb;
    quantize_block_warp(x + m * K + sb * QK, lane, qs + m * K + sb * QK, bsums + blk * 16, d + blk);
}

cudaError_t launch_quantize(const float *x, int64_t M, int64_t K, float *d, int8_t *qs,
                            int16_t *bsums, cudaStream_t s) {
    const int64_t nblocks = M * (K / QK);
    if (nblocks == 0) return cudaSuccess;
    const int64_t grid = (nblocks + 7) / 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_q8k_kernel, x, K, nblocks, d, qs, bsums);
}

// ---------------------------------------------------------------------------
// Repack ([kq-arc], k4 kq-v2 commit: the transcode keeps the disk scale block
// as it is, and the planes dequantize bit-identically to the disk blocks).
// One thread per (row n, superblock sb) of the rows padded to whole groups
// of 16 moves each 16-byte piece of the GGUF-order block to its place in the
// grp16 image (kq_device.cuh); no value is changed, and the padding rows are
// zero.  The disk block is read as 16-bit words (210-byte Q6_K blocks are
// only 2-byte aligned).

__device__ __forceinline__ uint4 piece16(const uint16_t *src) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = static_cast<uint32_t>(src[2 * j]) | (static_cast<uint32_t>(src[2 * j + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// W1 of half h of one disk superblock: the sum over its 128 weights of
// |sub-scale| * |q| (Q4_K/Q5_K: q with its fifth bit; Q6_K: q - 32), in the
// GGUF element order (the same order the kernels unpack).
template <int F>
__device__ uint32_t half_l1(const uint8_t *blk, int h) {
    uint32_t w1 = 0;
    if constexpr (F == FMT_Q4_K || F == FMT_Q5_K) {
        const uint8_t *sc = blk + 4;
        const uint8_t *qh = blk + 16;
        const uint8_t *qs = blk + (F == FMT_Q5_K ? 48 : 16);
        for (int j = 4 * h; j < 4 * h + 4; ++j) {
            const uint32_t s = j < 4 ? (sc[j] & 63u) : ((sc[j + 4] & 15u) | ((uint32_t)(sc[j - 4] >> 6) << 4));
            uint32_t sum = 0;
            for (int l = 0; l < 32; ++l) {
                const uint8_t b = qs[32 * (j >> 1) + l];
                uint32_t q = (j & 1) ? (b >> 4) : (b & 15u);
                if constexpr (F == FMT_Q5_K) q += 16u * ((qh[l] >> j) & 1u);
                sum += q;
            }
            w1 += s * sum;
        }
    } else {
        const uint8_t *ql = blk + 64 * h, *qh = blk + 128 + 32 * h;
        const int8_t *sc = reinterpret_cast<const int8_t *>(blk + 192);
        for (int t = 0; t < 4; ++t)
            for (int l = 0; l < 32; ++l) {
                const uint8_t b = ql[32 * (t & 1) + l];
                const int q = (int)((t < 2 ? (b & 15u) : (b >> 4)) | (((qh[l] >> (2 * t)) & 3u) << 4));
                const int s = sc[8 * h + 2 * t + l / 16];
                w1 += (uint32_t)((s < 0 ? -s : s) * (q < 32 ? 32 - q : q - 32));
            }
    }
    return w1;
}

template <int F>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ disk, int64_t N, int64_t nsb,
                                                     int64_t units, Planes P) {
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int64_t n = u / nsb, sb = u % nsb;
    const uint64_t ch = chunk_of(n, sb, nsb);
    const int r = (int)(n % GROUP_ROWS);
    uint8_t *p0 = const_cast<uint8_t *>(P.p0), *p1 = const_cast<uint8_t *>(P.p1);
    uint8_t *p2 = const_cast<uint8_t *>(P.p2), *p3 = const_cast<uint8_t *>(P.p3);
    const bool real = n < N;
    const uint16_t *b = reinterpret_cast<const uint16_t *>(disk + (real ? u : 0) * (int64_t)block_bytes(F));
    const uint4 zero = make_uint4(0, 0, 0, 0);
    auto piece = [&](int off16) { return real ? piece16(b + off16) : zero; };  // off16 in 16-bit words
    auto put = [&](uint8_t *dst, uint4 v) { *reinterpret_cast<uint4 *>(dst) = v; };
    if constexpr (F == FMT_Q4_K) {
        put(p1 + ch * 256 + 16 * r, piece(0));                                     // d, dmin, scales[12]
        for (int i = 0; i < 8; ++i) put(p0 + ch * 2048 + piece_offset(128, r, i), piece(8 + 8 * i));   // qs
    } else if constexpr (F == FMT_Q5_K) {
        put(p2 + ch * 256 + 16 * r, piece(0));                                     // d, dmin, scales[12]
        for (int i = 0; i < 2; ++i) put(p1 + ch * 512 + piece_offset(32, r, i), piece(8 + 8 * i));     // qh
        for (int i = 0; i < 8; ++i) put(p0 + ch * 2048 + piece_offset(128, r, i), piece(24 + 8 * i));  // qs
    } else {
        for (int i = 0; i < 8; ++i) put(p0 + ch * 2048 + piece_offset(128, r, i), piece(8 * i));       // ql
        for (int i = 0; i < 4; ++i) put(p1 + ch * 1024 + piece_offset(64, r, i), piece(64 + 8 * i));   // qh
        put(p2 + ch * 256 + 16 * r, piece(96));                                    // scales (int8)
        reinterpret_cast<uint16_t *>(p3 + ch * 32)[r] = real ? b[104] : uint16_t(0);  // d
    }
    // the group's bounds: the largest W1 of each half over its rows (the
    // plane is zero-filled before this kernel)
    if (real) {
        const uint8_t *blk = reinterpret_cast<const uint8_t *>(b);
        uint32_t *bound = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(P.p4)) + 2 * (int64_t)ch;
        atomicMax(bound, half_l1<F>(blk, 0));
        atomicMax(bound + 1, half_l1<F>(blk, 1));
    }
}

cudaError_t launch_repack(int f, const uint8_t *disk, int64_t N, int64_t K, uint8_t *packed,
                          cudaStream_t s) {
    const int64_t nsb = K / QK;
    const int64_t units = row_groups(N) * GROUP_ROWS * nsb;
    if (units == 0) return cudaSuccess;
    const Planes P = make_planes(f, packed, N, nsb);
    cudaError_t e = cudaMemsetAsync(const_cast<uint8_t *>(P.p4), 0, (size_t)row_groups(N) * nsb * BOUND_BYTES, s);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((units + 255) / 256);
    if (f == FMT_Q4_K) repack_kernel<FMT_Q4_K><<<grid, 256, 0, s>>>(disk, N, nsb, units, P);
    else if (f == FMT_Q5_K) repack_kernel<FMT_Q5_K><<<grid, 256, 0, s>>>(disk, N, nsb, units, P);
    else repack_kernel<FMT_Q6_K><<<grid, 256, 0, s>>>(disk, N, nsb, units, P);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Copy-in of a step's inputs from pinned host memory (mapped into the device
// address space) to device memory, as a kernel of the stream's launch chain:
// each thread loads its COPY_IN_VEC 16-byte words before the dependency wait
// (the source is written by the host, never by an earlier kernel, so the
// slow host reads overlap the previous kernel) and stores them after it.
// (Measured on GB300 in the decode chain, 75 KB per step: one word per
// thread in blocks of 128, 25.0 us per step, against 25.9 with four words
// and 25.3 with blocks of 32.)
#ifndef KQ_COPY_IN_VEC
#define KQ_COPY_IN_VEC 1
#endif
#ifndef KQ_COPY_IN_THREADS
#define KQ_COPY_IN_THREADS 128
#endif
constexpr int COPY_IN_VEC = KQ_COPY_IN_VEC;
constexpr int COPY_IN_THREADS = KQ_COPY_IN_THREADS;

__global__ void __launch_bounds__(COPY_IN_THREADS) copy_in_kernel(const uint4 *__restrict__ src,
                                                                  uint4 *__restrict__ dst, int64_t n16) {
    griddep_launch_dependents();
    const int64_t base = (int64_t)blockIdx.x * COPY_IN_THREADS * COPY_IN_VEC + threadIdx.x;
    uint4 v[COPY_IN_VEC];
#pragma unroll
    for (int k = 0; k < COPY_IN_VEC; ++k) {
        const int64_t i = base + (int64_t)k * COPY_IN_THREADS;
        if (i < n16) v[k] = src[i];
    }
    griddep_wait();  // earlier kernels may still read dst
#pragma unroll
    for (int k = 0; k < COPY_IN_VEC; ++k) {
        const int64_t i = base + (int64_t)k * COPY_IN_THREADS;
        if (i < n16) dst[i] = v[k];
    }
}

cudaError_t launch_copy_in(const void *src, void *dst, size_t bytes, cudaStream_t s) {
    const int64_t n16 = (int64_t)(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    const int64_t per_block = (int64_t)COPY_IN_THREADS * COPY_IN_VEC;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n16 + per_block - 1) / per_block));
    cfg.blockDim = dim3(COPY_IN_THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, copy_in_kernel, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
}

}  // namespace kq
