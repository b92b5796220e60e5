// kq_q8_0_gemm.cu - prefill GEMM of the Q8_0 rail: Q8_0 weights (blocks of
// 32: fp16 scale, 32 int8 quants) times Q8_0-form activations (one fp32
// scale per 32) for M token rows.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450):
// its chain-regrain commit gives the q8 projections their own Q8_0-form
// activation image, and its MoE prefill fix has the Q8_0 GEMMs read it.
// Per output y[m][n] = sum over 32-blocks b of d_w(n, b) * d_a(m, b) *
// isum(m, n, b), isum = sum_k q_w * q_a in int32, one float fold per block.
//
// The integer dot of one block is one warp-level integer MMA: mma.sync
// m16n8k32 s8 x s8 -> s32 takes K = 32, so each instruction is exactly one
// Q8_0 block of 16 weight rows x 8 tokens, exact in int32 (|isum| <= 32 *
// 128 * 128 = 2^19), and the fold follows per block in fp32.  (sm_103a has
// no integer tcgen05.mma; fp16 operands are exact for the quants, but the
// per-block scales would drain the accumulator every 32 columns.)
//
// Tiling: a block of 8 warps computes 128 weight rows (8 row groups of the
// image) x 64 tokens; warp w takes rows 32 * (w % 4) .. +31 and tokens
// 32 * (w / 4) .. +31 (2 x 4 MMA tiles).  The weights and activations of one
// 256-column superblock are staged per stage of a 3-deep cp.async ring:
// the 8 row groups' qs chunks as they are in the image (row r's 16-byte
// piece k at 256k + 16r: a lane's A fragment words are 32 distinct banks),
// their fp16 scale chunks, the 64 token rows' 256 quants padded to 272 bytes
// (B fragment words in distinct banks), and the tokens' 8 block scales.
#include "kq_internal.h"

#include <atomic>

namespace kq {
namespace {

constexpr int QG_BM = 128, QG_BT = 64, QG_THREADS = 256, QG_STAGES = 3;
constexpr int QG_W = 8 * 4096;           // qs chunks of 8 row groups
constexpr int QG_S = 8 * 256;            // fp16 scale chunks
constexpr int QG_AROW = 272;             // staged token row (256 quants + pad)
constexpr int QG_A = QG_BT * QG_AROW;
constexpr int QG_D = QG_BT * 8 * 4;      // tokens' block scales
constexpr int QG_STAGE = QG_W + QG_S + QG_A + QG_D;
constexpr int QG_SMEM = QG_STAGES * QG_STAGE;
static_assert(QG_STAGE % 16 == 0, "stage alignment");
static_assert(QG_SMEM <= 232448, "shared memory per block");

// 16-byte copy that writes zeros when !valid (src must still be a valid address)
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void mma_k32_s8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

// an int32 of magnitude below 2^22 as fp32, exactly: the bits of
// 1.5 * 2^23 + x, less 1.5 * 2^23
__device__ __forceinline__ float small_int_to_float(int x) {
    return __int_as_float(x + 0x4B400000) - 12582912.0f;
}

struct Q8GemmParams {
    const uint8_t *qs, *sc;  // the image's two planes
    const float *d_a;        // [M][K/32]
    const int8_t *q_a;       // [M][K]
    float *y;                // [M][N]
    int64_t N, K, M, nsb, groups;
};

__global__ void __launch_bounds__(QG_THREADS, 1) q8_0_gemm_kernel(const Q8GemmParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();
    griddep_wait();  // the activation image is written by the kernels before this one
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int t_tiles = (int)((p.M + QG_BT - 1) / QG_BT);
    const int64_t t0 = (int64_t)(blockIdx.x % t_tiles) * QG_BT;
    const int64_t g0 = (int64_t)(blockIdx.x / t_tiles) * 8;  // first row group of the tile
    const int64_t nb = p.K / 32;
    const uint32_t sbase = smem_addr(smem);

    // stage sb into ring slot `slot`
    auto load_stage = [&](int64_t sb, int slot) {
        const uint32_t st = sbase + (uint32_t)(slot * QG_STAGE);
        // weights: 8 chunks of 4096 B, 8 pieces per thread (zeros past the image)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int piece = tid + QG_THREADS * i;       // 0 .. 2047
            const int gi = piece >> 8, off = (piece & 255) * 16;
            const bool v = g0 + gi < p.groups;
            const uint8_t *src = p.qs + (v ? ((g0 + gi) * p.nsb + sb) * 4096 + off : 0);
            cp_async16_zfill(st + gi * 4096 + off, src, v);
        }
        if (tid < 128) {  // scales: 8 chunks of 256 B
            const int gi = tid >> 4, off = (tid & 15) * 16;
            const bool v = g0 + gi < p.groups;
            const uint8_t *src = p.sc + (v ? ((g0 + gi) * p.nsb + sb) * 256 + off : 0);
            cp_async16_zfill(st + QG_W + gi * 256 + off, src, v);
        }
        // activations: 64 token rows x 16 pieces, 4 per thread (zeros past M)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int piece = tid + QG_THREADS * i;       // 0 .. 1023
            const int ti = piece >> 4, k = piece & 15;
            const bool v = t0 + ti < p.M;
            const int8_t *src = p.q_a + (v ? (t0 + ti) * p.K + sb * 256 + 16 * k : 0);
            cp_async16_zfill(st + QG_W + QG_S + ti * QG_AROW + 16 * k, src, v);
        }
        if (tid < 128) {  // the tokens' 8 block scales, two pieces per token
            const int ti = tid >> 1, hf = tid & 1;
            const bool v = t0 + ti < p.M;
            const float *src = p.d_a + (v ? (t0 + ti) * nb + sb * 8 + 4 * hf : 0);
            cp_async16_zfill(st + QG_W + QG_S + QG_A + ti * 32 + 16 * hf, src, v);
        }
    };

    float y[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) y[mt][nt][i] = 0.0f;
    const int rs = warp & 3, ts = warp >> 2;

    for (int s = 0; s < QG_STAGES - 1; ++s) {
        if (s < p.nsb) load_stage(s, s);
        cp_async_commit();
    }
    for (int64_t sb = 0; sb < p.nsb; ++sb) {
        cp_async_wait<QG_STAGES - 2>();  // stage sb has landed (this thread's copies)
        __syncthreads();                 // everyone's copies; the slot refilled below is free
        {
            const int64_t nxt = sb + QG_STAGES - 1;
            if (nxt < p.nsb) load_stage(nxt, (int)(nxt % QG_STAGES));
            cp_async_commit();
        }
        const uint32_t st = sbase + (uint32_t)((sb % QG_STAGES) * QG_STAGE);
        const uint32_t wq = st, wsc = st + QG_W, aq = st + QG_W + QG_S, ad = st + QG_W + QG_S + QG_A;
#pragma unroll 2
        for (int b = 0; b < 8; ++b) {
            uint32_t af[2][4];
            float dw[2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint32_t base = wq + (uint32_t)((2 * rs + mt) * 4096);
                af[mt][0] = lds32(base + 256u * (2 * b) + 16u * gq + 4u * cq);
                af[mt][1] = lds32(base + 256u * (2 * b) + 16u * (gq + 8) + 4u * cq);
                af[mt][2] = lds32(base + 256u * (2 * b + 1) + 16u * gq + 4u * cq);
                af[mt][3] = lds32(base + 256u * (2 * b + 1) + 16u * (gq + 8) + 4u * cq);
                const uint32_t sc = wsc + (uint32_t)((2 * rs + mt) * 256) + 2u * b;
                dw[mt][0] = __half2float(__ushort_as_half((unsigned short)lds16(sc + 16u * gq)));
                dw[mt][1] = __half2float(__ushort_as_half((unsigned short)lds16(sc + 16u * (gq + 8))));
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int ti = 32 * ts + 8 * nt + gq;  // this lane's B column (token)
                const uint32_t ta = aq + (uint32_t)(ti * QG_AROW) + 32u * b + 4u * cq;
                const uint32_t b0 = lds32(ta), b1 = lds32(ta + 16u);
                const int tc = 32 * ts + 8 * nt + 2 * cq;  // this lane's accumulator tokens tc, tc + 1
                const float da0 = __uint_as_float(lds32(ad + (uint32_t)(tc * 32) + 4u * b));
                const float da1 = __uint_as_float(lds32(ad + (uint32_t)((tc + 1) * 32) + 4u * b));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    int c[4];
                    mma_k32_s8s8(c, af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
                    // c: (row gq, tokens tc, tc+1), (row gq+8, tokens tc, tc+1)
                    y[mt][nt][0] = fmaf(dw[mt][0] * da0, small_int_to_float(c[0]), y[mt][nt][0]);
                    y[mt][nt][1] = fmaf(dw[mt][0] * da1, small_int_to_float(c[1]), y[mt][nt][1]);
                    y[mt][nt][2] = fmaf(dw[mt][1] * da0, small_int_to_float(c[2]), y[mt][nt][2]);
                    y[mt][nt][3] = fmaf(dw[mt][1] * da1, small_int_to_float(c[3]), y[mt][nt][3]);
                }
            }
        }
    }
    cp_async_wait<0>();
    // outputs y[token][row]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t n = g0 * 16 + 32 * rs + 16 * mt + gq + 8 * (i >> 1);
                const int64_t t = t0 + 32 * ts + 8 * nt + 2 * cq + (i & 1);
                if (n < p.N && t < p.M) p.y[t * p.N + n] = y[mt][nt][i];
            }
}

}  // namespace

cudaError_t launch_gemm_q8_0(const void *packed, int64_t N, int64_t K, const float *d_a, const int8_t *q_a, int64_t M,
                             float *y, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    const uint64_t chunks = (uint64_t)row_groups(N) * (uint64_t)nsb;
    Q8GemmParams p;
    p.qs = static_cast<const uint8_t *>(packed);
    p.sc = p.qs + align256(chunks * 4096);
    p.d_a = d_a;
    p.q_a = q_a;
    p.y = y;
    p.N = N;
    p.K = K;
    p.M = M;
    p.nsb = nsb;
    p.groups = row_groups(N);
    const int64_t t_tiles = (M + QG_BT - 1) / QG_BT, n_tiles = (N + QG_BM - 1) / QG_BM;
    if (t_tiles * n_tiles > (int64_t)INT32_MAX) return cudaErrorNotSupported;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(q8_0_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QG_SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(t_tiles * n_tiles));
    cfg.blockDim = dim3(QG_THREADS);
    cfg.dynamicSmemBytes = QG_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q8_0_gemm_kernel, p);
}

}  // namespace kq
