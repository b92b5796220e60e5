// kq_gemm.cu - tensor-core prefill GEMM (tcgen05) and its MoE grouped form.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
//
// The contraction the page folds in int32 runs on the fp16 tensor pipe with
// exact small integers (sm_103a has no integer tcgen05.mma):
//   - a pre-pass turns the Q8_K activations of the M token rows into an fp16
//     image of q8 (exact, |q8| <= 127), of the per-16 bsums (exact, <= 2032)
//     and a transposed copy of d8, in the caller's workspace;
//   - each block owns 128 weight rows x up to 128 tokens; per superblock its
//     unpack warps expand the packed weights once into shared memory as fp16
//     w' = sc*q with the sub-scale folded in (Q4_K <= 945, Q5_K <= 1953:
//     exact): the kq v3 panel scratch, unpacked once per token block;
//     Q6_K's w' = sc*(q-32) is one exact fp16 FMA for |sc| <= 62, and when a tile holds a
//     larger sub-scale the weight is split into two exact planes,
//     sc*(v - (v&1)) (even, |.| <= 4096) and sc*(v&1), both multiplied into
//     the same accumulator;
//   - tcgen05.mma kind::f16 accumulates I = sum w'*q8 (the page's isum, or
//     iacc - 32*bacc for Q6_K) in fp32 TMEM; for Q4_K/Q5_K a second K=16 MMA
//     of the sub-mins (duplicated per 16) against the bsums gives msum;
//   - the epilogue folds once per superblock, y += d8*(d*I - dmin*msum), in
//     fp32 registers ([kq-arc], "The pieces": one float fold per superblock).
// The grouped (MoE) form runs one block per SM over a list of tiles (see the
// tile comment below), so short expert tiles do not pay a block's start-up
// and drain each.
// The fp32 accumulator is exact while every partial sum stays below 2^24 in
// magnitude (true for realistic activations; at adversarial extremes the
// sum is rounded like the fold's own float(isum)).
//
// Warp roles (14 warps): 0 TMA producer of the activation tiles, 1 MMA issuer
// (and TMEM owner); Q4_K/Q5_K: 2..5 weight unpack (thread = weight row),
// 6..13 epilogue (thread = row x 64 token columns, y in registers); Q6_K,
// whose unpack is the longer chain: 2..9 weight unpack (two threads per row,
// one 64-wide K sub-tile each), 10..13 epilogue (thread = row x every token
// column, y accumulated in TMEM columns 128..255, which Q6_K's missing mins
// leave free).  TMEM lane quadrant = warp % 4.  Stages are half superblocks (K = 128): an A ring of 2 slots,
// a B ring of 3 (Q6_K: 2); accumulators I and msum double-buffered by
// superblock parity.  Every mbarrier wait is bounded; on timeout the block
// records KQ_ERR_TIMEOUT in the device status word and winds down.
#include "kq_internal.h"
#include "kq_sm100.cuh"

#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <mutex>

namespace kq {

__device__ int g_status = 0;

using namespace sm100;

constexpr int BM = 128;      // weight rows per tile (MMA M)
constexpr int BT = 128;      // tokens per tile (MMA N, at most)
constexpr int NTHREADS = 448;
constexpr int W_TMA = 0, W_MMA = 1, W_UNPACK = 2;
constexpr int TILE_CAP = 128;          // grouped: most tiles one block runs
constexpr int MAX_GROUPED_E = 1024;    // grouped: most experts (more take the CUDA-core kernel)
// first epilogue warp: Q4_K/Q5_K 4 unpack + 8 epilogue warps; Q6_K 8 unpack
// (two threads per weight row) + 4 epilogue warps that keep y in TMEM
template <int F> constexpr int w_epi() { return F == FMT_Q6_K ? 10 : 6; }
template <int F> constexpr int n_unpack() { return w_epi<F>() - W_UNPACK; }
template <int F> constexpr int n_epi() { return NTHREADS / 32 - w_epi<F>(); }

template <int F>
struct Cfg {
    static constexpr bool kMins = F != FMT_Q6_K;
    static constexpr int NB = F == FMT_Q6_K ? 2 : 3;              // B ring slots
    static constexpr int A_SLOT = F == FMT_Q6_K ? 65536 : 32768;  // 2 sub-tiles (x2 planes for Q6_K)
    static constexpr int B_SUB = BT * 128;                         // one 64-wide K sub-tile of tokens
    static constexpr int B_SLOT = 2 * B_SUB + (kMins ? BT * 32 : 0);
    static constexpr int OFF_A = 0;
    static constexpr int OFF_AMIN = 2 * A_SLOT;
    static constexpr int OFF_B = OFF_AMIN + (kMins ? BM * 32 : 0);
    static constexpr int OFF_SD = OFF_B + NB * B_SLOT;            // s_d, s_dmin [2][BM]
    static constexpr int OFF_D8 = OFF_SD + 2 * 2 * BM * 4;        // per epilogue warp [64] floats
    static constexpr int OFF_BAR = OFF_D8 + 8 * 64 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr int OFF_TILES = OFF_MISC + 128;              // grouped: the block's tile list
    static constexpr int OFF_OFFS = OFF_TILES + TILE_CAP * 16;    // grouped: the row offsets [E + 1]
    // grouped Q4_K: each unpack thread's row bytes for a half superblock (4
    // qs pieces + the scale block, 16 B each) staged by cp.async RS - 1 halves
    // ahead, [RS][RCH chunks][BM rows] x 16 B (rows contiguous per chunk: no
    // bank conflicts)
    static constexpr int RS = F == FMT_Q4_K ? 3 : 0, RCH = 5;
    static constexpr int OFF_RAW = OFF_OFFS + (MAX_GROUPED_E + 4) * 4;
    static constexpr int SMEM = OFF_RAW + RS * RCH * BM * 16 + 1024;  // + alignment slack
    static constexpr int SMEM_DENSE = OFF_RAW + 1024;                  // the dense kernel stages no rows
    static_assert(SMEM <= 232448, "shared memory per block");
    static_assert(OFF_RAW % 16 == 0, "cp.async needs 16-byte aligned destinations");
    static_assert(OFF_B % 1024 == 0, "B tiles need 1024-byte alignment");
    static_assert(B_SLOT % 1024 == 0, "B slots need 1024-byte alignment");
};

// barrier indices
enum { BAR_FULL_A = 0, BAR_EMPTY_A = 2, BAR_FULL_B = 4, BAR_EMPTY_B = 7, BAR_ACC_FULL = 10, BAR_ACC_EMPTY = 12,
       BAR_SD_FULL = 14, BAR_MMA_DONE = 16, BAR_TILES = 17 };

struct GemmParams {
    const uint8_t *packed;
    uint64_t expert_bytes;
    int64_t N, K, nsb, M;
    const int32_t *offsets;  // grouped: [E+1]; dense: nullptr
    int64_t E;
    const float *d8t;        // workspace: d8 transposed [nsb][Mp]
    int64_t Mp;
    float *y;
};

__device__ __forceinline__ void set_timeout() { atomicExch(&g_status, 1); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t h2_splat(float v) {
    const unsigned short h = __half_as_ushort(__float2half_rn(v));
    return static_cast<uint32_t>(h) | (static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// byte pairs (0,1), (2,3) of a word, each as the low byte of one fp16 lane
// whose high byte is 0x64 (the fp16 1024 + byte)
constexpr uint32_t SEL_01 = 0x4140, SEL_23 = 0x4342;
constexpr uint32_t MAGIC = 0x64646464u;

// ---------------------------------------------------------------------------
// Unpack of one weight row x one 64-wide K sub-tile of a half superblock into
// the A operand (128-byte swizzled K-major fp16 rows).  `a_row` is the shared
// address of the sub-tile base; the row's 8 chunks of 8 fp16 are written at
// sw128_offset(r, 8q).

// Q4_K/Q5_K: sub-tile = chunk c of the superblock (64 elements): elements
// 64c + l (low nibbles of qs[32c + l], sub-scale sc_2c) at K 0..31 and
// 64c + 32 + l (high nibbles, sc_2c+1) at K 32..63; Q5_K ORs bit 2c / 2c+1 of
// qh[l] in as value 16.  w' = q*sc is built exactly in fp16 as
// (1024 + q)*sc - 1024*sc (low) and (1024 + 16q)*(sc/16) - 64*sc (high).
template <int F>
__device__ __forceinline__ void unpack_q45(uint32_t a_tile, int r, const uint32_t (&qs)[8], const uint32_t (&qh)[8],
                                           int c, int sc_lo, int sc_hi) {
    const uint32_t s_lo = h2_splat((float)sc_lo), o_lo = h2_splat(-1024.0f * sc_lo);
    const uint32_t s_hi = h2_splat(sc_hi * 0.0625f), o_hi = h2_splat(-64.0f * sc_hi);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // K 8q .. 8q+7: bytes 8q .. 8q+7 of the chunk
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const uint32_t word = qs[2 * q + w];
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t sel = pr ? SEL_23 : SEL_01;
                const uint32_t x = prmt(word, MAGIC, sel);
                uint32_t l = x & 0xFF0FFF0Fu, h = x & 0xFFF0FFF0u;
                if constexpr (F == FMT_Q5_K) {
                    const uint32_t hb = prmt(qh[2 * q + w], 0u, pr ? 0x4342u : 0x4140u) & 0x00FF00FFu;
                    const int b = 2 * c;  // low nibble's fifth bit
                    l |= (b <= 4 ? (hb << (4 - b)) : (hb >> (b - 4))) & 0x00100010u;
                    // high nibble's fifth bit (2c+1) lands on bit 8: value 256 = 16 * 16
                    h |= (hb << (7 - b)) & 0x01000100u;
                }
                lo[2 * w + pr] = h2_fma(l, s_lo, o_lo);
                hi[2 * w + pr] = h2_fma(h, s_hi, o_hi);
            }
        }
        sts128(a_tile + sw128_offset(r, 8 * q), lo[0], lo[1], lo[2], lo[3]);
        sts128(a_tile + sw128_offset(r, 32 + 8 * q), hi[0], hi[1], hi[2], hi[3]);
    }
}

// Q6_K: sub-tile j of half h holds groups t = 2j (K 0..31) and 2j+1 (K 32..63)
// of the half: element 128h + 32t + l is the low (t < 2) or high (t >= 2)
// nibble of ql[64h + 32(t&1) + l] with bits 2t..2t+1 of qh[32h + l] on top,
// sub-scale sc[8h + 2t + l/16] (byte 2(t - 2j) + l/16 of `scw`).  The 6-bit
// q of four elements is assembled in one word, then spread into fp16 lanes
// 1024 + q.  v = q - 32: P1 = v*sc = (1024 + q)*sc - 1056*sc in one fp16 FMA,
// exact for |sc| <= 62 (1056*sc and the result are exact fp16 integers); with
// `split` (some |sc| > 62), P1 = (v - (v&1))*sc and P2 = (v&1)*sc, each exact.
// `zero2` writes zeros to this thread's P2 rows instead.
__device__ __forceinline__ void unpack_q6(uint32_t a_tile, uint32_t a2_tile, int r, const uint32_t (&ql)[16],
                                          const uint32_t (&qh)[8], uint32_t scw, int j, bool split, bool zero2) {
    const uint32_t off1056 = h2_splat(1056.0f);
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        const int t = 2 * j + tt;
        // the group's two sub-scales (l < 16, l >= 16) and -1056 * each
        uint32_t s2v[2], c2v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int scv = (int)(int8_t)((scw >> (8 * (2 * tt + u))) & 0xFF);
            s2v[u] = h2_splat((float)scv);
            c2v[u] = h2_splat(-1056.0f * (float)scv);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // K 32tt + 8q .. +7: l = 8q .. 8q+7
            const uint32_t s2 = s2v[q >> 1], c2 = c2v[q >> 1];
            uint32_t p1[4], p2[4];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const uint32_t lword = ql[8 * (t & 1) + 2 * q + w];
                const uint32_t nib = ((t >= 2) ? (lword >> 4) : lword) & 0x0F0F0F0Fu;
                const uint32_t q6 = nib | (((qh[2 * q + w] >> (2 * t)) & 0x03030303u) << 4);  // four q, 0..63
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const uint32_t x = prmt(q6, MAGIC, pr ? SEL_23 : SEL_01);  // fp16 1024 + q
                    if (split) {
                        const uint32_t odd = x & 0x00010001u;
                        p1[2 * w + pr] = h2_mul(h2_sub(x ^ odd, off1056), s2);
                        p2[2 * w + pr] = h2_mul(odd * 0x3C00u, s2);     // fp16 1.0 in each odd lane
                    } else {
                        p1[2 * w + pr] = h2_fma(x, s2, c2);
                        p2[2 * w + pr] = 0u;
                    }
                }
            }
            sts128(a_tile + sw128_offset(r, 32 * tt + 8 * q), p1[0], p1[1], p1[2], p1[3]);
            if (split || zero2) sts128(a2_tile + sw128_offset(r, 32 * tt + 8 * q), p2[0], p2[1], p2[2], p2[3]);
        }
    }
}

// Raw packed bytes one unpack thread (one weight row) converts for one half
// superblock (K 128h .. 128h + 127).
struct RawQ4 { uint32_t qs[16]; uint4 hdr; };              // qs[64h .. 64h+64)
struct RawQ5 { uint32_t qs[16]; uint32_t qh[8]; uint4 hdr; };
struct RawQ6 { uint32_t ql[16]; uint32_t qh[8]; uint32_t sc[2]; uint32_t d; };  // ql/qh/sc of half h
template <int F> struct RawOf;
template <> struct RawOf<FMT_Q4_K> { using T = RawQ4; };
template <> struct RawOf<FMT_Q5_K> { using T = RawQ5; };
template <> struct RawOf<FMT_Q6_K> { using T = RawQ6; };

__device__ __forceinline__ void ld16w(uint32_t *dst, const uint8_t *src) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
    dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
}
// half h of row n's superblock sb, from the grp16 image (kq_device.cuh)
__device__ __forceinline__ void load_raw(RawQ4 &r, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int h) {
    const uint64_t ch = chunk_of(n, sb, nsb);
    const int rr = (int)(n % GROUP_ROWS);
    const uint8_t *q = P.p0 + ch * 2048 + 16 * (rr + 16 * h);
#pragma unroll
    for (int i = 0; i < 4; ++i) ld16w(r.qs + 4 * i, q + 512 * i);
    r.hdr = __ldg(reinterpret_cast<const uint4 *>(P.p1 + ch * 256 + 16 * rr));
}
__device__ __forceinline__ void load_raw(RawQ5 &r, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int h) {
    const uint64_t ch = chunk_of(n, sb, nsb);
    const int rr = (int)(n % GROUP_ROWS);
    const uint8_t *q = P.p0 + ch * 2048 + 16 * (rr + 16 * h);
#pragma unroll
    for (int i = 0; i < 4; ++i) ld16w(r.qs + 4 * i, q + 512 * i);
    ld16w(r.qh, P.p1 + ch * 512 + 16 * rr);
    ld16w(r.qh + 4, P.p1 + ch * 512 + 256 + 16 * rr);
    r.hdr = __ldg(reinterpret_cast<const uint4 *>(P.p2 + ch * 256 + 16 * rr));
}
__device__ __forceinline__ void load_raw(RawQ6 &r, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int h) {
    const uint64_t ch = chunk_of(n, sb, nsb);
    const int rr = (int)(n % GROUP_ROWS);
    const uint8_t *l = P.p0 + ch * 2048 + 16 * (rr + 16 * h);
#pragma unroll
    for (int i = 0; i < 4; ++i) ld16w(r.ql + 4 * i, l + 512 * i);
    ld16w(r.qh, P.p1 + ch * 1024 + 16 * (rr + 16 * h));
    ld16w(r.qh + 4, P.p1 + ch * 1024 + 512 + 16 * (rr + 16 * h));
    const uint2 sc = __ldg(reinterpret_cast<const uint2 *>(P.p2 + ch * 256 + 16 * rr + 8 * h));
    r.sc[0] = sc.x;
    r.sc[1] = sc.y;
    r.d = __ldg(reinterpret_cast<const unsigned short *>(P.p3 + ch * 32) + rr);
}

// ---------------------------------------------------------------------------
// Output tiles: 128 weight rows x up to 128 tokens of one expert.
//
// Dense: one block per tile, tile i = blockIdx.x of t_tiles x w_tiles (token
// tile fastest, so neighbouring blocks share a weight panel).
//
// Grouped: a block per SM (at most), each running a list of tiles, and every
// role walks the same list, so the rings, the TMEM buffers and their phases
// run on across tiles (the unpack of a tile's first superblock overlaps the
// epilogue of the previous tile).  Tile indices: i < E * w_tiles is the first
// token tile of expert i / w_tiles, rows [o_e, min(o_e+1, o_e + 128)); the
// experts' later token tiles (past their first 128 rows) follow, in expert
// order.  Block b takes i = b, b + grid, ...: its first tile is known
// without the offsets, so its unpack starts before the dependency wait and
// the tile runs even when the expert has no rows (no MMA, no activation
// copy, no stores); its later tiles without rows are left out of the list.
// The TMA warp builds the list in shared memory once (the offsets staged
// there first), and the other roles read it from there.
struct Tile {
    int n0, t0, t_end;
    int e, ntok, n_mma;
};

__device__ __forceinline__ int w_tiles_of(const GemmParams &p) { return (int)((p.N + BM - 1) / BM); }

__device__ __forceinline__ void finish_tile(Tile &t) {
    const int nt = t.t_end - t.t0;
    t.ntok = nt < 0 ? 0 : nt;
    t.n_mma = (t.ntok + 15) & ~15;
}

// Dense tile of this block.
__device__ __forceinline__ Tile dense_tile(const GemmParams &p) {
    const int t_tiles = (int)((p.M + BT - 1) / BT);
    const int i = (int)blockIdx.x;
    Tile t;
    t.e = 0;
    t.n0 = (i / t_tiles) * BM;
    t.t0 = (i % t_tiles) * BT;
    t.t_end = (t.t0 + BT < p.M) ? t.t0 + BT : (int)p.M;
    finish_tile(t);
    return t;
}

// Grouped list entry k (written by build_tile_list).
__device__ __forceinline__ Tile list_tile(const int4 *list, int k) {
    const int4 v = list[k];
    Tile t;
    t.e = v.x;
    t.n0 = v.y;
    t.t0 = v.z;
    t.t_end = v.w;
    finish_tile(t);
    return t;
}

// Rows [a, b) of expert e from the staged offsets, clamped to [0, M].
__device__ __forceinline__ void expert_rows(const int *offs, int M, int e, int &a, int &b) {
    a = offs[e];
    b = offs[e + 1];
    a = a < 0 ? 0 : (a > M ? M : a);
    b = b < a ? a : (b > M ? M : b);
}

// Exclusive warp prefix sum of v; *total gets the warp's sum.
__device__ __forceinline__ int warp_excl_sum(int v, int lane, int *total) {
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    return incl - v;
}

// Grouped: the block's tile list (warp-collective, after the dependency
// wait); returns the number of tiles.  list entries: {e, n0, t0, t_end}.
__device__ int build_tile_list(const GemmParams &p, int *offs, int4 *list, int lane) {
    const int E = (int)p.E, M = (int)p.M, w_tiles = w_tiles_of(p);
    for (int i = lane; i <= E; i += 32) offs[i] = p.offsets[i];
    __syncwarp();
    const int64_t S = (int64_t)E * w_tiles;
    const int64_t bid = blockIdx.x, grid = gridDim.x;
    int count = 0;
    // first token tiles: i = bid + k * grid < S
    const int n_first = bid < S ? (int)((S - 1 - bid) / grid + 1) : 0;
    for (int k0 = 0; k0 < n_first; k0 += 32) {
        const int k = k0 + lane;
        int4 v = make_int4(0, 0, 0, 0);
        bool run = false;
        if (k < n_first) {
            const int64_t i = bid + (int64_t)k * grid;
            int a, b;
            v.x = (int)(i / w_tiles);
            v.y = (int)(i % w_tiles) * BM;
            expert_rows(offs, M, v.x, a, b);
            v.z = a;
            v.w = (a + BT < b) ? a + BT : b;
            run = k == 0 || v.w > v.z;
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, run);
        const int pos = count + __popc(m & ((1u << lane) - 1));
        if (run && pos < TILE_CAP) list[pos] = v;
        count += __popc(m);
    }
    // later token tiles: index S + j * w_tiles + wt for the j-th later token
    // tile in expert order; this block takes those congruent to bid
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        int a = 0, b = 0, later = 0;
        if (e < E) {
            expert_rows(offs, M, e, a, b);
            const int tiles = (b - a + BT - 1) / BT;
            later = tiles > 1 ? tiles - 1 : 0;
        }
        int sum;
        const int j0 = base + warp_excl_sum(later, lane, &sum);
        // this lane's index range [lo, hi) and the first index congruent to bid
        const int64_t lo = S + (int64_t)j0 * w_tiles, hi = lo + (int64_t)later * w_tiles;
        const int64_t first = lo + ((bid - lo) % grid + grid) % grid;
        const int n = first < hi ? (int)((hi - 1 - first) / grid + 1) : 0;
        int n_all;
        const int pos0 = count + warp_excl_sum(n, lane, &n_all);
        for (int q = 0; q < n; ++q) {
            const int64_t o = first + (int64_t)q * grid - S;
            const int j = (int)(o / w_tiles);
            const int t0 = a + (1 + j - j0) * BT;
            if (pos0 + q < TILE_CAP)
                list[pos0 + q] = make_int4(e, (int)(o % w_tiles) * BM, t0, (t0 + BT < b) ? t0 + BT : b);
        }
        count += n_all;
        base += sum;
    }
    return count < TILE_CAP ? count : TILE_CAP;
}

// Start streaming a tile's weight rows (contiguous in every plane) into L2.
template <int F>
__device__ __forceinline__ void prefetch_tile(const GemmParams &p, const Tile &t) {
    const Planes P = make_planes(F, p.packed + (uint64_t)t.e * p.expert_bytes, p.N, p.nsb);
    int u[4];
    plane_unit_bytes(F, u);
    const int64_t rows = row_groups(p.N) * GROUP_ROWS;
    const int64_t n0 = t.n0, r1 = (n0 + BM < rows ? n0 + BM : rows);
    const uint8_t *base[4] = {P.p0, P.p1, P.p2, P.p3};
    for (int q = 0; q < 4; ++q)
        if (u[q] && r1 > n0) prefetch_l2_bulk(base[q] + (uint64_t)n0 * p.nsb * u[q], (uint64_t)(r1 - n0) * p.nsb * u[q]);
}

template <int F, bool G>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a16, const __grid_constant__ CUtensorMap map_b16,
                const GemmParams p) {
    using C = Cfg<F>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    float *s_d = reinterpret_cast<float *>(smem + C::OFF_SD);
    float *s_dmin = s_d + 2 * BM;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);  // [0] tmem base, [1] tile count
    int *s_flag = reinterpret_cast<int *>(misc + 8);                     // Q6_K split flags [2 halves][8 warps]
    int4 *s_list = reinterpret_cast<int4 *>(smem + C::OFF_TILES);        // grouped tile list

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = p.nsb;
    // Programmatic dependent launch: the next kernel may be scheduled now.
    // This grid reads what earlier kernels wrote (the activation image, the
    // scales, the expert offsets) only after griddepcontrol.wait; the unpack
    // warps, which read only the packed weights, start before it.
    griddep_launch_dependents();

    // grouped: blocks below E * w_tiles start on the first token tile of an
    // expert, known without the offsets
    const bool static_first = !G || (int64_t)blockIdx.x < p.E * w_tiles_of(p);

    // ---- setup
    if (threadIdx.x == 0) {
        mbar_init(&bar[BAR_FULL_A + 0], n_unpack<F>());
        mbar_init(&bar[BAR_FULL_A + 1], n_unpack<F>());
        mbar_init(&bar[BAR_EMPTY_A + 0], 1);
        mbar_init(&bar[BAR_EMPTY_A + 1], 1);
        for (int i = 0; i < C::NB; ++i) {
            mbar_init(&bar[BAR_FULL_B + i], 1);
            mbar_init(&bar[BAR_EMPTY_B + i], 1);
        }
        mbar_init(&bar[BAR_ACC_FULL + 0], 1);
        mbar_init(&bar[BAR_ACC_FULL + 1], 1);
        mbar_init(&bar[BAR_ACC_EMPTY + 0], n_epi<F>());
        mbar_init(&bar[BAR_ACC_EMPTY + 1], n_epi<F>());
        mbar_init(&bar[BAR_SD_FULL + 0], 4);
        mbar_init(&bar[BAR_SD_FULL + 1], 4);
        mbar_init(&bar[BAR_MMA_DONE], 1);
        mbar_init(&bar[BAR_TILES], 1);
        mbar_fence_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // TMEM columns: I[b] at 256b, msum[b] at 256b + 128.  Buffer b and the
    // phases follow g, the block's count of superblock steps over all tiles.
    bool ok = true;

    if (warp == W_TMA) {
        // ------------------------------------------------ activation tiles
        griddep_wait();
        int ntiles = 1;
        if constexpr (G) {
            ntiles = build_tile_list(p, reinterpret_cast<int *>(smem + C::OFF_OFFS), s_list, lane);
            __threadfence_block();
            __syncwarp();
            if (lane == 0) {
                misc[1] = (uint32_t)ntiles;
                mbar_arrive(&bar[BAR_TILES]);
            }
        }
        int64_t use = 0;
        if (lane == 0) {
            tma_prefetch_desc(&map_a16);
            if (C::kMins) tma_prefetch_desc(&map_b16);
            if (ntiles > 0) prefetch_tile<F>(p, G ? list_tile(s_list, 0) : dense_tile(p));
            for (int k = 0; k < ntiles && ok; ++k) {
                const Tile t = G ? list_tile(s_list, k) : dense_tile(p);
                // the next tile's weights stream into L2 while this one runs
                if (k + 1 < ntiles) prefetch_tile<F>(p, list_tile(s_list, k + 1));
                for (int64_t sb = 0; sb < nsb && ok && t.ntok > 0; ++sb) {
                    for (int h = 0; h < 2 && ok; ++h, ++use) {
                        const int slot = (int)(use % C::NB);
                        const uint32_t par = (uint32_t)((use / C::NB) & 1);
                        if (!mbar_wait(&bar[BAR_EMPTY_B + slot], par ^ 1)) { ok = false; break; }
                        uint8_t *bs = smem + C::OFF_B + slot * C::B_SLOT;
                        const bool mins = C::kMins && h == 0;
                        mbar_arrive_expect_tx(&bar[BAR_FULL_B + slot], 2 * C::B_SUB + (mins ? BT * 32 : 0));
                        const int k0 = (int)(sb * QK + 128 * h);
                        tma_load_2d(bs, &map_a16, k0, t.t0, &bar[BAR_FULL_B + slot]);
                        tma_load_2d(bs + C::B_SUB, &map_a16, k0 + 64, t.t0, &bar[BAR_FULL_B + slot]);
                        if (mins) tma_load_2d(bs + 2 * C::B_SUB, &map_b16, (int)(sb * 16), t.t0, &bar[BAR_FULL_B + slot]);
                    }
                }
            }
            if (!ok) {
                set_timeout();
                // let the copies already issued land before the block exits
                for (int s = 0; s < C::NB; ++s)
                    if (use > s) mbar_wait(&bar[BAR_FULL_B + ((use - 1 - s) % C::NB)], (uint32_t)(((use - 1 - s) / C::NB) & 1));
            }
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------ MMA issue
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        const uint32_t amin = smem_u32(smem + C::OFF_AMIN);
        const uint32_t b_base = smem_u32(smem + C::OFF_B);
        int64_t g = 0, use = 0;
        if (lane == 0) {
            int ntiles = 1;
            if constexpr (G) {
                ok = mbar_wait(&bar[BAR_TILES], 0);
                ntiles = ok ? (int)misc[1] : 0;
            }
            for (int k = 0; k < ntiles && ok; ++k) {
                const Tile t = G ? list_tile(s_list, k) : dense_tile(p);
                const uint32_t idesc = idesc_f16_f32(BM, t.n_mma > 0 ? t.n_mma : 16);
                for (int64_t sb = 0; sb < nsb && ok; ++sb, ++g) {
                    const int b = (int)(g & 1);
                    const uint32_t acc_i = tmem + 256 * b, acc_m = tmem + 256 * b + 128;
                    if (!mbar_wait(&bar[BAR_ACC_EMPTY + b], (uint32_t)(((g >> 1) & 1) ^ 1))) { ok = false; break; }
                    tc_fence_after();
                    for (int h = 0; h < 2; ++h) {
                        const int slot = (int)(use % C::NB);
                        if (!mbar_wait(&bar[BAR_FULL_A + h], (uint32_t)(g & 1)) ||
                            (t.ntok > 0 && !mbar_wait(&bar[BAR_FULL_B + slot], (uint32_t)((use / C::NB) & 1)))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (t.ntok == 0) {  // a first tile without rows: release the A slot unread
                            mbar_arrive(&bar[BAR_EMPTY_A + h]);
                            continue;
                        }
                        const uint32_t a_slot = a_base + h * C::A_SLOT;
                        const uint32_t b_slot = b_base + slot * C::B_SLOT;
                        int planes = 1;
                        if constexpr (F == FMT_Q6_K) {
                            int any = 0;
                            for (int w = 0; w < n_unpack<F>(); ++w) any |= s_flag[8 * h + w];
                            planes = any ? 2 : 1;
                        }
                        for (int pl = 0; pl < planes; ++pl) {
                            for (int j = 0; j < 2; ++j) {
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t ad =
                                        smem_desc(a_slot + pl * 32768 + j * 16384 + 32 * kk, 16, 1024, SWZ_128B);
                                    const uint64_t bd = smem_desc(b_slot + j * C::B_SUB + 32 * kk, 16, 1024, SWZ_128B);
                                    umma_f16(acc_i, ad, bd, idesc, (h | j | kk | pl) != 0);
                                }
                            }
                        }
                        if (C::kMins && h == 0) {
                            const uint64_t ad = smem_desc(amin, 16, 256, SWZ_32B);
                            const uint64_t bd = smem_desc(b_slot + 2 * C::B_SUB, 16, 256, SWZ_32B);
                            umma_f16(acc_m, ad, bd, idesc, 0);
                        }
                        umma_commit(&bar[BAR_EMPTY_A + h]);
                        umma_commit(&bar[BAR_EMPTY_B + slot]);
                        ++use;
                    }
                    if (!ok) break;
                    if (t.ntok > 0) umma_commit(&bar[BAR_ACC_FULL + b]);
                    else mbar_arrive(&bar[BAR_ACC_FULL + b]);
                }
            }
            // all MMAs issued by this thread complete before TMEM is released
            umma_commit(&bar[BAR_MMA_DONE]);
            if (!mbar_wait(&bar[BAR_MMA_DONE], 0)) ok = false;
            if (!ok) set_timeout();
        }
    } else if (warp < w_epi<F>()) {
        // ------------------------------------------------ weight unpack
        const int uw = warp - W_UNPACK;          // 0..3 (Q6_K 0..7)
        const int r = 32 * (uw & 3) + lane;      // tile row
        const int my_jj = uw >> 2;               // Q6_K: this thread's K sub-tile of each half
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        if constexpr (F == FMT_Q4_K && G) {
        // ---- grouped Q4_K: the row's bytes of each half superblock arrive by
        // cp.async in this thread's shared-memory ring, RS - 1 halves ahead:
        // the experts' weights stream from HBM, and the register prefetch of
        // one half left the warp waiting out an HBM latency per half (MoE gate
        // 116 -> 101 us).  The dense GEMM, whose weight panels are re-read by
        // its token tiles from L2, keeps the register prefetch (the ring
        // measured 3 % slower there).
        const uint32_t raw = smem_u32(smem + C::OFF_RAW);
        auto slot_addr = [&](int slot, int c) -> uint32_t { return raw + (uint32_t)(((slot * C::RCH + c) * BM + r) * 16); };
        const int nstage = 2 * (int)nsb;
        int ntiles = -1;  // the list length, read once it is needed
        // tile k's expert and first row; false past the last tile
        auto tile_rows = [&](int k, int &e, int &n0) -> bool {
            if (k == 0 && static_first) {
                const int wt = w_tiles_of(p);
                e = (int)(blockIdx.x / wt);
                n0 = (int)(blockIdx.x % wt) * BM;
                return true;
            }
            if (ntiles < 0) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0))) {
                    ok = false;
                    ntiles = 0;
                    return false;
                }
                ntiles = (int)misc[1];
            }
            if (k >= ntiles) return false;
            const int4 v = s_list[k];
            e = v.x;
            n0 = v.y;
            return true;
        };
        // copy cursor: tile kc, half-stage hc of it, this row's plane pointers
        int kc = 0, hc = 0;
        bool c_on = false;
        const uint8_t *cq = nullptr, *chd = nullptr;
        auto enter_tile = [&](int k) {
            int e, n0;
            c_on = tile_rows(k, e, n0);
            if (!c_on) return;
            const Planes P = make_planes(F, p.packed + (uint64_t)e * p.expert_bytes, p.N, nsb);
            const int64_t row = n0 + r < p.N ? n0 + r : p.N - 1;
            const uint64_t ch0 = chunk_of(row, 0, nsb);
            const int rr = (int)(row % GROUP_ROWS);
            cq = P.p0 + ch0 * 2048 + 16 * rr;
            chd = P.p1 + ch0 * 256 + 16 * rr;
        };
        auto issue = [&](int cs) {
            if (c_on) {
                const int sb = hc >> 1, h = hc & 1, slot = cs % C::RS;
                const uint8_t *q = cq + (uint64_t)sb * 2048 + 256 * h;
#pragma unroll
                for (int i = 0; i < 4; ++i) cp_async16(slot_addr(slot, i), q + 512 * i);
                cp_async16(slot_addr(slot, 4), chd + (uint64_t)sb * 256);
                if (++hc == nstage) {
                    hc = 0;
                    enter_tile(++kc);
                }
            }
            cp_async_commit();  // one group per half-stage, empty past the end
        };
        enter_tile(0);
        for (int i = 0; i < C::RS - 1; ++i) issue(i);
        int g = 0, hs_all = 0;
        for (int k = 0; ok; ++k) {
            int e_unused, n0_unused;
            if ((k > 0 || !static_first) && !tile_rows(k, e_unused, n0_unused)) break;
            for (int hs = 0; hs < nstage; ++hs, ++hs_all) {
                const int sb = hs >> 1, gg = g + sb, h = hs & 1;
                issue(hs_all + C::RS - 1);          // into the slot read one half-stage ago
                cp_async_wait<C::RS - 1>();          // this half-stage's group has landed
                const int slot = hs_all % C::RS;
                uint32_t qs[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = lds128(slot_addr(slot, i));
                    qs[4 * i] = v.x;
                    qs[4 * i + 1] = v.y;
                    qs[4 * i + 2] = v.z;
                    qs[4 * i + 3] = v.w;
                }
                const uint4 hdr = lds128(slot_addr(slot, 4));
                bool w_ok = mbar_wait(&bar[BAR_EMPTY_A + h], (uint32_t)((gg & 1) ^ 1));
                if (h == 0 && w_ok) w_ok = mbar_wait(&bar[BAR_ACC_EMPTY + (gg & 1)], (uint32_t)(((gg >> 1) & 1) ^ 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                const uint32_t a_slot = a_base + h * C::A_SLOT;
                const ScaleMin sm = unpack_scale_min(hdr);
                uint32_t qh0[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) qh0[i] = 0u;
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int cch = 2 * h + jj;  // chunk of the superblock; sub-blocks 2c, 2c+1
                    const uint32_t scw = cch < 2 ? sm.sc_lo : sm.sc_hi;
                    const int sc_lo = byte_of(scw, 2 * (cch & 1)), sc_hi = byte_of(scw, 2 * (cch & 1) + 1);
                    uint32_t qsc[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) qsc[i] = qs[8 * jj + i];
                    unpack_q45<F>(a_slot + jj * 16384, r, qsc, qh0, cch, sc_lo, sc_hi);
                }
                if (h == 0) {
                    // sub-mins duplicated per 16: K i of the mins operand holds m_{i/2}
                    const uint32_t amin = smem_u32(smem + C::OFF_AMIN);
                    uint32_t mw[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mw[i] = h2_splat((float)byte_of(i < 4 ? sm.m_lo : sm.m_hi, i & 3));
                    sts128(amin + sw32_offset(r, 0), mw[0], mw[1], mw[2], mw[3]);
                    sts128(amin + sw32_offset(r, 8), mw[4], mw[5], mw[6], mw[7]);
                    s_d[(gg & 1) * BM + r] = half_lo(hdr.x);
                    s_dmin[(gg & 1) * BM + r] = half_hi(hdr.x);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[BAR_FULL_A + h]);
                    if (h == 0) mbar_arrive(&bar[BAR_SD_FULL + (gg & 1)]);
                }
            }
            g += (int)nsb;
        }
        cp_async_wait<0>();  // no copy outlives the block
        if (!ok && lane == 0) set_timeout();
        } else {
        using Raw = typename RawOf<F>::T;
        Raw cur, nxt;
        // Q6_K: this thread's P2 rows of the half-0 / half-1 slot may be non-zero
        bool p2_dirty0 = true, p2_dirty1 = true;
        const int nstage = 2 * (int)nsb;
        int k = 0, g = 0, ntiles = -1;  // ntiles: grouped list length, read once it is needed
        Tile t;
        bool have = true;
        if constexpr (!G) {
            t = dense_tile(p);
        } else if (static_first) {
            const int w_tiles = w_tiles_of(p);
            t.e = (int)(blockIdx.x / w_tiles);
            t.n0 = (int)(blockIdx.x % w_tiles) * BM;
        } else {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0));
            ntiles = ok ? (int)misc[1] : 0;
            have = ntiles > 0;
            if (have) t = list_tile(s_list, 0);
        }
        // this thread's weight row of the tile
        int e_cur = t.e, row = t.n0 + r < p.N ? t.n0 + r : (int)p.N - 1;
        if (have) load_raw(cur, make_planes(F, p.packed + (uint64_t)e_cur * p.expert_bytes, p.N, nsb), row, 0, nsb, 0);
        while (have && ok) {
            bool have_n = false;
            int e_nxt = e_cur, n0_nxt = 0;
            const Planes P = make_planes(F, p.packed + (uint64_t)e_cur * p.expert_bytes, p.N, nsb);
            for (int hs = 0; hs < nstage; ++hs) {
                const int sb = hs >> 1, gg = g + sb;
                const int h = hs & 1;
                // the next half's bytes (the next tile's first half at the
                // end of a tile) are in flight while this one is converted
                if (hs + 1 < nstage) {
                    load_raw(nxt, P, row, (hs + 1) >> 1, nsb, (hs + 1) & 1);
                } else if constexpr (G) {
                    if (ntiles < 0) {
                        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0))) {
                            ok = false;
                            break;
                        }
                        ntiles = (int)misc[1];
                    }
                    have_n = k + 1 < ntiles;
                    if (have_n) {
                        const int4 v = s_list[k + 1];
                        e_nxt = v.x;
                        n0_nxt = v.y;
                        // the next tile's planes: this expert's, shifted by whole expert images
                        const int64_t delta = (int64_t)(e_nxt - e_cur) * (int64_t)p.expert_bytes;
                        const Planes Q{P.p0 + delta, P.p1 + delta, P.p2 + delta, P.p3 + delta};
                        const int rn = n0_nxt + r < p.N ? n0_nxt + r : (int)p.N - 1;
                        load_raw(nxt, Q, rn, 0, nsb, 0);
                    }
                }
                bool w_ok = mbar_wait(&bar[BAR_EMPTY_A + h], (uint32_t)((gg & 1) ^ 1));
                if (h == 0 && w_ok) w_ok = mbar_wait(&bar[BAR_ACC_EMPTY + (gg & 1)], (uint32_t)(((gg >> 1) & 1) ^ 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                const uint32_t a_slot = a_base + h * C::A_SLOT;
                float d = 0.0f, dmin = 0.0f;
                if constexpr (F == FMT_Q6_K) {
                    const uint32_t scj = my_jj ? cur.sc[1] : cur.sc[0];
                    bool big = false;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int v = (int)(int8_t)((scj >> (8 * i)) & 0xFF);
                        big |= (v > 62 || v < -62);
                    }
                    const unsigned any = __ballot_sync(0xFFFFFFFFu, big);
                    if (lane == 0) s_flag[8 * h + uw] = any ? 1 : 0;
                    const uint32_t a_tile = a_slot + my_jj * 16384;
                    const bool dirty = h ? p2_dirty1 : p2_dirty0;
                    unpack_q6(a_tile, a_tile + 32768, r, cur.ql, cur.qh, scj, my_jj, big, !big && dirty);
                    if (h) p2_dirty1 = big;
                    else p2_dirty0 = big;
                    d = __half2float(__ushort_as_half((unsigned short)cur.d));
                } else {
                    const ScaleMin sm = unpack_scale_min(cur.hdr);
                    uint32_t qh0[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if constexpr (F == FMT_Q5_K) qh0[i] = cur.qh[i];
                        else qh0[i] = 0u;
                    }
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int cch = 2 * h + jj;  // chunk of the superblock; sub-blocks 2c, 2c+1
                        const uint32_t scw = cch < 2 ? sm.sc_lo : sm.sc_hi;
                        const int sc_lo = byte_of(scw, 2 * (cch & 1)), sc_hi = byte_of(scw, 2 * (cch & 1) + 1);
                        uint32_t qsc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) qsc[i] = cur.qs[8 * jj + i];
                        unpack_q45<F>(a_slot + jj * 16384, r, qsc, qh0, cch, sc_lo, sc_hi);
                    }
                    if (h == 0) {
                        // sub-mins duplicated per 16: K i of the mins operand holds m_{i/2}
                        const uint32_t amin = smem_u32(smem + C::OFF_AMIN);
                        uint32_t mw[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) mw[i] = h2_splat((float)byte_of(i < 4 ? sm.m_lo : sm.m_hi, i & 3));
                        sts128(amin + sw32_offset(r, 0), mw[0], mw[1], mw[2], mw[3]);
                        sts128(amin + sw32_offset(r, 8), mw[4], mw[5], mw[6], mw[7]);
                    }
                    d = half_lo(cur.hdr.x);
                    dmin = half_hi(cur.hdr.x);
                }
                if (h == 0 && my_jj == 0) {
                    s_d[(gg & 1) * BM + r] = d;
                    s_dmin[(gg & 1) * BM + r] = dmin;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[BAR_FULL_A + h]);
                    if (h == 0 && my_jj == 0) mbar_arrive(&bar[BAR_SD_FULL + (gg & 1)]);
                }
                cur = nxt;
            }
            g += (int)nsb;
            ++k;
            have = have_n;
            e_cur = e_nxt;
            row = n0_nxt + r < p.N ? n0_nxt + r : (int)p.N - 1;
        }
        if (!ok && lane == 0) set_timeout();
        }
    } else if constexpr (F == FMT_Q6_K) {
        // ------------------------------------------------ epilogue, Q6_K
        // 4 warps, thread = weight row x every token column; y accumulates
        // in TMEM columns 128..255 (the mins slot of buffer 0, which Q6_K
        // does not use), read back once at the end of each tile
        const int ew = warp - w_epi<F>();    // 0..3
        const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
        const int r = 32 * quad + lane;
        float *s_d8 = reinterpret_cast<float *>(smem + C::OFF_D8) + 128 * ew;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16);
        const uint32_t y_tm = lane_addr + 128;
        griddep_wait();  // the scales are written by the kernels before this one
        int ntiles = 1;
        if constexpr (G) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0));
            ntiles = ok ? (int)misc[1] : 0;
        }
        int64_t g = 0;
        for (int k = 0; k < ntiles && ok; ++k) {
            const Tile t = G ? list_tile(s_list, k) : dense_tile(p);
            const int64_t n = t.n0 + r;
            const int nchunk = t.n_mma / 8;
            for (int64_t sb = 0; sb < nsb; ++sb) {
                const int64_t gg = g + sb;
                const int b = (int)(gg & 1);
                // the 128 token scales d8 of the superblock
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t tc = t.t0 + 32 * q + lane;
                    s_d8[32 * q + lane] = tc < t.t_end ? __ldg(p.d8t + sb * p.Mp + tc) : 0.0f;
                }
                __syncwarp();
                bool w_ok = mbar_wait(&bar[BAR_SD_FULL + b], (uint32_t)((gg >> 1) & 1));
                if (w_ok) w_ok = mbar_wait(&bar[BAR_ACC_FULL + b], (uint32_t)((gg >> 1) & 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float dd = s_d[b * BM + r];
                for (int c = 0; c < nchunk; ++c) {
                    uint32_t vi[8], vy[8];
                    tmem_ld8(lane_addr + 256 * b + 8 * c, vi);
                    if (sb > 0) tmem_ld8(y_tm + 8 * c, vy);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float yo = sb > 0 ? __uint_as_float(vy[i]) : 0.0f;
                        vy[i] = __float_as_uint(fmaf(s_d8[8 * c + i], dd * __uint_as_float(vi[i]), yo));
                    }
                    tmem_st8(y_tm + 8 * c, vy);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[BAR_ACC_EMPTY + b]);
            }
            if (!ok) break;
            tc_fence_after();
            for (int c = 0; c < nchunk; ++c) {
                uint32_t vy[8];
                tmem_ld8(y_tm + 8 * c, vy);
                tmem_wait_ld();
                if (n < p.N) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t tt = t.t0 + 8 * c + i;
                        if (tt < t.t_end) p.y[tt * p.N + n] = __uint_as_float(vy[i]);
                    }
                }
            }
            g += nsb;
        }
        if (!ok && lane == 0) set_timeout();
    } else {
        // ------------------------------------------------ epilogue
        const int ew = warp - w_epi<F>();    // 0..7
        const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
        const int ch = ew >> 2;              // token columns 64*ch .. +63
        const int r = 32 * quad + lane;
        float *s_d8 = reinterpret_cast<float *>(smem + C::OFF_D8) + 64 * ew;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16);
        griddep_wait();  // the scales are written by the kernels before this one
        int ntiles = 1;
        if constexpr (G) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0));
            ntiles = ok ? (int)misc[1] : 0;
        }
        int64_t g = 0;
        for (int k = 0; k < ntiles && ok; ++k) {
            const Tile t = G ? list_tile(s_list, k) : dense_tile(p);
            float y[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) y[i] = 0.0f;
            const bool cols = 64 * ch < t.n_mma;
            for (int64_t sb = 0; sb < nsb; ++sb) {
                const int64_t gg = g + sb;
                const int b = (int)(gg & 1);
                // this warp's 64 token scales d8 for the superblock
                {
                    const int64_t tc = t.t0 + 64 * ch + lane;
                    s_d8[lane] = tc < t.t_end ? __ldg(p.d8t + sb * p.Mp + tc) : 0.0f;
                    s_d8[lane + 32] = (tc + 32) < t.t_end ? __ldg(p.d8t + sb * p.Mp + tc + 32) : 0.0f;
                    __syncwarp();
                }
                bool w_ok = mbar_wait(&bar[BAR_SD_FULL + b], (uint32_t)((gg >> 1) & 1));
                if (w_ok) w_ok = mbar_wait(&bar[BAR_ACC_FULL + b], (uint32_t)((gg >> 1) & 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float dd = s_d[b * BM + r], dm = s_dmin[b * BM + r];
                if (cols) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t vi[16], vm[16];
                        tmem_ld16(lane_addr + 256 * b + 64 * ch + 16 * cc, vi);
                        if (C::kMins) tmem_ld16(lane_addr + 256 * b + 128 + 64 * ch + 16 * cc, vm);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float iv = __uint_as_float(vi[i]);
                            float tv = dd * iv;
                            if (C::kMins) tv = fmaf(-dm, __uint_as_float(vm[i]), tv);
                            y[16 * cc + i] = fmaf(s_d8[16 * cc + i], tv, y[16 * cc + i]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[BAR_ACC_EMPTY + b]);
            }
            if (!ok) break;
            const int n = t.n0 + r;
            if (n < p.N && cols) {
                const int c0 = t.t0 + 64 * ch, lim = t.t_end - c0;
                float *yp = p.y + (int64_t)c0 * p.N + n;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < lim) yp[(int64_t)i * p.N] = y[i];
            }
            g += nsb;
        }
        if (!ok && lane == 0) set_timeout();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// Workspace pre-pass: Q8_K planes -> fp16 q8 image [M][K], fp16 bsums
// [M][K/16] and d8 transposed [K/256][Mp].  One thread per 8 quants.
__global__ void __launch_bounds__(256) act_image_kernel(const int8_t *__restrict__ qs, const int16_t *__restrict__ bs,
                                                        const float *__restrict__ d8, int64_t M, int64_t K,
                                                        int64_t Mp, __half *__restrict__ a16,
                                                        __half *__restrict__ b16, float *__restrict__ d8t) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 quants
    const int64_t groups = M * K / 8;
    if (i < groups) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(qs) + i);
        uint32_t o[4];
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int8_t a = (int8_t)((w[k >> 1] >> (16 * (k & 1))) & 0xFF);
            const int8_t b = (int8_t)((w[k >> 1] >> (16 * (k & 1) + 8)) & 0xFF);
            const __half2 h = __halves2half2(__int2half_rn(a), __int2half_rn(b));
            o[k] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(a16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
        if ((i & 1) == 0) {  // one bsum per 16 quants
            const int64_t bi = i >> 1;
            b16[bi] = __int2half_rn((int)bs[bi]);
        }
        const int64_t nsb = K / QK;
        if ((i & 31) == 0) {  // one d8 per 256 quants
            const int64_t blk = i >> 5;
            const int64_t m = blk / nsb, s = blk % nsb;
            d8t[s * Mp + m] = d8[blk];
        }
    }
}

// ---------------------------------------------------------------------------
// host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

static bool make_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WsLayout {
    uint64_t a16, b16, d8t, total;
    int64_t Mp;
};

static WsLayout ws_layout(int64_t M, int64_t K) {
    WsLayout w;
    w.Mp = (M + 3) & ~int64_t(3);
    w.a16 = 0;
    w.b16 = align256((uint64_t)M * K * 2);
    w.d8t = w.b16 + align256((uint64_t)M * (K / 16) * 2);
    w.total = w.d8t + align256((uint64_t)(K / QK) * w.Mp * 4);
    return w;
}

// M below which the CUDA-core token-group kernel is used instead

size_t gemm_workspace_bytes(int, int64_t M, int64_t, int64_t K) {
    if (M < GEMM_TC_MIN_M) return 0;
    return (size_t)ws_layout(M, K).total;
}

template <int F>
static cudaError_t launch_gemm_f(const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, const int32_t *offsets,
                                 int64_t E, uint64_t expert_bytes, float *y, uint8_t *ws, cudaStream_t s) {
    using Cf = Cfg<F>;
    const WsLayout L = ws_layout(M, K);
    __half *a16 = reinterpret_cast<__half *>(ws + L.a16);
    __half *b16 = reinterpret_cast<__half *>(ws + L.b16);
    float *d8t = reinterpret_cast<float *>(ws + L.d8t);
    {
        const int64_t groups = M * K / 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((groups + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
        cudaError_t e = cudaLaunchKernelEx(&cfg, act_image_kernel, a.qs, a.bsums, a.d, M, K, L.Mp, a16, b16, d8t);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap ma, mb;
    if (!make_map_2d(&ma, a16, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, BT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!make_map_2d(&mb, b16, (uint64_t)(K / 16), (uint64_t)M, (uint64_t)(K / 16) * 2, 16, BT,
                     CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    // the shared-memory limit is a per-device attribute of the kernel: set it
    // once on every device the process launches on
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<F, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_kernel<F, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    GemmParams p{};
    p.packed = static_cast<const uint8_t *>(packed);
    p.expert_bytes = expert_bytes;
    p.N = N;
    p.K = K;
    p.nsb = K / QK;
    p.M = M;
    p.offsets = offsets;
    p.E = E;
    p.d8t = d8t;
    p.Mp = L.Mp;
    p.y = y;
    // dense: one block per tile; grouped: a block per SM walking a list of
    // tiles (the experts' first token tiles, plus at most M / BT later ones),
    // with enough blocks that no list exceeds TILE_CAP
    const int64_t w_tiles = (N + BM - 1) / BM;
    const int64_t t_tiles = (M + BT - 1) / BT;
    const int64_t tiles = offsets ? (E + M / BT) * w_tiles : t_tiles * w_tiles;
    if (tiles <= 0) return cudaSuccess;
    if (tiles > (int64_t)INT32_MAX || N > (int64_t)INT32_MAX - BM) return cudaErrorNotSupported;
    if (offsets && E > MAX_GROUPED_E) return cudaErrorNotSupported;
    int64_t blocks = tiles;
    if (offsets) {
        static std::atomic<int> sms[64];
        int n_sm = sms[dev].load(std::memory_order_relaxed);
        if (!n_sm) {
            if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
                return cudaErrorInvalidDevice;
            sms[dev].store(n_sm, std::memory_order_relaxed);
        }
        const int64_t need = (tiles + TILE_CAP - 3) / (TILE_CAP - 2);
        blocks = tiles < n_sm ? tiles : n_sm;
        if (blocks < need) blocks = need;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = offsets ? Cf::SMEM : Cf::SMEM_DENSE;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    if (offsets) return cudaLaunchKernelEx(&cfg, gemm_kernel<F, true>, ma, mb, p);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<F, false>, ma, mb, p);
}

cudaError_t launch_gemm_tc(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, const int32_t *offsets,
                           int64_t E, uint64_t expert_bytes, float *y, void *workspace, size_t workspace_bytes,
                           cudaStream_t s) {
    if (M < GEMM_TC_MIN_M || !workspace) return cudaErrorNotSupported;
    if (workspace_bytes < ws_layout(M, K).total) return cudaErrorInvalidValue;
    if (M > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX / 2) return cudaErrorNotSupported;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (f == FMT_Q4_K) return launch_gemm_f<FMT_Q4_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, s);
    if (f == FMT_Q5_K) return launch_gemm_f<FMT_Q5_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, s);
    return launch_gemm_f<FMT_Q6_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, s);
}

// Test hook: one block whose single bounded wait is never satisfied, so the
// wait gives up after limit_ns and records the timeout exactly as a stuck
// pipeline stage would (no fault, no hang).
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ uint64_t b;
    if (threadIdx.x == 0) {
        mbar_init(&b, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&b, 0, limit_ns)) set_timeout();
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

int read_and_clear_status(cudaStream_t s, int *status) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    *status = v;
    return 0;
}

}  // namespace kq
