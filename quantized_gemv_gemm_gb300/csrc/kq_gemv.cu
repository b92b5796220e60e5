// kq_gemv.cu - the decode GEMV (M = 1) over the packed image, and the int32
// partials test hook, which runs the same copy, read and fold code.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
//
// The GEMV streams the packed planes from HBM once ([kq-arc], kq v3 commit:
// decode time is set by DRAM traffic, so the planes stay bit-packed and no
// byte-expanded copy of them exists in DRAM) and folds every superblock in
// int32 with one float fold per superblock ([kq-arc], "The pieces", kq v2).
//
// Lane geometry.  A warp owns 16 weight rows at a time; lane l serves row
// l & 15 and half h = l >> 4 of every superblock, weights 128h .. 128h+127:
//   Q4_K/Q5_K: qs bytes 64h .. 64h+63 = chunks 2h, 2h+1 (byte 32c + i holds
//     element 64c + i in its low nibble, sub-block 2c, and element 64c+32+i
//     in its high nibble, sub-block 2c+1), so sub-blocks 4h .. 4h+3, with
//     sub-scales and sub-mins 4h .. 4h+3 = one word of each once decoded;
//     Q5_K adds bit 2c / 2c+1 of qh[i] (all 32 qh bytes) as value 16;
//   Q6_K: ql bytes 64h .. 64h+63 and qh bytes 32h .. 32h+31 = the sixteen-
//     element groups 8h .. 8h+7, with signed sub-scales 8h .. 8h+7.
// Each shared-memory phase (8 lanes) serves one half of 8 rows at the same
// superblock, so the activation reads are broadcasts and the weight reads
// are consecutive 16-byte pieces: no bank conflicts.
//
// Work split.  Rows are taken in groups of 16 (one per warp) across all the
// matrices; G groups.  A task is R = 8/S row groups x S superblock slices,
// one (group, slice) per warp of a 256-thread block; the S partial sums of
// a row are added in shared memory in a fixed order, so the result does not
// depend on timing.  The grid is persistent: every block takes the same
// number of consecutive tasks; S is the smallest of 1, 2, 4, 8 that gives
// every block slot at least one task.
//
// Memory pipeline.  Each warp has a ring of D superblock stages in shared
// memory.  An item (16 rows x one superblock) is one contiguous chunk of
// each plane of the grp16 image, already in the stage's order, so lane 0
// fetches it with one TMA bulk copy (cp.async.bulk) per plane, completing
// on the stage's mbarrier; the copies run D items ahead of the fold along
// the block's tasks, and the bytes in flight cost neither registers nor
// per-lane instructions.  Before griddepcontrol.wait a block touches only the packed
// weights (read-only on this path), so under programmatic dependent launch
// its first stages stream while the previous kernel finishes; every block
// signals griddepcontrol.launch_dependents on entry, since the next kernel
// waits for this grid's completion before it reads anything.  After the
// wait the block stages the activation row in shared memory (copied from
// the Q8_K planes, or quantized from the fp32 row bit-identically to
// kq_quantize_q8k) with the sums the fold needs.
#include "kq_internal.h"
#include "kq_sm100.cuh"

namespace kq {

// Tuning constants (compile time; the defaults are the measured choice):
// resident blocks per SM, whether a block lets the next kernel launch on
// entry (1) or once its activation row is staged (0), and the bytes of
// weights each block keeps streaming into L2 ahead of the task it folds
// (0: no bulk prefetch).
#ifndef KQ_GEMV_BLOCKS_PER_SM
#define KQ_GEMV_BLOCKS_PER_SM 2
#endif
#ifndef KQ_GEMV_EARLY_TRIGGER
#define KQ_GEMV_EARLY_TRIGGER 1
#endif
#ifndef KQ_GEMV_L2_WINDOW_KB
#define KQ_GEMV_L2_WINDOW_KB 0
#endif

// ---------------------------------------------------------------------------
// One superblock item of a warp = 16 rows x one superblock = the item's
// chunk of every plane, back to back (kq_device.cuh gives each chunk's
// inner order):
//   Q4_K: qs 2048 | hdr 256                     = 2304 B
//   Q5_K: qs 2048 | qh 512 | hdr 256            = 2816 B
//   Q6_K: ql 2048 | qh 1024 | sc 256 | d 32     = 3360 B
template <int F> struct GemvFmt;
template <> struct GemvFmt<FMT_Q4_K> { static constexpr int SLOT = 2304, D = 4; };
template <> struct GemvFmt<FMT_Q5_K> { static constexpr int SLOT = 2816, D = 4; };
template <> struct GemvFmt<FMT_Q6_K> { static constexpr int SLOT = 3360, D = 3; };
constexpr int GEMV_MAX_D = 4;

template <int F> constexpr int gemv_ring_bytes() { return 8 * GemvFmt<F>::D * GemvFmt<F>::SLOT; }

// staged row after the rings: quants [K] | sums [K/256][32 B] | d8 [K/256]
template <int F>
inline size_t gemv_smem_bytes(int64_t K) {
    return (size_t)gemv_ring_bytes<F>() + (size_t)(K + K / 8 + K / 64);
}

struct ItemQ4 { uint4 q[4]; uint4 hdr; };
struct ItemQ5 { uint4 q[4]; uint4 qh[2]; uint4 hdr; };
struct ItemQ6 { uint4 ql[4]; uint4 qh[2]; uint2 sc; uint32_t d; };
template <int F> struct ItemOf;
template <> struct ItemOf<FMT_Q4_K> { using T = ItemQ4; };
template <> struct ItemOf<FMT_Q5_K> { using T = ItemQ5; };
template <> struct ItemOf<FMT_Q6_K> { using T = ItemQ6; };

// The warp's plane pointers at the chunk of its row group's next superblock
// to fetch; one chunk further on is the next superblock.
struct ChunkPtr {
    const uint8_t *a, *b, *c, *d;
};

template <int F>
__device__ __forceinline__ ChunkPtr chunk_ptr(const Planes &P, uint64_t ch) {
    ChunkPtr q;
    q.a = P.p0 + ch * 2048;
    if constexpr (F == FMT_Q4_K) {
        q.b = P.p1 + ch * 256;
        q.c = q.d = nullptr;
    } else if constexpr (F == FMT_Q5_K) {
        q.b = P.p1 + ch * 512;
        q.c = P.p2 + ch * 256;
        q.d = nullptr;
    } else {
        q.b = P.p1 + ch * 1024;
        q.c = P.p2 + ch * 256;
        q.d = P.p3 + ch * 32;
    }
    return q;
}

// TMA bulk copy global -> shared of `bytes` (16-byte aligned, a multiple of
// 16), completing as transaction bytes on the mbarrier at shared address bar
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Lane 0: fetch one item into the stage at st (its mbarrier at bar) and step
// the chunk pointers; with on = 0 only arrive, so the stage's phase still
// completes for an item of a row group past the end.
template <int F>
__device__ __forceinline__ void item_issue(ChunkPtr &cp, uint32_t st, uint32_t bar, bool on) {
    constexpr int SLOT = GemvFmt<F>::SLOT;
    if (!on) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    } else {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(SLOT) : "memory");
        bulk_g2s(st, cp.a, 2048, bar);
        if constexpr (F == FMT_Q4_K) {
            bulk_g2s(st + 2048, cp.b, 256, bar);
        } else if constexpr (F == FMT_Q5_K) {
            bulk_g2s(st + 2048, cp.b, 512, bar);
            bulk_g2s(st + 2560, cp.c, 256, bar);
        } else {
            bulk_g2s(st + 2048, cp.b, 1024, bar);
            bulk_g2s(st + 3072, cp.c, 256, bar);
            bulk_g2s(st + 3328, cp.d, 32, bar);
        }
    }
    cp.a += 2048;
    if constexpr (F == FMT_Q4_K) {
        cp.b += 256;
    } else if constexpr (F == FMT_Q5_K) {
        cp.b += 512;
        cp.c += 256;
    } else {
        cp.b += 1024;
        cp.c += 256;
        cp.d += 32;
    }
}

// Per-lane offsets inside a stage: lane-major pieces at 16 * lane, row-major
// pieces at 16 * (lane & 15).
struct LaneOff {
    uint32_t q, r;
};
__device__ __forceinline__ LaneOff lane_off(int lane) { return LaneOff{16u * lane, 16u * (lane & 15)}; }

// read a landed item (stage at shared address st) into registers
__device__ __forceinline__ void item_read(ItemQ4 &w, uint32_t st, LaneOff lo, int) {
    const uint32_t sq = st + lo.q;
    w.q[0] = lds128o<0>(sq);
    w.q[1] = lds128o<512>(sq);
    w.q[2] = lds128o<1024>(sq);
    w.q[3] = lds128o<1536>(sq);
    w.hdr = lds128o<2048>(st + lo.r);
}
__device__ __forceinline__ void item_read(ItemQ5 &w, uint32_t st, LaneOff lo, int) {
    const uint32_t sq = st + lo.q, sr = st + lo.r;
    w.q[0] = lds128o<0>(sq);
    w.q[1] = lds128o<512>(sq);
    w.q[2] = lds128o<1024>(sq);
    w.q[3] = lds128o<1536>(sq);
    w.qh[0] = lds128o<2048>(sr);
    w.qh[1] = lds128o<2048 + 256>(sr);
    w.hdr = lds128o<2560>(sr);
}
__device__ __forceinline__ void item_read(ItemQ6 &w, uint32_t st, LaneOff lo, int h) {
    const uint32_t sq = st + lo.q, sr = st + lo.r;
    w.ql[0] = lds128o<0>(sq);
    w.ql[1] = lds128o<512>(sq);
    w.ql[2] = lds128o<1024>(sq);
    w.ql[3] = lds128o<1536>(sq);
    w.qh[0] = lds128o<2048>(sq);
    w.qh[1] = lds128o<2560>(sq);
    w.sc = lds64(sr + 3072 + 8 * h);
    w.d = lds16(st + 3328 + (lo.r >> 3));
}

// ---------------------------------------------------------------------------
// The lane's integer fold of one item against the staged activation
// superblock: a = shared address of the 128 activation quants of the
// lane's half (superblock base + 128h), sums = shared address of the
// lane's half of the superblock's 32-byte sum block (base + 16h).
//   Q4_K/Q5_K: isum = sum over sub-blocks 4h .. 4h+3 of sc_j * dot32_j,
//              msum = sum of m_j * S_j (S_j = sum of the 32 activation
//              quants of sub-block j)
//   Q6_K     : isum = iacc - 32 * bacc over groups 8h .. 8h+7, msum = 0
// The two lanes of a row add up to the superblock's isum / msum of the
// fold ([kq-arc], k4 and k5/k6 kq-v2 commits).

__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// dot of 16 unsigned weight bytes with the 16 signed activation bytes at
// shared address a + OFF, accumulated
template <int OFF>
__device__ __forceinline__ int dot16(uint4 q, uint32_t a, int acc) {
    const uint4 v = lds128o<OFF>(a);
    acc = dp4a_us(q.x, (int)v.x, acc);
    acc = dp4a_us(q.y, (int)v.y, acc);
    acc = dp4a_us(q.z, (int)v.z, acc);
    return dp4a_us(q.w, (int)v.w, acc);
}
__device__ __forceinline__ int byte_u(uint32_t w, int i) { return static_cast<int>(__byte_perm(w, 0u, 0x4440u + i)); }
__device__ __forceinline__ int byte_s(uint32_t w, int i) {
    return static_cast<int>(static_cast<int8_t>(__byte_perm(w, 0u, 0x4440u + i)));
}
__device__ __forceinline__ int half_s(uint32_t w, int i) { return static_cast<int>(static_cast<int16_t>(w >> (16 * i))); }

// sub-scale and sub-min words of the lane's half: bytes 0..3 = sub-blocks 4h .. 4h+3
__device__ __forceinline__ void scale_words(uint4 hdr, int h, uint32_t &scw, uint32_t &mw) {
    const uint32_t sl = hdr.y & 0x3F3F3F3Fu;
    const uint32_t sh = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t ml = hdr.z & 0x3F3F3F3Fu;
    const uint32_t mh = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    scw = h ? sh : sl;
    mw = h ? mh : ml;
}

__device__ __forceinline__ void item_fold(const ItemQ4 &w, int h, uint32_t a, uint32_t sums, int &isum, int &msum) {
    constexpr uint32_t LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
    // low nibbles as they are; high nibbles left in place (16 x q)
    int dl0 = dot16<0>(and4(w.q[0], LO), a, 0);
    dl0 = dot16<16>(and4(w.q[1], LO), a, dl0);
    int dh0 = dot16<32>(and4(w.q[0], HI), a, 0);
    dh0 = dot16<48>(and4(w.q[1], HI), a, dh0);
    int dl1 = dot16<64>(and4(w.q[2], LO), a, 0);
    dl1 = dot16<80>(and4(w.q[3], LO), a, dl1);
    int dh1 = dot16<96>(and4(w.q[2], HI), a, 0);
    dh1 = dot16<112>(and4(w.q[3], HI), a, dh1);
    uint32_t scw, mw;
    scale_words(w.hdr, h, scw, mw);
    isum = byte_u(scw, 0) * dl0 + byte_u(scw, 2) * dl1 + ((byte_u(scw, 1) * dh0 + byte_u(scw, 3) * dh1) >> 4);
    const uint4 S = lds128o<0>(sums);
    msum = byte_u(mw, 0) * (int)S.x + byte_u(mw, 1) * (int)S.y + byte_u(mw, 2) * (int)S.z + byte_u(mw, 3) * (int)S.w;
}

// bit b of every byte of x moved to bit 4 (a rotation: b - 4 mod 32 to the right)
__device__ __forceinline__ uint4 bit_to4(uint4 x, int b) {
    const int r = (b - 4) & 31;
    return make_uint4(__funnelshift_r(x.x, x.x, r) & 0x10101010u, __funnelshift_r(x.y, x.y, r) & 0x10101010u,
                      __funnelshift_r(x.z, x.z, r) & 0x10101010u, __funnelshift_r(x.w, x.w, r) & 0x10101010u);
}

__device__ __forceinline__ void item_fold(const ItemQ5 &w, int h, uint32_t a, uint32_t sums, int &isum, int &msum) {
    constexpr uint32_t LO = 0x0F0F0F0Fu;
    // chunk 2h: bits 4h (low nibbles), 4h+1 (high); chunk 2h+1: bits 4h+2, 4h+3;
    // pieces 0, 2 use qh[0..15], pieces 1, 3 use qh[16..31]
    int dl0 = dot16<0>(or4(and4(w.q[0], LO), bit_to4(w.qh[0], 4 * h)), a, 0);
    dl0 = dot16<16>(or4(and4(w.q[1], LO), bit_to4(w.qh[1], 4 * h)), a, dl0);
    int dh0 = dot16<32>(or4(and4(shr4(w.q[0], 4), LO), bit_to4(w.qh[0], 4 * h + 1)), a, 0);
    dh0 = dot16<48>(or4(and4(shr4(w.q[1], 4), LO), bit_to4(w.qh[1], 4 * h + 1)), a, dh0);
    int dl1 = dot16<64>(or4(and4(w.q[2], LO), bit_to4(w.qh[0], 4 * h + 2)), a, 0);
    dl1 = dot16<80>(or4(and4(w.q[3], LO), bit_to4(w.qh[1], 4 * h + 2)), a, dl1);
    int dh1 = dot16<96>(or4(and4(shr4(w.q[2], 4), LO), bit_to4(w.qh[0], 4 * h + 3)), a, 0);
    dh1 = dot16<112>(or4(and4(shr4(w.q[3], 4), LO), bit_to4(w.qh[1], 4 * h + 3)), a, dh1);
    uint32_t scw, mw;
    scale_words(w.hdr, h, scw, mw);
    isum = byte_u(scw, 0) * dl0 + byte_u(scw, 1) * dh0 + byte_u(scw, 2) * dl1 + byte_u(scw, 3) * dh1;
    const uint4 S = lds128o<0>(sums);
    msum = byte_u(mw, 0) * (int)S.x + byte_u(mw, 1) * (int)S.y + byte_u(mw, 2) * (int)S.z + byte_u(mw, 3) * (int)S.w;
}

__device__ __forceinline__ uint4 shl4(uint4 v, int s) { return make_uint4(v.x << s, v.y << s, v.z << s, v.w << s); }

__device__ __forceinline__ void item_fold(const ItemQ6 &w, int, uint32_t a, uint32_t sums, int &isum, int &msum) {
    constexpr uint32_t LO = 0x0F0F0F0Fu, HB = 0x30303030u;
    // piece k (ql bytes 64h + 16k, qh piece k & 1): low nibbles = group k with
    // qh bits 2(k>>1) .. +1; high nibbles = group k + 4 with bits 4 + 2(k>>1) .. +1
    int dt[8];
    dt[0] = dot16<0>(or4(and4(w.ql[0], LO), and4(shl4(w.qh[0], 4), HB)), a, 0);
    dt[1] = dot16<16>(or4(and4(w.ql[1], LO), and4(shl4(w.qh[1], 4), HB)), a, 0);
    dt[2] = dot16<32>(or4(and4(w.ql[2], LO), and4(shl4(w.qh[0], 2), HB)), a, 0);
    dt[3] = dot16<48>(or4(and4(w.ql[3], LO), and4(shl4(w.qh[1], 2), HB)), a, 0);
    dt[4] = dot16<64>(or4(and4(shr4(w.ql[0], 4), LO), and4(w.qh[0], HB)), a, 0);
    dt[5] = dot16<80>(or4(and4(shr4(w.ql[1], 4), LO), and4(w.qh[1], HB)), a, 0);
    dt[6] = dot16<96>(or4(and4(shr4(w.ql[2], 4), LO), and4(shr4(w.qh[0], 2), HB)), a, 0);
    dt[7] = dot16<112>(or4(and4(shr4(w.ql[3], 4), LO), and4(shr4(w.qh[1], 2), HB)), a, 0);
    const uint4 B = lds128o<0>(sums);  // bsums 8h .. 8h+7
    const uint32_t bw[4] = {B.x, B.y, B.z, B.w};
    int iacc = 0, bacc = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int sc = byte_s(t < 4 ? w.sc.x : w.sc.y, t & 3);
        iacc += sc * dt[t];
        bacc += sc * half_s(bw[t >> 1], t & 1);
    }
    isum = iacc - 32 * bacc;
    msum = 0;
}

__device__ __forceinline__ float item_d(const ItemQ4 &w) { return half_lo(w.hdr.x); }
__device__ __forceinline__ float item_d(const ItemQ5 &w) { return half_lo(w.hdr.x); }
__device__ __forceinline__ float item_d(const ItemQ6 &w) { return half_lo(w.d); }
__device__ __forceinline__ float item_dmin(const ItemQ4 &w) { return half_hi(w.hdr.x); }
__device__ __forceinline__ float item_dmin(const ItemQ5 &w) { return half_hi(w.hdr.x); }
__device__ __forceinline__ float item_dmin(const ItemQ6 &) { return 0.0f; }

// ---------------------------------------------------------------------------
struct GemvParams {
    int nmat;
    const uint8_t *packed[GEMV_MAX_MATRICES];
    int64_t N[GEMV_MAX_MATRICES];
    float *y[GEMV_MAX_MATRICES];
    int64_t gpre[GEMV_MAX_MATRICES + 1];  // prefix sums of 16-row groups
    int64_t K, nsb;
    int S;                                 // slices per row group (1, 2, 4, 8)
    int64_t tasks, tpc;                    // task count, tasks per block
    int64_t pf;                            // tasks kept streaming into L2 ahead (0: none)
    const float *x;                        // fp32 row (fused quantize), or nullptr
    const float *d8;                       // else: the Q8_K planes of the row
    const int8_t *qs;
    const int16_t *bs;
};

// Bounded wait on a stage's mbarrier (about one second): on expiry the
// kernel records KQ_ERR_TIMEOUT in the status word and carries on with
// whatever the stage holds, so no wait can hang the GPU.
__device__ int g_gemv_status = 0;

__device__ __forceinline__ void stage_wait(uint64_t *bar, uint32_t parity) {
    if (!sm100::mbar_wait(bar, parity)) atomicExch(&g_gemv_status, 1);
}

template <int F>
__global__ void __launch_bounds__(256, KQ_GEMV_BLOCKS_PER_SM) gemv_kernel(const GemvParams p) {
    constexpr int D = GemvFmt<F>::D, SLOT = GemvFmt<F>::SLOT;
    using Item = typename ItemOf<F>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Planes s_planes[GEMV_MAX_MATRICES];
    __shared__ float red[2][8][16];
    __shared__ uint64_t s_bar[8][GEMV_MAX_D];
    // the next kernel may be scheduled now: it waits for this grid to
    // complete before it reads anything this grid writes
    if (KQ_GEMV_EARLY_TRIGGER) griddep_launch_dependents();
    const int64_t K = p.K, nsb = p.nsb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r16 = lane & 15, h = lane >> 4;
    const uint32_t ring_s = smem_addr(smem + (size_t)warp * D * SLOT);
    uint64_t *bars = s_bar[warp];
    int8_t *s_qs = reinterpret_cast<int8_t *>(smem + gemv_ring_bytes<F>());
    uint8_t *s_sum = smem + gemv_ring_bytes<F>() + K;
    float *s_d8 = reinterpret_cast<float *>(smem + gemv_ring_bytes<F>() + K + K / 8);
    const uint32_t qs_s = smem_addr(s_qs), sum_s = smem_addr(s_sum), d8_s = smem_addr(s_d8);

    const int S = p.S, R = 8 / S;
    const int rg = warp / S, slice = warp % S;
    const int s0 = (int)(slice * nsb / S), len = (int)((slice + 1) * nsb / S) - s0;
    const int64_t t_begin = (int64_t)blockIdx.x * p.tpc;
    const int64_t left = p.tasks - t_begin;
    const int ntask = (int)(left <= 0 ? 0 : (left < p.tpc ? left : p.tpc));
    const int64_t G = p.gpre[p.nmat];
    if (threadIdx.x < p.nmat) s_planes[threadIdx.x] = make_planes(F, p.packed[threadIdx.x], p.N[threadIdx.x], nsb);
    if (lane == 0) {
        for (int i = 0; i < D; ++i) sm100::mbar_init(&bars[i], 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();

    // task tl of this block -> this warp's matrix, row group (and this lane's
    // row) and the chunk pointers of its slice's first superblock
    auto task_ptr = [&](int tl, int &m, int64_t &n, bool &valid) {
        const int64_t g = (t_begin + tl) * R + rg;
        valid = g < G;
        m = 0;
        while (m + 1 < p.nmat && g >= p.gpre[m + 1]) ++m;
        const int64_t gl = valid ? g - p.gpre[m] : 0;
        n = gl * GROUP_ROWS + r16;
        return chunk_ptr<F>(s_planes[m], (uint64_t)gl * nsb + s0);
    };
    // L2 prefetch of a whole task (its row groups are contiguous in every plane)
    auto prefetch_task = [&](int64_t tl) {
        if (tl >= ntask) return;
        const int64_t g0 = (t_begin + tl) * R, g1 = g0 + R < G ? g0 + R : G;
        int u[4];
        plane_unit_bytes(F, u);
        for (int m = 0; m < p.nmat; ++m) {
            const int64_t a = g0 > p.gpre[m] ? g0 : p.gpre[m], b = g1 < p.gpre[m + 1] ? g1 : p.gpre[m + 1];
            if (a >= b) continue;
            const uint64_t c0 = (uint64_t)(a - p.gpre[m]) * nsb, c1 = (uint64_t)(b - p.gpre[m]) * nsb;
            const uint8_t *base[4] = {s_planes[m].p0, s_planes[m].p1, s_planes[m].p2, s_planes[m].p3};
            for (int q = 0; q < 4; ++q)
                if (u[q]) prefetch_l2_bulk(base[q] + c0 * GROUP_ROWS * u[q], (c1 - c0) * GROUP_ROWS * u[q]);
        }
    };
    if (threadIdx.x == 0 && p.pf > 0)
        for (int64_t tl = 0; tl < p.pf; ++tl) prefetch_task(tl);

    // issue side (lane 0): runs D items ahead of the fold along the block's
    // tasks; one mbarrier phase per item and stage
    const LaneOff lo = lane_off(lane);
    const int total = ntask * len;
    ChunkPtr icp{};
    int irem = 0, itl = 0, iss = 0, it = 0;
    bool ion = false;
    if (ntask > 0) {
        int mm;
        int64_t nn;
        icp = task_ptr(0, mm, nn, ion);
        irem = len;
    }
    auto issue = [&]() {
        if (it < total) {
            if (lane == 0) item_issue<F>(icp, ring_s + iss * SLOT, smem_addr(&bars[iss]), ion);
            iss = iss + 1 == D ? 0 : iss + 1;
            if (--irem == 0 && ++itl < ntask) {
                int mm;
                int64_t nn;
                icp = task_ptr(itl, mm, nn, ion);
                irem = len;
            }
        }
        ++it;
    };
    for (int i = 0; i < D; ++i) issue();

    // activations: written by the kernels before this one
    griddep_wait();
    constexpr bool PAIRS = F != FMT_Q6_K;
    if (p.x) {
        // up to four blocks per warp per round, all loads issued first
        for (int64_t b0 = warp; b0 < nsb; b0 += 32) {
            float4 v[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t b = b0 + 8 * j;
                if (b < nsb) {
                    const float4 *xp = reinterpret_cast<const float4 *>(p.x + b * QK + 8 * lane);
                    v[j][0] = xp[0];
                    v[j][1] = xp[1];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t b = b0 + 8 * j;
                if (b < nsb) stage_block_from_x<PAIRS>(v[j][0], v[j][1], lane, s_qs + b * QK, s_sum + b * 32, s_d8 + b);
            }
        }
    } else {
        const uint4 *gq = reinterpret_cast<const uint4 *>(p.qs);
        for (int64_t i = threadIdx.x; i < K / 16; i += 256) reinterpret_cast<uint4 *>(s_qs)[i] = gq[i];
        if constexpr (PAIRS) {
            // sum of each 32-element sub-block = two consecutive bsums
            const int *gb = reinterpret_cast<const int *>(p.bs);
            for (int64_t i = threadIdx.x; i < K / 32; i += 256) {
                const int v = gb[i];
                reinterpret_cast<int *>(s_sum)[i] = (int)(int16_t)(v & 0xFFFF) + (v >> 16);
            }
        } else {
            const uint4 *gb = reinterpret_cast<const uint4 *>(p.bs);
            for (int64_t i = threadIdx.x; i < K / 128; i += 256) reinterpret_cast<uint4 *>(s_sum)[i] = gb[i];
        }
        for (int64_t i = threadIdx.x; i < nsb; i += 256) s_d8[i] = p.d8[i];
    }
    __syncthreads();
    if (!KQ_GEMV_EARLY_TRIGGER) griddep_launch_dependents();

    int tl = 0, j = 0, rs = 0;
    uint32_t rph = 0;  // parity of the current use of stage rs
    int m = 0;
    int64_t n = 0;
    bool valid = false;
    if (ntask > 0) task_ptr(0, m, n, valid);
    // running shared addresses of the current item's activation superblock
    // (the lane's half), sums and scale
    uint32_t a_cur = qs_s + (uint32_t)s0 * QK + 128 * h, s_cur = sum_s + (uint32_t)s0 * 32 + 16 * h;
    uint32_t d_cur = d8_s + 4 * (uint32_t)s0;
    float acc = 0.0f;
#pragma unroll 1
    for (int i = 0; i < total; ++i) {
        stage_wait(&bars[rs], rph);
        const uint32_t st = ring_s + rs * SLOT;
        Item cur;
        item_read(cur, st, lo, h);
        // every lane's reads of the stage are done before it is refilled
        __syncwarp();
        if (lane == 0) sm100::fence_proxy_async_smem();
        issue();  // item i + D into the stage just read
        if (++rs == D) {
            rs = 0;
            rph ^= 1u;
        }
        // rows past the last row group fold whatever the stage holds; their
        // sums are never written
        int isum, msum;
        item_fold(cur, h, a_cur, s_cur, isum, msum);
        const float d8 = __uint_as_float(lds32(d_cur));
        acc = fmaf(item_d(cur) * d8, static_cast<float>(isum), acc);
        if constexpr (F != FMT_Q6_K) acc = fmaf(-(item_dmin(cur) * d8), static_cast<float>(msum), acc);
        a_cur += QK;
        s_cur += 32;
        d_cur += 4;
        if (++j == len) {
            // end of a task: add the row's two halves, then its slices
            if (threadIdx.x == 0 && p.pf > 0) prefetch_task(tl + p.pf);
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
            if (h == 0) red[tl & 1][warp][r16] = acc;
            __syncthreads();
            if (slice == 0 && h == 0 && valid && n < p.N[m]) {
                float v = 0.0f;
                for (int q = 0; q < S; ++q) v += red[tl & 1][rg * S + q][r16];
                p.y[m][n] = v;
            }
            acc = 0.0f;
            j = 0;
            a_cur -= (uint32_t)len * QK;
            s_cur -= (uint32_t)len * 32;
            d_cur -= (uint32_t)len * 4;
            if (++tl < ntask) task_ptr(tl, m, n, valid);
        }
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

constexpr int64_t GEMV_L2_WINDOW = int64_t(KQ_GEMV_L2_WINDOW_KB) * 1024;

template <int F>
static cudaError_t launch_gemv_t(GemvParams p, cudaStream_t s) {
    p.gpre[0] = 0;
    for (int m = 0; m < p.nmat; ++m) p.gpre[m + 1] = p.gpre[m] + (p.N[m] + 15) / 16;
    const int64_t G = p.gpre[p.nmat];
    if (G == 0) return cudaSuccess;
    const int64_t slots = (int64_t)KQ_GEMV_BLOCKS_PER_SM * sm_count();
    int S = 1;
    while (S < 8 && 2 * S <= p.nsb && (G * S + 7) / 8 < slots) S *= 2;
    p.S = S;
    const int64_t R = 8 / S;
    p.tasks = (G + R - 1) / R;
    p.tpc = (p.tasks + slots - 1) / slots;
    const int64_t blocks = (p.tasks + p.tpc - 1) / p.tpc;
    const int64_t task_bytes = (R * 16) * p.nsb * block_bytes(F) / S;
    const int64_t pf = (GEMV_L2_WINDOW + task_bytes - 1) / task_bytes;
    p.pf = GEMV_L2_WINDOW == 0 ? 0 : (pf < 1 ? 1 : (pf > p.tpc ? p.tpc : pf));
    static bool attr_set[64][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!attr_set[dev][F]) {
        const cudaError_t e = cudaFuncSetAttribute(gemv_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)gemv_smem_bytes<F>(GEMV_MAX_K));
        if (e != cudaSuccess) return e;
        attr_set[dev][F] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = gemv_smem_bytes<F>(p.K);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<F>, p);
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

// ---------------------------------------------------------------------------
// Test hook: int32 partials per (token, row, superblock) through the
// GEMV's own path: one warp fetches the item of 16 rows x one superblock
// with item_issue, reads it back with item_read and folds it with
// item_fold against the token's superblock staged as the GEMV stages it.
template <int F>
__global__ void __launch_bounds__(256) partials_kernel(const uint8_t *packed, int64_t N, int64_t nsb, int64_t K,
                                                       Q8K a, int64_t M, int32_t *isum_out, int32_t *msum_out) {
    constexpr int SLOT = GemvFmt<F>::SLOT;
    __shared__ __align__(128) uint8_t s_item[8][SLOT];
    __shared__ __align__(16) int8_t s_act[8][QK];
    __shared__ __align__(16) int s_sum[8][8];
    __shared__ uint64_t s_bar[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r16 = lane & 15, h = lane >> 4;
    const int64_t g = (int64_t)blockIdx.x * 8 + warp;  // row group
    const int64_t n = g * GROUP_ROWS + r16;
    const int64_t sb = blockIdx.y;
    const int64_t tok = blockIdx.z;
    const bool on = g < row_groups(N);
    reinterpret_cast<uint2 *>(s_act[warp])[lane] = reinterpret_cast<const uint2 *>(a.qs + tok * K + sb * QK)[lane];
    const int16_t *gb = a.bsums + (tok * nsb + sb) * 16;
    if constexpr (F != FMT_Q6_K) {
        if (lane < 8) s_sum[warp][lane] = (int)gb[2 * lane] + (int)gb[2 * lane + 1];
    } else {
        if (lane < 16) reinterpret_cast<int16_t *>(s_sum[warp])[lane] = gb[lane];
    }
    if (lane == 0) {
        sm100::mbar_init(&s_bar[warp], 1);
        sm100::mbar_fence_init();
    }
    __syncwarp();
    const Planes P = make_planes(F, packed, N, nsb);
    ChunkPtr cp = chunk_ptr<F>(P, (uint64_t)(on ? g : 0) * nsb + sb);
    if (lane == 0) item_issue<F>(cp, smem_addr(s_item[warp]), smem_addr(&s_bar[warp]), on);
    stage_wait(&s_bar[warp], 0);
    typename ItemOf<F>::T w;
    item_read(w, smem_addr(s_item[warp]), lane_off(lane), h);
    int isum, msum;
    item_fold(w, h, smem_addr(s_act[warp]) + 128 * h, smem_addr(s_sum[warp]) + 16 * h, isum, msum);
    isum += __shfl_xor_sync(0xFFFFFFFFu, isum, 16);
    msum += __shfl_xor_sync(0xFFFFFFFFu, msum, 16);
    if (h == 0 && n < N) {
        const int64_t o = (tok * N + n) * nsb + sb;
        isum_out[o] = isum;
        msum_out[o] = msum;
    }
}

cudaError_t launch_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                            int32_t *isum, int32_t *msum, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    dim3 grid((unsigned)((N + 127) / 128), (unsigned)nsb, (unsigned)M);
    const uint8_t *pk = static_cast<const uint8_t *>(packed);
    if (f == FMT_Q4_K) partials_kernel<FMT_Q4_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    else if (f == FMT_Q5_K) partials_kernel<FMT_Q5_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    else partials_kernel<FMT_Q6_K><<<grid, 256, 0, s>>>(pk, N, nsb, K, a, M, isum, msum);
    return cudaGetLastError();
}

int read_and_clear_gemv_status(cudaStream_t s, int *status) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_gemv_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_gemv_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    *status = v;
    return 0;
}

}  // namespace kq
