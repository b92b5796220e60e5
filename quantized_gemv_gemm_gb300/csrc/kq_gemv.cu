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
// Work split.  Rows are taken in groups of 16 across all the matrices (G
// groups); an item is one row group x one superblock, items ordered
// g * K/256 + sb.  The grid has one block per SM, and block b takes the
// items [b*I/B, (b+1)*I/B) of the I = G*K/256, its eight warps an even
// eighth of those each, so every warp folds the same number of items (to
// one) whatever the matrix shapes.  A block is given at most half an SM
// (110 KB of shared memory, 128 registers a thread), so the next GEMV's
// block fits beside it.  A warp stores the rows of a row group it folds
// whole; a row group split between warps is added in shared memory in warp
// order; one split between two blocks (at most two, as every block holds at
// least K/256 items) is finished by the block that arrives second, which
// adds the two partial sums kept in the caller's workspace.  Every sum has
// a fixed order (two terms commute exactly), so the result does not depend
// on timing.  Without a workspace the blocks take whole row groups instead.
//
// Memory pipeline.  Each warp has a ring of D superblock stages in shared
// memory.  An item (16 rows x one superblock) is one contiguous chunk of
// each plane of the grp16 image, already in the stage's order, so lane 0
// fetches it with one TMA bulk copy (cp.async.bulk) per plane, completing
// on the stage's mbarrier; the copies run D items ahead of the fold along
// the warp's range, and the bytes in flight cost neither registers nor
// per-lane instructions.  Before griddepcontrol.wait a block touches only the packed
// weights (read-only on this path), so under programmatic dependent launch
// its first stages stream while the previous kernel finishes; every block
// signals griddepcontrol.launch_dependents on entry, since the next kernel
// waits for this grid's completion before it reads anything.  After the
// wait the block stages the activation row in shared memory (copied from
// the Q8_K planes, or quantized from the fp32 row bit-identically to
// kq_quantize_q8k) with the sums the fold needs.
#include <atomic>
#include <type_traits>

#include "kq_internal.h"
#include "kq_sm100.cuh"

namespace kq {

// ---------------------------------------------------------------------------
// One superblock item of a warp = 16 rows x one superblock = the item's
// chunk of every plane, back to back (kq_device.cuh gives each chunk's
// inner order):
//   Q4_K: qs 2048 | hdr 256                     = 2304 B
//   Q5_K: qs 2048 | qh 512 | hdr 256            = 2816 B
//   Q6_K: ql 2048 | qh 1024 | sc 256 | d 32     = 3360 B
template <int F> struct GemvFmt;
template <> struct GemvFmt<FMT_Q4_K> { static constexpr int SLOT = 2304; };
template <> struct GemvFmt<FMT_Q5_K> { static constexpr int SLOT = 2816; };
template <> struct GemvFmt<FMT_Q6_K> { static constexpr int SLOT = 3360; };
constexpr int GEMV_MAX_D = 6;

// Shared memory of one block: the warps' rings (8 x D x SLOT), then the
// staged row: quants [K] | sums [K/256][32 B] | d8 [K/256].
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
// 16), completing as transaction bytes on the mbarrier at shared address
// bar, with the L2 cache policy pol
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// L2 policy of the weight stream: every packed byte is read once per call,
// so its lines go first when L2 needs room, and the activations and other
// data the surrounding kernels reuse stay in L2
__device__ __forceinline__ uint64_t weight_stream_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Lane 0: fetch one item into the stage at st (its mbarrier at bar) and step
// the chunk pointers; with on = 0 only arrive, so the stage's phase still
// completes for an item of a row group past the end.
template <int F>
__device__ __forceinline__ void item_issue(ChunkPtr &cp, uint32_t st, uint32_t bar, bool on, uint64_t pol) {
    constexpr int SLOT = GemvFmt<F>::SLOT;
    if (!on) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    } else {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(SLOT) : "memory");
        bulk_g2s(st, cp.a, 2048, bar, pol);
        if constexpr (F == FMT_Q4_K) {
            bulk_g2s(st + 2048, cp.b, 256, bar, pol);
        } else if constexpr (F == FMT_Q5_K) {
            bulk_g2s(st + 2048, cp.b, 512, bar, pol);
            bulk_g2s(st + 2560, cp.c, 256, bar, pol);
        } else {
            bulk_g2s(st + 2048, cp.b, 1024, bar, pol);
            bulk_g2s(st + 3072, cp.c, 256, bar, pol);
            bulk_g2s(st + 3328, cp.d, 32, bar, pol);
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
// Tensor-core fold of one item for a pass of 8 tokens (T = 8, Q4_K and
// Q6_K): the warp's 16 weight rows x the pass's token rows with the
// integer warp MMA, u8 weights x s8 activations -> s32 (exact).  Q4_K takes
// one m16n8k32 per 32-element sub-block (its scale and min are per row),
// Q6_K one m16n8k16 per 16-element group.  Fragment ownership (PTX ISA,
// m16n8k32 / m16n8k16 with 8-bit operands): lane (gq = lane / 4,
// cq = lane % 4) holds A bytes 4cq..4cq+3 of rows gq and gq+8 (and 16 bytes
// further for k32), B bytes 4cq..4cq+3 (and +16) of token column gq, and
// the accumulators (row gq, tokens 2cq, 2cq+1) and (row gq+8, the same
// tokens).  The weights come from the stage already in shared memory; the
// reads of one item are all issued before the stage is handed back.
// (Measured on GB300, the Qwen3-4B-shaped layer through kq_gemv_fused_batch:
// M = 8 in 76.8 instead of 84.6 us; at M = 4, where half of each MMA's
// token columns are empty, 62.7 instead of 51.9 us, so T = 4 keeps dp4a.)
template <int F, int T> struct MmaFold {
    static constexpr bool on = T >= 8 && (F == FMT_Q4_K || F == FMT_Q6_K);
};

__device__ __forceinline__ void mma_k32_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}
__device__ __forceinline__ void mma_k16_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// the lane's raw share of a Q4_K item: [half][row gq / gq+8][piece] words
// (bytes 4cq..4cq+3 of the row's 16-byte piece), and the two rows' headers
struct MmaQ4 {
    uint32_t q[2][2][4];
    uint4 hdr[2];
};
struct MmaQ6 {
    uint32_t ql[2][2][4];
    uint32_t qh[2][2][2];
    uint4 sc[2];     // the 16 int8 group scales of rows gq, gq+8
    uint32_t d[2];   // their fp16 d
};

__device__ __forceinline__ void mma_read(MmaQ4 &w, uint32_t st, int gq, int cq) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int pc = 0; pc < 4; ++pc)
                w.q[h2][rr][pc] = lds32(st + 16u * (gq + 8 * rr + 16 * h2) + 512u * pc + 4u * cq);
    w.hdr[0] = lds128(st + 2048u + 16u * gq);
    w.hdr[1] = lds128(st + 2048u + 16u * (gq + 8));
}
__device__ __forceinline__ void mma_read(MmaQ6 &w, uint32_t st, int gq, int cq) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t r = gq + 8 * rr + 16 * h2;
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) w.ql[h2][rr][pc] = lds32(st + 16u * r + 512u * pc + 4u * cq);
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) w.qh[h2][rr][pc] = lds32(st + 2048u + 512u * pc + 16u * r + 4u * cq);
        }
    w.sc[0] = lds128(st + 3072u + 16u * gq);
    w.sc[1] = lds128(st + 3072u + 16u * (gq + 8));
    w.d[0] = lds16(st + 3328u + 2u * gq);
    w.d[1] = lds16(st + 3328u + 2u * (gq + 8));
}

// Integer sums of one item for the pass: isum[rr * 2 + k], msum[rr * 2 + k]
// (row gq + 8 rr, token 2cq + k) -- Q4_K isum = sum_j sc_j * dot32_j and
// msum = sum_j m_j * (bs_2j + bs_2j+1); Q6_K isum = iacc - 32 * bacc and
// msum = 0.  act = shared address of token 0's activation superblock, sums
// of its sums; tokens are tstride apart; tokens at or past ntok are not read
// (their columns are zero and their sums left 0).
__device__ __forceinline__ void mma_isums(const MmaQ4 &w, int gq, int cq, int ntok, uint32_t act, uint32_t sums,
                                          uint32_t tstride, int (&isum)[4], int (&msum)[4]) {
    constexpr uint32_t LO = 0x0F0F0F0Fu;
    const bool bt = gq < ntok;
    const uint32_t ab = act + (uint32_t)gq * tstride + 4u * cq;
    uint32_t scw[2][2], mw[2][2];  // [row][half]
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        scale_words(w.hdr[rr], 0, scw[rr][0], mw[rr][0]);
        scale_words(w.hdr[rr], 1, scw[rr][1], mw[rr][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) isum[i] = msum[i] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int h2 = j >> 2, jj = j & 3, pp = (jj >> 1) * 2, sh = 4 * (jj & 1);
        const uint32_t a0 = (w.q[h2][0][pp] >> sh) & LO, a1 = (w.q[h2][1][pp] >> sh) & LO;
        const uint32_t a2 = (w.q[h2][0][pp + 1] >> sh) & LO, a3 = (w.q[h2][1][pp + 1] >> sh) & LO;
        const uint32_t b0 = bt ? lds32(ab + 32u * j) : 0u, b1 = bt ? lds32(ab + 32u * j + 16u) : 0u;
        int dd[4];
        mma_k32_u8s8(dd, a0, a1, a2, a3, b0, b1);
        const int s0 = byte_u(scw[0][h2], jj), s1 = byte_u(scw[1][h2], jj);
        isum[0] += s0 * dd[0];
        isum[1] += s0 * dd[1];
        isum[2] += s1 * dd[2];
        isum[3] += s1 * dd[3];
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int t = 2 * cq + k;
        if (t < ntok) {
            const uint32_t so = sums + (uint32_t)t * tstride;
            const uint4 S0 = lds128(so), S1 = lds128(so + 16u);  // the 8 sub-block sums
            const int Sv[8] = {(int)S0.x, (int)S0.y, (int)S0.z, (int)S0.w, (int)S1.x, (int)S1.y, (int)S1.z, (int)S1.w};
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                int m = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) m += byte_u(mw[rr][j >> 2], j & 3) * Sv[j];
                msum[rr * 2 + k] = m;
            }
        }
    }
}

__device__ __forceinline__ void mma_isums(const MmaQ6 &w, int gq, int cq, int ntok, uint32_t act, uint32_t sums,
                                          uint32_t tstride, int (&isum)[4], int (&msum)[4]) {
    constexpr uint32_t LO = 0x0F0F0F0Fu, HB = 0x30303030u;
    const bool bt = gq < ntok;
    const uint32_t ab = act + (uint32_t)gq * tstride + 4u * cq;
    int iacc[4] = {0, 0, 0, 0};
    const uint32_t scv[2][4] = {{w.sc[0].x, w.sc[0].y, w.sc[0].z, w.sc[0].w},
                                {w.sc[1].x, w.sc[1].y, w.sc[1].z, w.sc[1].w}};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            // group t of the half: piece t % 4 (low nibbles for t < 4), high
            // bits from qh piece t % 2 at bits 2 (t / 2), +1 of each byte
            const int pc = t & 3, pq = t & 1, ns = t < 4 ? 0 : 4;
            uint32_t a[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const uint32_t lo = (w.ql[h2][rr][pc] >> ns) & LO;
                const uint32_t qh = w.qh[h2][rr][pq];
                const int sel = t >> 1;  // 0: << 4, 1: << 2, 2: as is, 3: >> 2
                const uint32_t hb = sel == 0 ? (qh << 4) : (sel == 1 ? (qh << 2) : (sel == 2 ? qh : (qh >> 2)));
                a[rr] = lo | (hb & HB);
            }
            const uint32_t b0 = bt ? lds32(ab + 128u * h2 + 16u * t) : 0u;
            int dd[4];
            mma_k16_u8s8(dd, a[0], a[1], b0);
            const int grp = 8 * h2 + t;
            const int s0 = byte_s(scv[0][grp >> 2], grp & 3), s1 = byte_s(scv[1][grp >> 2], grp & 3);
            iacc[0] += s0 * dd[0];
            iacc[1] += s0 * dd[1];
            iacc[2] += s1 * dd[2];
            iacc[3] += s1 * dd[3];
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) isum[i] = msum[i] = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int t = 2 * cq + k;
        if (t < ntok) {
            const uint32_t so = sums + (uint32_t)t * tstride;
            const uint4 B0 = lds128(so), B1 = lds128(so + 16u);  // the 16 int16 bsums
            const uint32_t bw[8] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w};
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                int bacc = 0;
#pragma unroll
                for (int grp = 0; grp < 16; ++grp)
                    bacc += byte_s(scv[rr][grp >> 2], grp & 3) * half_s(bw[grp >> 1], grp & 1);
                isum[rr * 2 + k] = iacc[rr * 2 + k] - 32 * bacc;
            }
        }
    }
}

// Fold of one item for the pass: acc[rr * 2 + k] (row gq + 8 rr, token
// 2cq + k) += d * d8 * isum - dmin * d8 * msum, from the integer sums
// above; d8s = shared address of token 0's scale (tokens tstride apart).
template <typename MItem>
__device__ __forceinline__ void mma_fold(const MItem &w, int gq, int cq, int ntok, uint32_t act, uint32_t sums,
                                         uint32_t d8s, uint32_t tstride, float (&acc)[4]) {
    int isum[4], msum[4];
    mma_isums(w, gq, cq, ntok, act, sums, tstride, isum, msum);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int t = 2 * cq + k;
        if (t < ntok) {
            const float d8 = __uint_as_float(lds32(d8s + (uint32_t)t * tstride));
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                if constexpr (std::is_same<MItem, MmaQ4>::value) {
                    const float dw = half_lo(w.hdr[rr].x), dmw = half_hi(w.hdr[rr].x);
                    const float a = fmaf(dw * d8, static_cast<float>(isum[rr * 2 + k]), acc[rr * 2 + k]);
                    acc[rr * 2 + k] = fmaf(-(dmw * d8), static_cast<float>(msum[rr * 2 + k]), a);
                } else {
                    const float dw = half_lo(w.d[rr]);
                    acc[rr * 2 + k] = fmaf(dw * d8, static_cast<float>(isum[rr * 2 + k]), acc[rr * 2 + k]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// Staging of one activation superblock from the fp32 row (the fused
// quantize, bit-identical to kq_quantize_q8k through q8k_lane): the 256
// quants, the block scale, and the sums the fold needs -- for Q4_K and Q5_K
// the int32 sum of each 32-element sub-block (bs_2j + bs_2j+1, the factor of
// sub-min j), for Q6_K the 16 int16 bsums; both forms take 32 bytes.  The
// lane holds elements 8*lane .. 8*lane+7 in v0, v1.
template <bool PAIRS>
__device__ __forceinline__ void stage_block_from_x(float4 v0, float4 v1, int lane, int8_t *qb, void *sb, float *db) {
    int part;
    float d8;
    const uint2 w = q8k_lane(v0, v1, part, d8);
    *reinterpret_cast<uint2 *>(qb + 8 * lane) = w;
    part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);        // 16-element sums
    if constexpr (PAIRS) {
        part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);    // 32-element sums
        if ((lane & 3) == 0) static_cast<int *>(sb)[lane >> 2] = part;
    } else {
        if ((lane & 1) == 0) static_cast<int16_t *>(sb)[lane >> 1] = static_cast<int16_t>(part);
    }
    if (lane == 0) *db = d8;
}

// The same for the J blocks b0, b0 + 8, ..., b0 + 8(J-1) of the row x (those
// below nsb are stored), one warp, with the blocks' steps interleaved: each
// block's chain (max, divide, round, sums) is independent of the others', so
// J blocks take about the latency of one.  Every step is q8k_lane's (an all-
// zero block gets iscale 0, hence every q = 0, as q8k_lane gives it).
template <bool PAIRS, int J>
__device__ __forceinline__ void stage_blocks_from_x(const float *x, int64_t nsb, int64_t b0, int lane, int8_t *qs,
                                                    uint8_t *sums, float *d8s) {
    float4 v0[J], v1[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t b = b0 + 8 * j;
        if (b < nsb) {
            const float4 *xp = reinterpret_cast<const float4 *>(x + b * QK + 8 * lane);
            v0[j] = xp[0];
            v1[j] = xp[1];
        } else {
            v0[j] = v1[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
    }
    float amax[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        float ax = fmaxf(fmaxf(fabsf(v0[j].x), fabsf(v0[j].y)), fmaxf(fabsf(v0[j].z), fabsf(v0[j].w)));
        ax = fmaxf(ax, fmaxf(fmaxf(fabsf(v1[j].x), fabsf(v1[j].y)), fmaxf(fabsf(v1[j].z), fabsf(v1[j].w))));
        amax[j] = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(ax)));
    }
    float iscale[J];
#pragma unroll
    for (int j = 0; j < J; ++j) iscale[j] = amax[j] == 0.0f ? 0.0f : __fdiv_rn(127.0f, amax[j]);
    int part[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const float v[8] = {v0[j].x, v0[j].y, v0[j].z, v0[j].w, v1[j].x, v1[j].y, v1[j].z, v1[j].w};
        uint32_t lo = 0, hi = 0;
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = max(-127, min(127, __float2int_rn(__fmul_rn(v[i], iscale[j]))));
            sum += q;
            if (i < 4) lo |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
            else hi |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i - 4));
        }
        part[j] = sum;
        const int64_t b = b0 + 8 * j;
        if (b < nsb) *reinterpret_cast<uint2 *>(qs + b * QK + 8 * lane) = make_uint2(lo, hi);
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        part[j] += __shfl_xor_sync(0xFFFFFFFFu, part[j], 1);        // 16-element sums
        if constexpr (PAIRS) part[j] += __shfl_xor_sync(0xFFFFFFFFu, part[j], 2);  // 32-element sums
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t b = b0 + 8 * j;
        if (b >= nsb) continue;
        if constexpr (PAIRS) {
            if ((lane & 3) == 0) reinterpret_cast<int *>(sums + b * 32)[lane >> 2] = part[j];
        } else {
            if ((lane & 1) == 0) reinterpret_cast<int16_t *>(sums + b * 32)[lane >> 1] = static_cast<int16_t>(part[j]);
        }
        if (lane == 0) d8s[b] = amax[j] == 0.0f ? 0.0f : __fdiv_rn(amax[j], 127.0f);
    }
}

struct GemvParams {
    int nmat;
    const uint8_t *packed[GEMV_MAX_MATRICES];
    int64_t N[GEMV_MAX_MATRICES];
    float *y[GEMV_MAX_MATRICES];
    int64_t gpre[GEMV_MAX_MATRICES + 1];  // prefix sums of 16-row groups
    int64_t K, nsb;
    int64_t items;                         // G * nsb (row group x superblock items)
    int split;                             // block ranges may cut a row group in two
    int D;                                 // ring stages per warp
    unsigned long long *ws;                // [grid][16] words of the row groups cut between blocks
    const float *x;                        // fp32 row (fused quantize), or nullptr
    const float *d8;                       // else: the Q8_K planes of the rows
    const int8_t *qs;
    const int16_t *bs;
    int ntok;                              // token rows folded per pass (1..T of the kernel)
    int64_t stage_stride;                  // bytes between the staged rows of two tokens
    // grouped (MoE) rows: matrix m is row m % ntok of the activations times
    // the weights, in set m / ntok, of the expert whose row range
    // [offsets[e], offsets[e+1]) holds that row; packed[m] is the start of
    // that set's experts (back to back, expert_bytes[set] each)
    const int32_t *offsets;
    int64_t E;
    uint64_t expert_bytes[GEMV_FUSED_MAX];
};

// Bounded wait on a stage's mbarrier (about one second): on expiry the
// kernel records KQ_ERR_TIMEOUT in the status word and carries on with
// whatever the stage holds, so no wait can hang the GPU.
__device__ int g_gemv_status = 0;

__device__ __forceinline__ void stage_wait(uint64_t *bar, uint32_t parity) {
    if (!sm100::mbar_wait(bar, parity)) atomicExch(&g_gemv_status, 1);
}

// a workspace word holding a partial sum (low 32 bits) carries this tag
constexpr unsigned long long GEMV_TAG = 1ull << 32;

// first item of block b's range: whole row groups when split == 0
__device__ __forceinline__ int64_t block_item(const GemvParams &p, int64_t b, int64_t B, int64_t G) {
    return p.split ? b * p.items / B : (b * G / B) * p.nsb;
}

// T: the most token rows one pass folds (1 for decode; 2, 4, 8 for small
// batches, which read each weight item once for all their tokens).  Token t's
// activation row is staged at stage_stride * t, and its output row is
// y[m] + t * N[m].
// GR: grouped rows (MoE decode) -- the matrices are found on the device from
// the expert offsets, after the wait: with ntok activation rows and nmat =
// sets * ntok matrices, matrix m is activation row m % ntok times that row's
// expert in weight set m / ntok (e.g. gate and up sharing the rows).
template <int F, int T, bool GR>
__global__ void __launch_bounds__(256, 2) gemv_kernel(const GemvParams p) {
    constexpr int SLOT = GemvFmt<F>::SLOT;
    using Item = typename ItemOf<F>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Planes s_planes[GEMV_MAX_MATRICES];
    // the matrices' row-group prefix sums, row counts and outputs
    __shared__ int64_t s_gpre[GEMV_MAX_MATRICES + 1], s_n[GEMV_MAX_MATRICES];
    __shared__ float *s_y[GEMV_MAX_MATRICES];
    __shared__ uint64_t s_bar[8][GEMV_MAX_D];
    // a warp's partial sums of the row groups it shares with other warps or
    // blocks: slot 0 = the group its range starts inside, slot 1 = the group
    // it ends inside; and, where the warp finishes such a group, how: the
    // mask of the warps that hold a part (0: another warp finishes it), the
    // matrix, the group's first output row in it, and the cut between blocks
    // (-1: none)
    __shared__ float s_rec[8][2][T][16];
    // grouped: the expert of each activation row (-1: none)
    __shared__ int64_t s_row_e[GEMV_MAX_MATRICES];
    __shared__ int s_fin_mask[8][2], s_fin_m[8][2];
    __shared__ int64_t s_fin_row[8][2], s_fin_cut[8][2];
    // the next kernel may be scheduled now: it waits for this grid to
    // complete before it reads anything this grid writes
    griddep_launch_dependents();
    const int64_t K = p.K, nsb = p.nsb;
    const int D = p.D;
    const int ntok = (T == 1 && !GR) ? 1 : p.ntok;
    const uint32_t tstride = (T == 1 && !GR) ? 0u : (uint32_t)p.stage_stride;
    // grouped: matrix m's staged row (m % ntok) is at (m % ntok) * mstride
    const uint32_t mstride = GR ? tstride : 0u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r16 = lane & 15, h = lane >> 4;
    const uint32_t ring_s = smem_addr(smem + (size_t)warp * D * SLOT);
    uint64_t *bars = s_bar[warp];
    const size_t ring_bytes = (size_t)8 * D * SLOT;
    int8_t *s_qs = reinterpret_cast<int8_t *>(smem + ring_bytes);
    uint8_t *s_sum = smem + ring_bytes + K;
    float *s_d8 = reinterpret_cast<float *>(smem + ring_bytes + K + K / 8);
    const uint32_t qs_s = smem_addr(s_qs), sum_s = smem_addr(s_sum), d8_s = smem_addr(s_d8);

    // this block's items [I0, I1) and this warp's [w0, w1), in the order
    // item = g * nsb + sb over the row groups of all the matrices
    const int64_t G = p.gpre[p.nmat], B = gridDim.x;
    const int64_t I0 = block_item(p, blockIdx.x, B, G), I1 = block_item(p, blockIdx.x + 1, B, G);
    const int64_t w0 = I0 + warp * (I1 - I0) / 8, w1 = I0 + (warp + 1) * (I1 - I0) / 8;
    // Stage the activation rows in shared memory (need: bit t set = token
    // row t is read by this block's matrices).
    constexpr bool PAIRS = F != FMT_Q6_K;
    auto stage_rows = [&](uint32_t need) {
        if ((T > 1 || GR) && p.x) {
            // several fp32 rows: block vb of the rows laid end to end is block
            // vb % nsb of token row vb / nsb, staged in that token's row (32-bit
            // index arithmetic: nvb <= 16 * 160, and a 64-bit division is a
            // long instruction sequence)
            const uint32_t nsb32 = (uint32_t)nsb, nvb = (uint32_t)ntok * nsb32;
            for (uint32_t vb0 = warp; vb0 < nvb; vb0 += 64) {
                float4 v[8][2];
                uint32_t tj[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t vb = vb0 + 8 * j;
                    tj[j] = vb / nsb32;
                    if (vb < nvb && ((need >> tj[j]) & 1u)) {
                        const float4 *xp = reinterpret_cast<const float4 *>(p.x + (int64_t)vb * QK + 8 * lane);
                        v[j][0] = xp[0];
                        v[j][1] = xp[1];
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t vb = vb0 + 8 * j;
                    if (vb < nvb && ((need >> tj[j]) & 1u)) {
                        const uint32_t t = tj[j], b = vb - t * nsb32;
                        const size_t o = (size_t)t * tstride;
                        stage_block_from_x<PAIRS>(v[j][0], v[j][1], lane, reinterpret_cast<int8_t *>(
                                                  reinterpret_cast<uint8_t *>(s_qs) + o) + b * QK, s_sum + o + b * 32,
                                                  reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(s_d8) + o) + b);
                    }
                }
            }
        } else if (p.x) {
            // up to four blocks per warp per round (warp w: blocks w, w + 8,
            // ...), quantized together (measured: five or eight at once are
            // slower -- the registers run out)
            for (int64_t b0 = warp; b0 < nsb; b0 += 32) {
                const int64_t mine = (nsb - b0 + 7) / 8;  // this warp's blocks in the round
                if (mine > 2) stage_blocks_from_x<PAIRS, 4>(p.x, nsb, b0, lane, s_qs, s_sum, s_d8);
                else if (mine > 1) stage_blocks_from_x<PAIRS, 2>(p.x, nsb, b0, lane, s_qs, s_sum, s_d8);
                else stage_blocks_from_x<PAIRS, 1>(p.x, nsb, b0, lane, s_qs, s_sum, s_d8);
            }
        } else {
            for (int t = 0; t < ntok; ++t) {
                if (!((need >> t) & 1u)) continue;
                uint8_t *tq = reinterpret_cast<uint8_t *>(s_qs) + (size_t)t * tstride;
                uint8_t *ts = s_sum + (size_t)t * tstride;
                float *td = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(s_d8) + (size_t)t * tstride);
                const uint4 *gq = reinterpret_cast<const uint4 *>(p.qs + t * K);
                for (int64_t i = threadIdx.x; i < K / 16; i += 256) reinterpret_cast<uint4 *>(tq)[i] = gq[i];
                if constexpr (PAIRS) {
                    // sum of each 32-element sub-block = two consecutive bsums
                    const int *gb = reinterpret_cast<const int *>(p.bs + t * (K / 16));
                    for (int64_t i = threadIdx.x; i < K / 32; i += 256) {
                        const int v = gb[i];
                        reinterpret_cast<int *>(ts)[i] = (int)(int16_t)(v & 0xFFFF) + (v >> 16);
                    }
                } else {
                    const uint4 *gb = reinterpret_cast<const uint4 *>(p.bs + t * (K / 16));
                    for (int64_t i = threadIdx.x; i < K / 128; i += 256) reinterpret_cast<uint4 *>(ts)[i] = gb[i];
                }
                for (int64_t i = threadIdx.x; i < nsb; i += 256) td[i] = p.d8[t * nsb + i];
            }
        }
    };
    // the token rows this block's matrices read (grouped: matrix m reads row
    // m % ntok, and a block's items span a few consecutive matrices, so it
    // stages only those rows; otherwise all of them)
    uint32_t need = 0xFFFFFFFFu;
    if constexpr (GR) {
        need = 0u;
        if (I0 < I1) {
            auto mat = [&](int64_t g) {
                int m = 0;
                while (m + 1 < p.nmat && g >= p.gpre[m + 1]) ++m;
                return m;
            };
            const int mB = mat((I1 - 1) / nsb);
            for (int mm = mat(I0 / nsb); mm <= mB; ++mm) need |= 1u << (mm % ntok);
        }
    }
    // Set-up that needs nothing written by earlier kernels: the row-group
    // prefix sums, the mbarriers, the non-grouped matrices' planes.
    if constexpr (GR) {
        if (threadIdx.x < GEMV_MAX_MATRICES) s_row_e[threadIdx.x] = -1;
    } else if (threadIdx.x < p.nmat) {
        s_planes[threadIdx.x] = make_planes(F, p.packed[threadIdx.x], p.N[threadIdx.x], nsb);
        s_n[threadIdx.x] = p.N[threadIdx.x];
        s_y[threadIdx.x] = p.y[threadIdx.x];
    }
    if (threadIdx.x <= p.nmat) s_gpre[threadIdx.x] = p.gpre[threadIdx.x];
    if (lane == 0) {
        for (int i = 0; i < D; ++i) sm100::mbar_init(&bars[i], 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();

    // matrix holding row group g
    const int nmat = p.nmat;
    auto matrix_of_group = [&](int64_t g) {
        int m = 0;
        while (m + 1 < nmat && g >= s_gpre[m + 1]) ++m;
        return m;
    };

    // issue side (lane 0): runs D items ahead of the fold along the warp's
    // range; one mbarrier phase per item and stage.  Within a matrix the
    // items are consecutive chunks of every plane.
    const LaneOff lo = lane_off(lane);
    const uint64_t pol = weight_stream_policy();
    int64_t iit = w0, inext = 0;
    int im = 0, iss = 0;
    ChunkPtr icp{};
    // fold side: row group g (of matrix m), superblock sb of the current item
    const int64_t g0 = w0 / nsb;
    const int sb0 = (int)(w0 - g0 * nsb);
    const int m0 = matrix_of_group(g0);
    // Plan of the shared row groups, made before the wait so that none of
    // it is on the path after the previous kernel completes.
    if (lane < 2) {
        const int slot = lane;
        const int64_t g = slot == 0 ? g0 : (w1 - 1) / nsb;
        const bool rec = w0 < w1 && (slot == 0 ? g * nsb < w0 : (g * nsb >= w0 && (g + 1) * nsb > w1));
        int mask = 0;
        if (rec) {
            const int64_t lo = g * nsb, hi = lo + nsb;
            for (int w = 0; w < 8; ++w) {
                const int64_t a = I0 + w * (I1 - I0) / 8, b = I0 + (w + 1) * (I1 - I0) / 8;
                if (a < b && a < hi && b > lo) mask |= 1 << w;
            }
            if ((mask & ((1 << warp) - 1)) != 0) mask = 0;  // a lower warp finishes it
            const int mm = matrix_of_group(g);
            s_fin_m[warp][slot] = mm;
            s_fin_row[warp][slot] = (g - s_gpre[mm]) * GROUP_ROWS;
            s_fin_cut[warp][slot] = lo < I0 ? (int64_t)blockIdx.x - 1 : (hi > I1 ? (int64_t)blockIdx.x : -1);
        }
        s_fin_mask[warp][slot] = rec ? mask : -1;
    }
    if constexpr (GR) {
        // the expert offsets are written by the kernels before this one.
        // Expert e holds rows [offsets[e], offsets[e+1]); the ranges are
        // disjoint, so each of the first ntok rows is claimed by at most one
        // expert.  All experts are looked at in parallel: one round trip to
        // the offsets instead of a binary search's chain of dependent loads.
        griddep_wait();
        for (int64_t e = threadIdx.x; e < p.E; e += blockDim.x) {
            const int64_t lo = p.offsets[e], hi = p.offsets[e + 1];
            for (int64_t m = lo < 0 ? 0 : lo; m < hi && m < ntok; ++m) s_row_e[m] = e;
        }
        __syncthreads();
        if (threadIdx.x < p.nmat) {
            const int mm = threadIdx.x;
            const int set = mm / ntok, m = mm - set * ntok;  // weight set, activation row
            const int64_t e = s_row_e[m];
            const bool in = e >= 0;
            // (packed, N, y are per matrix: the set's values repeated ntok times)
            s_planes[mm] = make_planes(F, p.packed[mm] + (in ? (uint64_t)e * p.expert_bytes[set] : 0), p.N[mm], nsb);
            s_n[mm] = in ? p.N[mm] : 0;  // a row of no expert is not written
            s_y[mm] = p.y[mm] + (int64_t)m * p.N[mm];
        }
        __syncthreads();
    }
    if (w0 < w1) {
        im = m0;
        icp = chunk_ptr<F>(s_planes[im], (uint64_t)(w0 - s_gpre[im] * nsb));
        inext = s_gpre[im + 1] * nsb;
    }
    auto issue = [&]() {
        if (iit < w1) {
            if (iit == inext) {
                im = matrix_of_group(s_gpre[im + 1]);
                icp = chunk_ptr<F>(s_planes[im], 0);
                inext = s_gpre[im + 1] * nsb;
            }
            if (lane == 0) item_issue<F>(icp, ring_s + iss * SLOT, smem_addr(&bars[iss]), true, pol);
            iss = iss + 1 == D ? 0 : iss + 1;
            ++iit;
        }
    };
    for (int i = 0; i < D; ++i) issue();

    // activations: written by the kernels before this one (grouped: the
    // wait is above); staged while the first items stream in
    if constexpr (!GR) griddep_wait();
    stage_rows(need);
    __syncthreads();

    int rs = 0;
    uint32_t rph = 0;  // parity of the current use of stage rs
    int64_t g = g0;
    int sb = sb0;
    int m = m0;
    // running shared addresses of the current item's activation superblock
    // (the lane's half), sums and scale
    // staged activation row of matrix m (grouped: m % ntok; else mstride = 0)
    auto row_off = [&](int mat) -> uint32_t { return GR ? (uint32_t)(mat % ntok) * mstride : 0u; };
    uint32_t a_cur = qs_s + row_off(m) + (uint32_t)sb * QK + 128 * h;
    uint32_t s_cur = sum_s + row_off(m) + (uint32_t)sb * 32 + 16 * h;
    uint32_t d_cur = d8_s + row_off(m) + 4 * (uint32_t)sb;
    float acc[T];
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t] = 0.0f;
    constexpr bool MMA = MmaFold<F, T>::on;
    using MItem = typename std::conditional<F == FMT_Q6_K, MmaQ6, MmaQ4>::type;
    const int gq = lane >> 2, cq = lane & 3;
    float macc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
    for (int64_t it = w0; it < w1; ++it) {
        stage_wait(&bars[rs], rph);
        const uint32_t st = ring_s + rs * SLOT;
        Item cur;
        MItem mcur;
        if constexpr (MMA) mma_read(mcur, st, gq, cq);
        else item_read(cur, st, lo, h);
        // every lane's reads of the stage are done before it is refilled
        __syncwarp();
        if (lane == 0 && iit < w1) sm100::fence_proxy_async_smem();
        issue();  // item it + D into the stage just read
        if (++rs == D) {
            rs = 0;
            rph ^= 1u;
        }
        if constexpr (T == 1) {
            int isum, msum;
            item_fold(cur, h, a_cur, s_cur, isum, msum);
            const float d8 = __uint_as_float(lds32(d_cur));
            acc[0] = fmaf(item_d(cur) * d8, static_cast<float>(isum), acc[0]);
            if constexpr (F != FMT_Q6_K) acc[0] = fmaf(-(item_dmin(cur) * d8), static_cast<float>(msum), acc[0]);
        } else if constexpr (MMA) {
            mma_fold(mcur, gq, cq, ntok, a_cur - 128u * h, s_cur - 16u * h, d_cur, tstride, macc);
        } else {
            const float dw = item_d(cur), dmw = item_dmin(cur);
#pragma unroll
            for (int t = 0; t < T; ++t) {
                if (t < ntok) {
                    int isum, msum;
                    item_fold(cur, h, a_cur + t * tstride, s_cur + t * tstride, isum, msum);
                    const float d8 = __uint_as_float(lds32(d_cur + t * tstride));
                    acc[t] = fmaf(dw * d8, static_cast<float>(isum), acc[t]);
                    if constexpr (F != FMT_Q6_K) acc[t] = fmaf(-(dmw * d8), static_cast<float>(msum), acc[t]);
                }
            }
        }
        a_cur += QK;
        s_cur += 32;
        d_cur += 4;
        if (++sb == nsb || it + 1 == w1) {
            // the warp is done with row group g: add the row's two halves
            if constexpr (T == 1) {
                const float v = acc[0] + __shfl_xor_sync(0xFFFFFFFFu, acc[0], 16);
                acc[0] = 0.0f;
                if (g * nsb >= w0 && (g + 1) * nsb <= w1) {
                    // the whole row group is this warp's
                    const int64_t n = (g - s_gpre[m]) * GROUP_ROWS + r16;
                    if (h == 0 && n < s_n[m]) s_y[m][n] = v;
                } else if (h == 0) {
                    s_rec[warp][g * nsb < w0 ? 0 : 1][0][r16] = v;
                }
            } else if constexpr (MMA) {
                // each (row, token) sum is one lane's: no halves to add
                const bool whole = g * nsb >= w0 && (g + 1) * nsb <= w1;
                const int64_t nb = (g - s_gpre[m]) * GROUP_ROWS;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = gq + 8 * (q >> 1), t = 2 * cq + (q & 1);
                    if (t < ntok) {
                        if (whole) {
                            if (nb + row < s_n[m]) s_y[m][t * s_n[m] + nb + row] = macc[q];
                        } else {
                            s_rec[warp][g * nsb < w0 ? 0 : 1][t][row] = macc[q];
                        }
                    }
                    macc[q] = 0.0f;
                }
            } else {
                const bool whole = g * nsb >= w0 && (g + 1) * nsb <= w1;
                const int64_t n = (g - s_gpre[m]) * GROUP_ROWS + r16;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float v = acc[t] + __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16);
                    acc[t] = 0.0f;
                    if (t < ntok && h == 0) {
                        if (whole) {
                            if (n < s_n[m]) s_y[m][t * s_n[m] + n] = v;
                        } else {
                            s_rec[warp][g * nsb < w0 ? 0 : 1][t][r16] = v;
                        }
                    }
                }
            }
            if (sb == nsb) {
                sb = 0;
                ++g;
                while (m + 1 < nmat && g >= s_gpre[m + 1]) ++m;
                a_cur = qs_s + row_off(m) + 128 * h;
                s_cur = sum_s + row_off(m) + 16 * h;
                d_cur = d8_s + row_off(m);
            }
        }
    }
    __syncthreads();

    // Row groups shared by several warps: the lowest of them adds all the
    // warps' partial sums in warp order.  A row group this block holds only
    // part of is finished by whichever of its two blocks arrives second,
    // which adds the two blocks' partial sums: a sum of two terms, so the
    // result does not depend on which block that is.  No wait and no fence:
    // the exchanged word carries the value itself.
#pragma unroll 1
    for (int slot = 0; slot < 2; ++slot) {
        const int mask = s_fin_mask[warp][slot];
        if (mask <= 0) continue;
        // every warp after the first that holds part of the group holds it
        // in its slot 0
        const int mm = s_fin_m[warp][slot];
        const int64_t n = s_fin_row[warp][slot] + r16, cut = s_fin_cut[warp][slot];
        if constexpr (T > 1) {
            // (a launch folding several tokens never cuts row groups)
            for (int t = 0; t < ntok; ++t) {
                float v = s_rec[warp][slot][t][r16];
#pragma unroll
                for (int w = 1; w < 8; ++w)
                    if (w > warp && ((mask >> w) & 1)) v += s_rec[w][0][t][r16];
                if (h == 0 && n < s_n[mm]) s_y[mm][t * s_n[mm] + n] = v;
            }
            continue;
        }
        float v = s_rec[warp][slot][0][r16];
#pragma unroll
        for (int w = 1; w < 8; ++w)
            if (w > warp && ((mask >> w) & 1)) v += s_rec[w][0][0][r16];
        if (cut < 0) {
            if (h == 0 && n < s_n[mm]) s_y[mm][n] = v;
            continue;
        }
        // The row group is cut between blocks cut and cut + 1.  Each of the
        // two swaps its partial sum, tagged, into the row's workspace word;
        // the one that gets the other's tagged value back arrives second,
        // adds the two and empties the word for the next call.
        unsigned long long *word = p.ws + cut * 16 + r16;
        if (h == 0) {
            const unsigned long long old = atomicExch(word, GEMV_TAG | __float_as_uint(v));
            if (old & GEMV_TAG) {
                if (n < s_n[mm]) s_y[mm][n] = v + __uint_as_float((uint32_t)old);
                *word = 0ull;
            }
        }
    }
}

static int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Above this many items per SM a launch takes two blocks per SM (more warps
// folding), giving up the room for the next kernel's block -- unless K is
// very long, since every block quantizes the whole row.  (Measured on GB300,
// the 27B-shaped FFN at M = 1 with its down projection of K = 17408 in two
// blocks per SM: 32.8 vs 34.2 us per gate/up + down step.)
#ifndef KQ_GEMV_TWO_BLOCKS_ITEMS_PER_SM
#define KQ_GEMV_TWO_BLOCKS_ITEMS_PER_SM 100
#endif
#ifndef KQ_GEMV_TWO_BLOCKS_MAX_NSB
#define KQ_GEMV_TWO_BLOCKS_MAX_NSB 80
#endif

// Blocks per SM of a grouped-rows (MoE decode) launch: its weights are
// known only after the wait, so nothing is prefetched beside the previous
// kernel, and more warps folding is what counts.
#ifndef KQ_GEMV_GR_BLOCKS_PER_SM
#define KQ_GEMV_GR_BLOCKS_PER_SM 2
#endif

#ifndef KQ_GEMV_CUT_ITEMS
#define KQ_GEMV_CUT_ITEMS 3
#endif

// Shared memory of one block (dynamic part), at most half an SM's so that
// a block of the next GEMV in the stream fits beside it and starts its
// weight stream while this one finishes.
constexpr int64_t GEMV_SMEM_BUDGET = 110 * 1024;

template <int F> constexpr int gemv_max_d() { return F == FMT_Q6_K ? 4 : (F == FMT_Q5_K ? 5 : 6); }

// Shared memory of a block folding several tokens per pass: it holds their
// staged rows, so it takes up to 200 KB for the ring and rows (212 KB when a
// long row leaves only the minimum ring): one block per SM, no room for the
// next kernel's block.
constexpr int64_t GEMV_BATCH_SMEM_BUDGET = 200 * 1024;
constexpr int64_t GEMV_BATCH_MAX_SMEM = 212 * 1024;  // + the static ~9 KB stays within 227 KB

// bytes of one token's staged row (quants, sums, scales), 16-byte aligned
inline int64_t gemv_stage_stride(int64_t K) { return (K + K / 8 + K / 64 + 15) & ~int64_t(15); }

template <int F, int T, bool GR = false>
static cudaError_t launch_gemv_t(GemvParams p, void *ws, size_t ws_bytes, cudaStream_t s) {
    p.gpre[0] = 0;
    for (int m = 0; m < p.nmat; ++m) p.gpre[m + 1] = p.gpre[m] + (p.N[m] + 15) / 16;
    const int64_t G = p.gpre[p.nmat];
    if (G == 0) return cudaSuccess;
    p.items = G * p.nsb;
    p.stage_stride = gemv_stage_stride(p.K);
    if (T == 1 && !GR) p.ntok = 1;
    // (a grouped launch stages its ntok activation rows; a pass of a few
    // tokens keeps to half an SM while its rows leave room for a 3-stage ring)
    const int64_t rows_bytes = (GR ? p.ntok : T) * gemv_stage_stride(p.K);
    const bool wide = (GR && KQ_GEMV_GR_BLOCKS_PER_SM == 1) ||
                      ((T > 1 || GR) && (GEMV_SMEM_BUDGET - rows_bytes) / (8 * GemvFmt<F>::SLOT) < 3);
    // one block per SM, each with an even share of the items; a row group
    // may then be cut between two blocks, which needs the workspace
    int64_t blocks = sm_count();
    if (T == 1 && !GR && p.items > (int64_t)KQ_GEMV_TWO_BLOCKS_ITEMS_PER_SM * blocks && p.nsb <= KQ_GEMV_TWO_BLOCKS_MAX_NSB)
        blocks *= 2;
    if (GR && !wide) blocks *= KQ_GEMV_GR_BLOCKS_PER_SM;
    if (blocks > GEMV_MAX_BLOCKS) blocks = GEMV_MAX_BLOCKS;
    if (blocks > G) blocks = G;  // every row group spans at most two blocks
    // cut row groups between blocks only where whole row groups would leave
    // the busiest warp KQ_GEMV_CUT_ITEMS or more items above an even share:
    // the exchange at a cut costs about as much as folding a few items
    const int64_t whole = (G + blocks - 1) / blocks * p.nsb, even = (p.items + blocks - 1) / blocks;
    p.split = T == 1 && !GR && ws != nullptr && ws_bytes >= GEMV_WORKSPACE_BYTES && blocks > 1 &&
              ((launch_flags() & LAUNCH_GEMV_SPLIT) || (whole + 7) / 8 - (even + 7) / 8 >= KQ_GEMV_CUT_ITEMS);
    p.ws = static_cast<unsigned long long *>(ws);
    const int64_t budget = wide ? GEMV_BATCH_SMEM_BUDGET : GEMV_SMEM_BUDGET;
    const int64_t stage_bytes = (GR ? p.ntok : T) * p.stage_stride;
    int64_t D = (budget - stage_bytes) / (8 * GemvFmt<F>::SLOT);
    if (D > gemv_max_d<F>()) D = gemv_max_d<F>();
    if (D < 2) D = 2;
    p.D = (int)D;
    const size_t smem = (size_t)(8 * D * GemvFmt<F>::SLOT + stage_bytes);
    // per-device attributes of this instantiation, set once on every device
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        // the largest this instantiation may ask for (a launch asks for what it uses)
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<F, T, GR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)((T > 1 || GR) ? GEMV_BATCH_MAX_SMEM : GEMV_SMEM_BUDGET));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemv_kernel<F, T, GR>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<F, T, GR>, p);
}

template <int F>
static cudaError_t launch_gemv_f(GemvParams p, void *ws, size_t ws_bytes, cudaStream_t s) {
    return launch_gemv_t<F, 1>(p, ws, ws_bytes, s);
}

cudaError_t launch_gemv(int f, int nmat, const void *const *packed, const int64_t *N, int64_t K, const float *x,
                        Q8K a, float *const *y, void *ws, size_t ws_bytes, cudaStream_t s) {
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
    if (f == FMT_Q4_K) return launch_gemv_f<FMT_Q4_K>(p, ws, ws_bytes, s);
    if (f == FMT_Q5_K) return launch_gemv_f<FMT_Q5_K>(p, ws, ws_bytes, s);
    return launch_gemv_f<FMT_Q6_K>(p, ws, ws_bytes, s);
}

// Small batches (M token rows, M < the tensor-core GEMM's minimum): passes of
// up to 8 tokens, each reading every weight item once for all its tokens.
int64_t gemv_batch_max_tokens(int64_t K) {
    int64_t t = 8;
    while (t > 1 && t * gemv_stage_stride(K) + 2 * 8 * 3360 > GEMV_BATCH_MAX_SMEM) t >>= 1;
    return t;
}

template <int F>
static cudaError_t launch_gemv_batch_f(GemvParams p, int64_t M, int64_t tmax, void *ws, size_t ws_bytes,
                                       cudaStream_t s) {
    float *y0[GEMV_MAX_MATRICES];
    for (int m = 0; m < p.nmat; ++m) y0[m] = p.y[m];
    const float *x0 = p.x;
    const int8_t *q0 = p.qs;
    const int16_t *b0 = p.bs;
    const float *d0 = p.d8;
    for (int64_t t0 = 0; t0 < M; t0 += tmax) {
        const int64_t n = M - t0 < tmax ? M - t0 : tmax;
        p.ntok = (int)n;
        for (int m = 0; m < p.nmat; ++m) p.y[m] = y0[m] + t0 * p.N[m];
        if (x0) {
            p.x = x0 + t0 * p.K;
        } else {
            p.qs = q0 + t0 * p.K;
            p.bs = b0 + t0 * (p.K / 16);
            p.d8 = d0 + t0 * p.nsb;
        }
        cudaError_t e;
        if (n > 4) e = launch_gemv_t<F, 8>(p, nullptr, 0, s);
        else if (n > 2) e = launch_gemv_t<F, 4>(p, nullptr, 0, s);
        else if (n > 1) e = launch_gemv_t<F, 2>(p, nullptr, 0, s);
        else e = launch_gemv_t<F, 1>(p, ws, ws_bytes, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Grouped rows (MoE decode: a few token rows, each routed to an expert):
// one launch over every row's expert matrix, from one read of each weight
// item per row.  False when the rows' staged activations do not fit.
bool gemv_grouped_fits(int64_t M, int64_t K, int sets) {
    return M >= 1 && sets >= 1 && M * sets <= GEMV_MAX_MATRICES &&
           M * gemv_stage_stride(K) + 2 * 8 * 3360 <= GEMV_BATCH_MAX_SMEM;
}

cudaError_t launch_gemv_grouped(int f, int sets, const void *const *packed, const int64_t *N, int64_t E,
                                const int32_t *offsets, uint64_t const *expert_bytes, int64_t K, Q8K a,
                                const float *x, int64_t M, float *const *y, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    GemvParams p{};
    p.nmat = (int)(sets * M);
    for (int m = 0; m < p.nmat; ++m) {
        p.packed[m] = static_cast<const uint8_t *>(packed[m / M]);  // the matrix's set: its experts,
        p.N[m] = N[m / M];     // their shape (launch_gemv_t takes the row-group prefix sums from N)
        p.y[m] = y[m / M];     // and its output
    }
    p.K = K;
    p.nsb = K / QK;
    p.x = x;
    p.d8 = a.d;
    p.qs = a.qs;
    p.bs = a.bsums;
    p.ntok = (int)M;
    p.offsets = offsets;
    p.E = E;
    for (int st = 0; st < sets; ++st) p.expert_bytes[st] = expert_bytes[st];
    if (f == FMT_Q4_K) return launch_gemv_t<FMT_Q4_K, 1, true>(p, nullptr, 0, s);
    if (f == FMT_Q5_K) return launch_gemv_t<FMT_Q5_K, 1, true>(p, nullptr, 0, s);
    return launch_gemv_t<FMT_Q6_K, 1, true>(p, nullptr, 0, s);
}

cudaError_t launch_gemv_batch(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, float *y,
                              cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    GemvParams p{};
    p.nmat = 1;
    p.packed[0] = static_cast<const uint8_t *>(packed);
    p.N[0] = N;
    p.y[0] = y;
    p.K = K;
    p.nsb = K / QK;
    p.x = nullptr;
    p.d8 = a.d;
    p.qs = a.qs;
    p.bs = a.bsums;
    const int64_t tmax = gemv_batch_max_tokens(K);
    if (f == FMT_Q4_K) return launch_gemv_batch_f<FMT_Q4_K>(p, M, tmax, nullptr, 0, s);
    if (f == FMT_Q5_K) return launch_gemv_batch_f<FMT_Q5_K>(p, M, tmax, nullptr, 0, s);
    return launch_gemv_batch_f<FMT_Q6_K>(p, M, tmax, nullptr, 0, s);
}

// The fused quantize + GEMV for a small batch: M fp32 rows x, up to four
// matrices sharing them, y[m] [M][N[m]].
cudaError_t launch_gemv_fused_batch(int f, int nmat, const void *const *packed, const int64_t *N, int64_t K,
                                    const float *x, int64_t M, float *const *y, void *ws, size_t ws_bytes,
                                    cudaStream_t s) {
    if (M == 0) return cudaSuccess;
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
    const int64_t tmax = gemv_batch_max_tokens(K);
    if (f == FMT_Q4_K) return launch_gemv_batch_f<FMT_Q4_K>(p, M, tmax, ws, ws_bytes, s);
    if (f == FMT_Q5_K) return launch_gemv_batch_f<FMT_Q5_K>(p, M, tmax, ws, ws_bytes, s);
    return launch_gemv_batch_f<FMT_Q6_K>(p, M, tmax, ws, ws_bytes, s);
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
    if (lane == 0) item_issue<F>(cp, smem_addr(s_item[warp]), smem_addr(&s_bar[warp]), on, weight_stream_policy());
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

// Test hook: the integer sums of the 8-token passes' integer-MMA fold
// (MmaFold, Q4_K and Q6_K), per (token, row, superblock).  One warp per
// (row group, superblock): the item is fetched with item_issue, the M <= 8
// token rows' superblock staged side by side as the batch kernel stages
// them (quants, then the sums the fold needs), and mma_read + mma_isums
// run on them as in the batch kernel.
template <int F>
__global__ void __launch_bounds__(32) mma_partials_kernel(const uint8_t *packed, int64_t N, int64_t nsb, int64_t K,
                                                          Q8K a, int ntok, int32_t *isum_out, int32_t *msum_out) {
    constexpr int SLOT = GemvFmt<F>::SLOT;
    constexpr uint32_t TSTRIDE = 304;  // 256 quants + 32 bytes of sums + d8, 16-byte aligned
    __shared__ __align__(128) uint8_t s_item[SLOT];
    __shared__ __align__(16) uint8_t s_tok[8 * TSTRIDE];
    __shared__ uint64_t s_bar;
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x, sb = blockIdx.y;
    for (int t = 0; t < ntok; ++t) {
        reinterpret_cast<uint2 *>(s_tok + t * TSTRIDE)[lane] =
            reinterpret_cast<const uint2 *>(a.qs + t * K + sb * QK)[lane];
        const int16_t *gb = a.bsums + (t * nsb + sb) * 16;
        if constexpr (F != FMT_Q6_K) {
            if (lane < 8) reinterpret_cast<int *>(s_tok + t * TSTRIDE + 256)[lane] = (int)gb[2 * lane] + (int)gb[2 * lane + 1];
        } else {
            if (lane < 16) reinterpret_cast<int16_t *>(s_tok + t * TSTRIDE + 256)[lane] = gb[lane];
        }
    }
    if (lane == 0) {
        sm100::mbar_init(&s_bar, 1);
        sm100::mbar_fence_init();
    }
    __syncwarp();
    const Planes P = make_planes(F, packed, N, nsb);
    ChunkPtr cp = chunk_ptr<F>(P, (uint64_t)g * nsb + sb);
    if (lane == 0) item_issue<F>(cp, smem_addr(s_item), smem_addr(&s_bar), true, weight_stream_policy());
    stage_wait(&s_bar, 0);
    using MItem = typename std::conditional<F == FMT_Q6_K, MmaQ6, MmaQ4>::type;
    const int gq = lane >> 2, cq = lane & 3;
    MItem w;
    mma_read(w, smem_addr(s_item), gq, cq);
    int isum[4], msum[4];
    mma_isums(w, gq, cq, ntok, smem_addr(s_tok), smem_addr(s_tok) + 256u, TSTRIDE, isum, msum);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int t = 2 * cq + k;
            const int64_t n = g * GROUP_ROWS + gq + 8 * rr;
            if (t < ntok && n < N) {
                const int64_t o = ((int64_t)t * N + n) * nsb + sb;
                isum_out[o] = isum[rr * 2 + k];
                msum_out[o] = msum[rr * 2 + k];
            }
        }
}

cudaError_t launch_mma_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, int32_t *isum,
                                int32_t *msum, cudaStream_t s) {
    if (M == 0 || N == 0) return cudaSuccess;
    const int64_t nsb = K / QK;
    dim3 grid((unsigned)row_groups(N), (unsigned)nsb);
    const uint8_t *pk = static_cast<const uint8_t *>(packed);
    if (f == FMT_Q4_K) mma_partials_kernel<FMT_Q4_K><<<grid, 32, 0, s>>>(pk, N, nsb, K, a, (int)M, isum, msum);
    else mma_partials_kernel<FMT_Q6_K><<<grid, 32, 0, s>>>(pk, N, nsb, K, a, (int)M, isum, msum);
    return cudaGetLastError();
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
