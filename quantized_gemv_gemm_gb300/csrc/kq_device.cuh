// kq_device.cuh - device-side building blocks shared by the libkq kernels:
// the packed-image layout, streaming loads, and the per-lane unpack + integer
// fold of one 256-weight superblock for each K-quant format.
//
// [kq-arc] = the page "dasLLAMA: K-quant kernel arc - kq v2 integer folds,
// kq v3 panel-scratch tiles, chain regrain, parity gates" (daScript #3450).
//
// Lane geometry (GEMV, small-M and partials kernels).  Four consecutive lanes
// ("a quad") own one weight row; lane c = lane & 3 of the quad owns 64 of the
// superblock's 256 weights, so one warp covers 8 rows of one superblock:
//   Q4_K/Q5_K: lane c reads qs bytes [16c, 16c+16) and [64+16c, 64+16c+16).
//     Byte b of qs holds element 64*(b/32) + b%32 (low nibble, sub-block
//     2*(b/32)) and element 64*(b/32) + 32 + b%32 (high nibble, sub-block
//     2*(b/32)+1), so lane c owns sub-blocks {2k, 2k+1, 2k+4, 2k+5}, k = c/2,
//     at element offsets 16*(c&1) .. +15 inside each.
//   Q6_K: lane c = (half h = c/2, p = c&1) reads ql[64h+16p ..+16],
//     ql[64h+32+16p ..+16] and qh[32h+16p ..+16]; it owns the four 16-wide
//     sub-blocks 8h + 2t + p, t = 0..3.
// Each warp-wide load instruction covers whole 32-byte sectors.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace kq {

constexpr int QK = 256;
constexpr int FMT_Q4_K = 1, FMT_Q5_K = 2, FMT_Q6_K = 3;

__host__ __device__ inline int block_bytes(int f) {
    return f == FMT_Q4_K ? 144 : f == FMT_Q5_K ? 176 : f == FMT_Q6_K ? 210 : 0;
}

__host__ __device__ inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// ---------------------------------------------------------------------------
// The packed image ("grp16"; the row interleave of [kq-arc]'s grp<mr>
// repack, with mr = 16 rows).  Rows are taken in groups of 16 (the last one
// padded with zero rows); each plane holds, for every (row group g,
// superblock sb) in the order g * nsb + sb, one chunk with that plane's
// bytes of the 16 rows' superblock sb.  Inside a chunk (r = row in the
// group, h = half of the superblock, lane = r + 16h):
//   qs / ql  128 B per row:  piece k (bytes 64h+16k .. +15) of row r at
//                            512k + 16*lane                  chunk 2048 B
//   hdr      Q4_K/Q5_K d, dmin, scales[12] of row r at 16r     256 B
//   qh (Q5)  32 B per row:   piece j (bytes 16j .. +15) at 256j + 16r      512 B
//   qh (Q6)  64 B per row:   piece j of half h (bytes 32h+16j ..) at
//                            512j + 16*lane                 1024 B
//   sc (Q6)  16 signed scales of row r at 16r                 256 B
//   d  (Q6)  fp16 d of row r at 2r                              32 B
// So every chunk is contiguous and 16-byte aligned (one bulk copy), a warp
// serving 16 rows x one superblock reads consecutive 16-byte pieces, and a
// row's next superblock is one chunk further on in every plane.  Every disk
// byte is kept as it is; only its place changes.  A small bounds plane
// (below) follows the data planes.
constexpr int GROUP_ROWS = 16;

__host__ __device__ inline int64_t row_groups(int64_t N) { return (N + GROUP_ROWS - 1) / GROUP_ROWS; }

// Bytes per row and superblock of each plane (chunk = 16 x this).
__host__ __device__ inline void plane_unit_bytes(int f, int u[4]) {
    u[0] = 128; u[1] = 0; u[2] = 0; u[3] = 0;
    if (f == FMT_Q4_K) { u[1] = 16; }
    else if (f == FMT_Q5_K) { u[1] = 32; u[2] = 16; }
    else if (f == FMT_Q6_K) { u[1] = 64; u[2] = 16; u[3] = 2; }
}

// Bounds plane (derived at repack time, read by the tensor-core GEMM only):
// per (row group g, superblock sb), in the order g * nsb + sb, two uint32:
// for each half of the superblock (K 0..127, 128..255) the largest over the
// group's 16 rows of W1 = sum |w'| = sum over the half's sub-blocks of
// |sub-scale| * sum |q| (Q4_K/Q5_K q, Q6_K q - 32).  Any partial sum of
// w' * a8 over a row's half is at most 128 * W1 in magnitude (|a8| <= 128),
// so an fp32 accumulator over it stays exact while 128 * W1 <= 2^24.
constexpr int BOUND_BYTES = 8;

// Offsets of the planes of an [N][K] image: the data planes 0..3, the
// bounds plane at off[4]; off[5] = total bytes.
__host__ __device__ inline void plane_offsets(int f, int64_t N, int64_t nsb, uint64_t off[6]) {
    int u[4];
    plane_unit_bytes(f, u);
    const uint64_t units = (uint64_t)row_groups(N) * GROUP_ROWS * (uint64_t)nsb;
    off[0] = 0;
    for (int i = 0; i < 4; ++i) off[i + 1] = off[i] + align256(units * (uint64_t)u[i]);
    off[5] = off[4] + align256((uint64_t)row_groups(N) * (uint64_t)nsb * BOUND_BYTES);
}

// Plane base pointers of one packed matrix (p4: the bounds plane).
struct Planes {
    const uint8_t *p0, *p1, *p2, *p3, *p4;
};

__host__ __device__ inline Planes make_planes(int f, const void *base, int64_t N, int64_t nsb) {
    uint64_t off[6];
    plane_offsets(f, N, nsb, off);
    const uint8_t *b = static_cast<const uint8_t *>(base);
    return Planes{b + off[0], b + off[1], b + off[2], b + off[3], b + off[4]};
}

// Chunk index of (row n, superblock sb): the chunk of n's row group at sb.
__host__ __device__ inline uint64_t chunk_of(int64_t n, int64_t sb, int64_t nsb) {
    return (uint64_t)(n / GROUP_ROWS) * (uint64_t)nsb + (uint64_t)sb;
}

// Byte offset, inside a chunk, of the 16-byte piece holding row r's bytes
// [16i, 16i+16) of a plane with `ub` bytes per row (ub = 128, 64, 32, 16);
// the d plane (ub = 2) is at 2r.
__host__ __device__ inline uint32_t piece_offset(int ub, int r, int i) {
    if (ub == 128) return 512u * (i & 3) + 16u * (r + 16 * (i >> 2));
    if (ub == 64) return 512u * (i & 1) + 16u * (r + 16 * (i >> 1));
    if (ub == 32) return 256u * i + 16u * r;
    return 16u * r;  // ub == 16
}

// ---------------------------------------------------------------------------
// loads

// Weight bytes are read exactly once per kernel: do not allocate them in L1.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Small data shared by the lanes of a quad (scale headers) and activations,
// which every warp of the block re-reads: keep them in L1.
__device__ __forceinline__ uint4 ld_keep(const void *p) {
    return __ldg(static_cast<const uint4 *>(p));
}
__device__ __forceinline__ int4 ld_act16(const int8_t *p) {
    return __ldg(reinterpret_cast<const int4 *>(p));
}

__device__ __forceinline__ int dp4a(uint32_t a, int b, int c) {
    return __dp4a(static_cast<int>(a), b, c);
}

__device__ __forceinline__ int dot16(uint4 q, int4 a) {
    int s = dp4a(q.x, a.x, 0);
    s = dp4a(q.y, a.y, s);
    s = dp4a(q.z, a.z, s);
    return dp4a(q.w, a.w, s);
}

__device__ __forceinline__ uint4 and4(uint4 v, uint32_t m) {
    return make_uint4(v.x & m, v.y & m, v.z & m, v.w & m);
}
__device__ __forceinline__ uint4 shr4(uint4 v, int s) {
    return make_uint4(v.x >> s, v.y >> s, v.z >> s, v.w >> s);
}

__device__ __forceinline__ float half_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// ---------------------------------------------------------------------------
// The 12-byte six-bit scale/min block of Q4_K and Q5_K ([kq-arc], k4 kq-v2
// commit: fp16 d and dmin, then 12 bytes of packed 6-bit fields; k5/k6
// commit: the Q5_K scale block is the Q4_K one).  With y, z, w = scale bytes 0..3, 4..7, 8..11
// (little-endian words), byte j of the results is:
//   sc_lo: sub-scale j   (j < 4) = low 6 bits of scale byte j
//   m_lo : sub-min j     (j < 4) = low 6 bits of scale byte 4+j
//   sc_hi: sub-scale 4+j = low nibble of byte 8+j | top 2 bits of byte j  << 4
//   m_hi : sub-min   4+j = high nibble of byte 8+j | top 2 bits of byte 4+j << 4
struct ScaleMin {
    uint32_t sc_lo, sc_hi, m_lo, m_hi;
};

__device__ __forceinline__ ScaleMin unpack_scale_min(uint4 hdr) {
    ScaleMin r;
    r.sc_lo = hdr.y & 0x3F3F3F3Fu;
    r.m_lo = hdr.z & 0x3F3F3F3Fu;
    r.sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    r.m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    return r;
}

__device__ __forceinline__ int byte_of(uint32_t w, int i) { return (w >> (8 * i)) & 0xFF; }

// ---------------------------------------------------------------------------
// Per-lane weight registers of one superblock, and their loads.

struct WQ4 { uint4 qa, qb, hdr; };
struct WQ5 { uint4 qa, qb, qh, hdr; };
struct WQ6 { uint4 la, lb, qh, sc; uint32_t d; };

template <int F> struct WRegs;
template <> struct WRegs<FMT_Q4_K> { using T = WQ4; };
template <> struct WRegs<FMT_Q5_K> { using T = WQ5; };
template <> struct WRegs<FMT_Q6_K> { using T = WQ6; };

// Per-lane plane pointers at (row n, superblock sb) for the quad geometry
// above; the row's next superblock is one chunk further on in every plane
// (chunk bytes 2048 / 256 / 512 / 1024 / 32), so a lane walks a row by
// adding i chunks (load_at).
struct LanePtr {
    const uint8_t *p0, *p1, *p2, *p3;
};

template <int F>
__device__ __forceinline__ LanePtr lane_ptr(const Planes &P, int64_t n, int64_t sb, int64_t nsb, int c) {
    const uint64_t ch = chunk_of(n, sb, nsb);
    const int r = (int)(n % GROUP_ROWS);
    LanePtr q;
    if constexpr (F == FMT_Q4_K || F == FMT_Q5_K) {
        // qs bytes [16c, 16c+16) = piece c; [64+16c, ..) = piece 4 + c
        q.p0 = P.p0 + ch * 2048 + piece_offset(128, r, c);
        if constexpr (F == FMT_Q4_K) {
            q.p1 = P.p1 + ch * 256 + 16 * r;
            q.p2 = q.p3 = nullptr;
        } else {
            q.p1 = P.p1 + ch * 512 + piece_offset(32, r, c & 1);
            q.p2 = P.p2 + ch * 256 + 16 * r;
            q.p3 = nullptr;
        }
    } else {
        const int h = c >> 1, p = c & 1;
        // ql bytes [64h+16p, ..) = piece 4h + p; [64h+32+16p, ..) = piece 4h + 2 + p
        q.p0 = P.p0 + ch * 2048 + piece_offset(128, r, 4 * h + p);
        q.p1 = P.p1 + ch * 1024 + piece_offset(64, r, 2 * h + p);
        q.p2 = P.p2 + ch * 256 + 16 * r;
        q.p3 = P.p3 + ch * 32 + 2 * r;
    }
    return q;
}

// piece 4 + c of qs sits 16 rows further on: +256 bytes; piece 2 + p of ql: +1024
__device__ __forceinline__ void load_at(WQ4 &w, const LanePtr &lp, int64_t i) {
    w.qa = ld_stream(lp.p0 + i * 2048);
    w.qb = ld_stream(lp.p0 + i * 2048 + 256);
    w.hdr = ld_keep(lp.p1 + i * 256);
}
__device__ __forceinline__ void load_at(WQ5 &w, const LanePtr &lp, int64_t i) {
    w.qa = ld_stream(lp.p0 + i * 2048);
    w.qb = ld_stream(lp.p0 + i * 2048 + 256);
    w.qh = ld_stream(lp.p1 + i * 512);
    w.hdr = ld_keep(lp.p2 + i * 256);
}
__device__ __forceinline__ void load_at(WQ6 &w, const LanePtr &lp, int64_t i) {
    w.la = ld_stream(lp.p0 + i * 2048);
    w.lb = ld_stream(lp.p0 + i * 2048 + 1024);
    w.qh = ld_stream(lp.p1 + i * 1024);
    w.sc = ld_keep(lp.p2 + i * 256);
    w.d = __ldg(reinterpret_cast<const unsigned short *>(lp.p3 + i * 32));
}

// one superblock of row n
template <typename W>
__device__ __forceinline__ void load_w(W &w, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int c);
template <>
__device__ __forceinline__ void load_w(WQ4 &w, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int c) {
    load_at(w, lane_ptr<FMT_Q4_K>(P, n, sb, nsb, c), 0);
}
template <>
__device__ __forceinline__ void load_w(WQ5 &w, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int c) {
    load_at(w, lane_ptr<FMT_Q5_K>(P, n, sb, nsb, c), 0);
}
template <>
__device__ __forceinline__ void load_w(WQ6 &w, const Planes &P, int64_t n, int64_t sb, int64_t nsb, int c) {
    load_at(w, lane_ptr<FMT_Q6_K>(P, n, sb, nsb, c), 0);
}

// ---------------------------------------------------------------------------
// Decoded per-lane quants: four groups of 16 stored quant bytes (one uint4
// each, bytes 0..63) with their sub-scales, plus the lane's share of the
// min term.  Decoding is done once per superblock and reused for every token.

struct LaneQ {
    uint4 g[4];     // stored quants of the lane's four 16-element groups
    int sc[4];      // sub-scale of each group
    int aoff[4];    // element offset of each group inside the superblock
    // Q4_K/Q5_K: lane c's mins m_{2c}, m_{2c+1} (bsums 4c..4c+3)
    // Q6_K: unused (the -32 offset goes through sc and the group's bsum)
    int m0, m1;
    float d, dmin;  // super-scales
};

__device__ __forceinline__ void decode_lane(const WQ4 &w, int c, LaneQ &L) {
    const int k = c >> 1, o = 16 * (c & 1);
    const ScaleMin s = unpack_scale_min(w.hdr);
    L.g[0] = and4(w.qa, 0x0F0F0F0Fu);            // sub-block 2k
    L.g[1] = and4(shr4(w.qa, 4), 0x0F0F0F0Fu);   // sub-block 2k+1
    L.g[2] = and4(w.qb, 0x0F0F0F0Fu);            // sub-block 2k+4
    L.g[3] = and4(shr4(w.qb, 4), 0x0F0F0F0Fu);   // sub-block 2k+5
    L.sc[0] = byte_of(s.sc_lo, 2 * k);
    L.sc[1] = byte_of(s.sc_lo, 2 * k + 1);
    L.sc[2] = byte_of(s.sc_hi, 2 * k);
    L.sc[3] = byte_of(s.sc_hi, 2 * k + 1);
    L.aoff[0] = 64 * k + o;
    L.aoff[1] = 64 * k + 32 + o;
    L.aoff[2] = 64 * (k + 2) + o;
    L.aoff[3] = 64 * (k + 2) + 32 + o;
    const uint32_t mw = (c < 2) ? s.m_lo : s.m_hi;
    L.m0 = byte_of(mw, 2 * (c & 1));
    L.m1 = byte_of(mw, 2 * (c & 1) + 1);
    L.d = half_lo(w.hdr.x);
    L.dmin = half_hi(w.hdr.x);
}

// Q5_K: the Q4_K walk plus the fifth bit ([kq-arc], k5/k6 commit: Q5_K
// differs from Q4_K only by OR-ing that high bit into each quant).  Element 64k+l takes bit 2k of
// qh[l], element 64k+32+l bit 2k+1; this lane's qh bytes are l in [o, o+16).
__device__ __forceinline__ uint4 q5_bit(uint4 qh, int bit) {
    // move bit `bit` of every byte to bit 4
    uint4 r;
    if (bit <= 4) {
        const int sh = 4 - bit;
        r = make_uint4(qh.x << sh, qh.y << sh, qh.z << sh, qh.w << sh);
    } else {
        r = shr4(qh, bit - 4);
    }
    return and4(r, 0x10101010u);
}

__device__ __forceinline__ uint4 or4(uint4 a, uint4 b) {
    return make_uint4(a.x | b.x, a.y | b.y, a.z | b.z, a.w | b.w);
}

__device__ __forceinline__ void decode_lane(const WQ5 &w, int c, LaneQ &L) {
    const int k = c >> 1;
    WQ4 w4{w.qa, w.qb, w.hdr};
    decode_lane(w4, c, L);
    L.g[0] = or4(L.g[0], q5_bit(w.qh, 2 * k));
    L.g[1] = or4(L.g[1], q5_bit(w.qh, 2 * k + 1));
    L.g[2] = or4(L.g[2], q5_bit(w.qh, 2 * k + 4));
    L.g[3] = or4(L.g[3], q5_bit(w.qh, 2 * k + 5));
}

// Q6_K ([kq-arc], k5/k6 commit: signed sub-scales, one per 16 weights): group t of lane
// (h, p) holds elements 128h + 32t + 16p .. +15 of sub-block 8h + 2t + p.
__device__ __forceinline__ void decode_lane(const WQ6 &w, int c, LaneQ &L) {
    const int h = c >> 1, p = c & 1;
    L.g[0] = or4(and4(w.la, 0x0F0F0F0Fu), make_uint4((w.qh.x << 4) & 0x30303030u, (w.qh.y << 4) & 0x30303030u,
                                                      (w.qh.z << 4) & 0x30303030u, (w.qh.w << 4) & 0x30303030u));
    L.g[1] = or4(and4(w.lb, 0x0F0F0F0Fu), make_uint4((w.qh.x << 2) & 0x30303030u, (w.qh.y << 2) & 0x30303030u,
                                                      (w.qh.z << 2) & 0x30303030u, (w.qh.w << 2) & 0x30303030u));
    L.g[2] = or4(and4(shr4(w.la, 4), 0x0F0F0F0Fu), and4(w.qh, 0x30303030u));
    L.g[3] = or4(and4(shr4(w.lb, 4), 0x0F0F0F0Fu), and4(shr4(w.qh, 2), 0x30303030u));
    // sub-block i = 8h + 2t + p sits in scale word 2h + t/2, byte 2(t&1) + p
    const uint32_t w01 = h ? w.sc.z : w.sc.x, w23 = h ? w.sc.w : w.sc.y;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t word = (t < 2) ? w01 : w23;
        L.sc[t] = static_cast<int>(static_cast<int8_t>((word >> (8 * (2 * (t & 1) + p))) & 0xFF));
        L.aoff[t] = 128 * h + 32 * t + 16 * p;
    }
    L.m0 = L.m1 = 0;
    L.d = half_lo(w.d);
    L.dmin = 0.0f;
}

// ---------------------------------------------------------------------------
// The lane's integer partials against one token's Q8_K superblock.
//   a8: the token's 256 quants of this superblock, bs: its 16 bsums.
// Q4_K/Q5_K: isum_lane = sum_g sc_g * dot16_g, msum_lane = m0*(bs_4c+bs_4c+1)
//            + m1*(bs_4c+2 + bs_4c+3)   ([kq-arc], k4 kq-v2 commit)
// Q6_K     : isum_lane = sum_t sc_t * dot16_t - 32 * sum_t sc_t * bs_(8h+2t+p),
//            msum_lane = 0                ([kq-arc], k5/k6 commit)
template <int F, bool SMEM = false>
__device__ __forceinline__ void lane_partials(const LaneQ &L, const int8_t *a8, const int16_t *bs, int c,
                                              int &isum, int &msum) {
    // SMEM: a8 / bs point into shared memory (plain loads); otherwise global
    // memory read through the read-only path.
    auto ld16 = [](const void *q) -> int4 {
        if constexpr (SMEM) return *reinterpret_cast<const int4 *>(q);
        else return __ldg(reinterpret_cast<const int4 *>(q));
    };
    int acc = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) acc += L.sc[g] * dot16(L.g[g], ld16(a8 + L.aoff[g]));
    if constexpr (F == FMT_Q6_K) {
        const int4 b = ld16(bs + 8 * (c >> 1));  // bs[8h .. 8h+7]
        const int p = c & 1;
        const uint32_t bw[4] = {(uint32_t)b.x, (uint32_t)b.y, (uint32_t)b.z, (uint32_t)b.w};
        int bacc = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int v = static_cast<int16_t>((bw[t] >> (16 * p)) & 0xFFFF);
            bacc += L.sc[t] * v;
        }
        isum = acc - 32 * bacc;
        msum = 0;
    } else {
        int2 b;
        if constexpr (SMEM) b = *reinterpret_cast<const int2 *>(bs + 4 * c);  // bs[4c .. 4c+3]
        else b = __ldg(reinterpret_cast<const int2 *>(bs + 4 * c));
        const int b0 = static_cast<int16_t>(b.x & 0xFFFF), b1 = static_cast<int16_t>(b.x >> 16);
        const int b2 = static_cast<int16_t>(b.y & 0xFFFF), b3 = static_cast<int16_t>(b.y >> 16);
        isum = acc;
        msum = L.m0 * (b0 + b1) + L.m1 * (b2 + b3);
    }
}

// Q8_K quantization of one 256-block by one warp ([kq-arc], k4 kq-v2 commit,
// quantize_q8_k_into: one fp32 scale per 256 values and a sum per 16).
// Lane l owns elements 8l .. 8l+7, given in v0 (8l .. 8l+3) and v1.
// amax = max|x| (a max over the bit patterns of |x|, which order like the
// values for finite floats); iscale = 127/amax and q = round_half_even(
// x*iscale), clamped to +-127, both single IEEE fp32 operations; d8 =
// amax/127 (0 when amax = 0, with every q = 0).  Returns the lane's eight
// quants packed in two words (element 8l in the low byte of .x) and sets
// part = the sum of the lane's eight quants, d8 = the block scale.
__device__ __forceinline__ uint2 q8k_lane(float4 v0, float4 v1, int &part, float &d8) {
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float ax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ax = fmaxf(ax, fabsf(v[i]));
    const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(ax)));
    int q[8];
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0;
    } else {
        const float iscale = __fdiv_rn(127.0f, amax);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = __float2int_rn(__fmul_rn(v[i], iscale));
            q[i] = max(-127, min(127, t));
        }
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo |= (static_cast<uint32_t>(q[i]) & 0xFFu) << (8 * i);
        hi |= (static_cast<uint32_t>(q[i + 4]) & 0xFFu) << (8 * i);
    }
    part = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    d8 = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, 127.0f);
    return make_uint2(lo, hi);
}

// The Q8_K planes of one block: xb its 256 floats (16-byte aligned); qb /
// bb / db its 256 quants, 16 bsums (bsum i = sum of q over 16i .. 16i+15,
// lanes 2i and 2i+1) and scale, in global or shared memory.
__device__ __forceinline__ void quantize_block_warp(const float *xb, int lane, int8_t *qb, int16_t *bb, float *db) {
    const float4 v0 = *reinterpret_cast<const float4 *>(xb + 8 * lane);
    const float4 v1 = *reinterpret_cast<const float4 *>(xb + 8 * lane + 4);
    int part;
    float d8;
    const uint2 w = q8k_lane(v0, v1, part, d8);
    *reinterpret_cast<uint2 *>(qb + 8 * lane) = w;
    part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
    if ((lane & 1) == 0) bb[lane >> 1] = static_cast<int16_t>(part);
    if (lane == 0) *db = d8;
}

// Bulk prefetch of [p, p + bytes) from HBM into L2 by the TMA engine
// (cp.async.bulk.prefetch.L2, a hint: nothing is written, nothing waits).
// p must be 16-byte aligned; the size is rounded down to 16 bytes and split
// into 32 KB requests.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint64_t bytes) {
    const uint8_t *b = static_cast<const uint8_t *>(p);
    bytes &= ~uint64_t(15);
    while (bytes) {
        const uint32_t n = bytes > 32768 ? 32768u : static_cast<uint32_t>(bytes);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b), "r"(n) : "memory");
        b += n;
        bytes -= n;
    }
}

// Asynchronous 16-byte copies global -> shared (cp.async, L2 only), in
// commit groups; cp_async_wait<N>() returns once at most N of this thread's
// groups are still in flight.  Both addresses must be 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
// the same copy, issued only where pred != 0 (predicated, no branch)
__device__ __forceinline__ void cp_async16_if(uint32_t dst_smem, const void *src, uint32_t pred) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.cg.shared.global [%0], [%1], 16;\n}\n" ::"r"(dst_smem),
        "l"(src), "r"(pred)
        : "memory");
}
// an 8-byte copy (both addresses 8-byte aligned), through L1
__device__ __forceinline__ void cp_async8(uint32_t dst_smem, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// The same with immediate byte offsets added to both addresses in the
// instruction itself (no address arithmetic in the caller).
template <int DST_OFF, int SRC_OFF>
__device__ __forceinline__ void cp_async16_if_off(uint32_t dst_smem, const void *src, uint32_t pred) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.cg.shared.global [%0+%3], [%1+%4], 16;\n}\n" ::"r"(
            dst_smem),
        "l"(src), "r"(pred), "n"(DST_OFF), "n"(SRC_OFF)
        : "memory");
}

// Shared-memory loads at 32-bit shared-window addresses (OFF: an immediate
// byte offset folded into the instruction).
template <int OFF>
__device__ __forceinline__ uint4 lds128o(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a), "n"(OFF));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t smem_addr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Programmatic dependent launch.  griddep_wait() blocks until the grids this
// one depends on have completed and their memory is visible (a no-op when
// the kernel was launched without the programmatic attribute);
// griddep_launch_dependents() lets the next kernel in the stream start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int quad_sum(int v) {
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    return v;
}

}  // namespace kq
