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
//     unpack warps expand the packed weights once as fp16 w' = sc*q with the
//     sub-scale folded in (Q4_K <= 945, Q5_K <= 1953: exact): the kq v3 panel
//     scratch, unpacked once per token block.  Q4_K/Q5_K write it into TMEM
//     (thread = weight row = TMEM lane, tcgen05.st) and the MMA reads its A
//     operand from there, so the tensor pipe's shared-memory reads are the
//     token tiles alone; Q6_K writes it into shared memory;
//     Q6_K's w' = sc*(q-32) is one exact fp16 FMA for |sc| <= 62, and when a tile holds a
//     larger sub-scale the weight is split into two exact planes,
//     sc*(v - (v&1)) (even, |.| <= 4096) and sc*(v&1), both multiplied into
//     the same accumulator;
//   - tcgen05.mma kind::f16 accumulates the page's integer sums in fp32
//     TMEM in "units" short enough that every partial sum stays an integer
//     below 2^24, where fp32 is exact: a unit is K = 128 for Q4_K
//     (128 * 945 * 127 < 2^24), K = 64 for Q5_K (64 * 1953 * 127 < 2^24);
//     for Q6_K it is chosen per tile half from the largest |sub-scale| in it:
//     K = 128 up to 32 (|w'| <= 1024), K = 64 up to 62 (|w'| <= 1984) and
//     K = 32 beyond (split planes of the same sign, |w'| <= 4096).  The
//     superblock's integer sum I (the page's isum, or iacc - 32*bacc for
//     Q6_K) is the exact sum of its units; for Q4_K/Q5_K a K=16 MMA of the
//     sub-mins (duplicated per 16) against the bsums gives msum
//     (16 * 63 * 2032 < 2^24);
//   - the epilogue folds each pair of units as d8*d*(Ua + Ub), and msum as
//     -d8*dmin*msum, in fp32 ([kq-arc], "The pieces": the float work is per
//     superblock, not per sub-block).  A debug variant of the same kernel
//     (kq_debug_gemm_partials) converts each unit to int32 instead and adds
//     them, giving I and msum bit for bit.
// The grouped (MoE) form runs one block per SM over a list of tiles (see the
// tile comment below), so short expert tiles do not pay a block's start-up
// and drain each.
//
// Warp roles (14 warps): 0 TMA producer of the activation tiles, 1 MMA issuer
// (and TMEM owner); Q4_K/Q5_K: 2..5 weight unpack (thread = weight row),
// 6..13 epilogue (thread = row x 64 token columns, y in registers); Q6_K,
// whose unpack is the longer chain: 2..9 weight unpack (two threads per row,
// one 64-wide K sub-tile each), 10..13 epilogue (thread = row x every token
// column, y accumulated in TMEM).  TMEM lane quadrant = warp % 4.  Stages
// are half superblocks (K = 128): a ring of token tiles (3 slots, Q6_K 2)
// with one full barrier per slot (every unpack warp's A rows of the half and
// the TMA tile) and one empty barrier (the commit after the half's MMAs,
// which frees both the tile and the half's A slot; A has 2 half slots, slot
// h of half i written once half i - 2 is empty).  TMEM (512 columns):
// Q4_K/Q5_K a ring of 2 unit accumulators,
// one msum (issued after the superblock's last unit and before that unit's
// commit, which covers both; folded with it) and
// the two A slots; Q6_K a ring of 3 units and y.  Every mbarrier
// wait is bounded; on timeout the block records KQ_ERR_TIMEOUT in the
// device status word and winds down.
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
    // Q4_K/Q5_K keep the unpacked weights (the A operand) in TMEM, Q6_K (two
    // planes, no room beside its y) in shared memory
    static constexpr bool kTmemA = F != FMT_Q6_K;
    // the ring of half superblocks: NB token tiles in flight; the A operand
    // has two half slots, A slot h of half i free once half i - 2 is empty
    static constexpr int NB = F == FMT_Q6_K ? 2 : 3;
    static_assert(NB >= 2 && NB <= 4, "ring of half superblocks");
    static constexpr int A_SLOT = kTmemA ? 0 : 65536;             // Q6_K: 2 sub-tiles x 2 planes
    static constexpr int B_SUB = BT * 128;                         // one 64-wide K sub-tile of tokens
    static constexpr int B_SLOT = 2 * B_SUB + (kMins ? BT * 32 : 0);
    static constexpr int AMIN_BYTES = BM * 32;                     // one superblock's sub-mins operand
    static constexpr int OFF_A = 0;
    static constexpr int OFF_AMIN = 2 * A_SLOT;                    // by superblock parity
    static constexpr int OFF_B = OFF_AMIN + (kMins ? 2 * AMIN_BYTES : 0);
    static constexpr int OFF_SD = OFF_B + NB * B_SLOT;            // s_d, s_dmin [2][BM]
    static constexpr int OFF_D8 = OFF_SD + 2 * 2 * BM * 4;        // per epilogue warp [64] floats
    static constexpr int OFF_BAR = OFF_D8 + 8 * 64 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr int OFF_TILES = OFF_MISC + 256;              // grouped: the block's tile list
    static constexpr int OFF_OFFS = OFF_TILES + TILE_CAP * 16;    // grouped: the row offsets [E + 1]
    // grouped Q4_K: each unpack thread's row bytes for a half superblock (4
    // qs pieces + the scale block, 16 B each) staged by cp.async RS - 1 halves
    // ahead, [RS][RCH chunks][BM rows] x 16 B (rows contiguous per chunk: no
    // bank conflicts)
    static constexpr int RS = F == FMT_Q4_K ? 3 : 0, RCH = 5;
    static constexpr int OFF_RAW = OFF_OFFS + (MAX_GROUPED_E + 4) * 4;
    static constexpr int OFF_RBND = OFF_RAW + RS * RCH * BM * 16;     // and its W1 bounds, [RS][BM] x 8 B
    static constexpr int SMEM = OFF_RBND + RS * BM * 8 + 1024;        // + alignment slack
    static constexpr int SMEM_DENSE = OFF_RAW + 1024;                  // the dense kernel stages no rows
    static_assert(SMEM <= 232448, "shared memory per block");
    static_assert(OFF_RAW % 16 == 0, "cp.async needs 16-byte aligned destinations");
    static_assert(OFF_B % 1024 == 0, "B tiles need 1024-byte alignment");
    static_assert(B_SLOT % 1024 == 0, "B slots need 1024-byte alignment");
};

// barrier indices: the operand ring of half superblocks (FULL: the half's
// A operand unpacked and its token tile landed; EMPTY: its MMAs complete,
// so both its A slot and its B slot may be refilled), the ring of unit
// accumulators (U), the msum accumulator (M), the per-superblock weight
// scales and unit plans (SD, by superblock parity), MMA completion, the
// tile list
enum { BAR_FULL = 0, BAR_EMPTY = 4, BAR_U_FULL = 10, BAR_U_EMPTY = 13,
       BAR_M_EMPTY = 18, BAR_SD_FULL = 20, BAR_SD_EMPTY = 22, BAR_MMA_DONE = 24, BAR_TILES = 25,
       BAR_EPI = 26, BAR_END = 27 };

// TMEM (512 columns): a ring of unit accumulators of 128 columns from column
// 0 (Q4_K/Q5_K 2 slots, Q6_K 3); Q4_K/Q5_K then msum (columns 256..383) and
// the A operand, 64 columns per half superblock (384..511); Q6_K y (384..511).
template <int F> constexpr int n_units() { return F == FMT_Q6_K ? 3 : 2; }
constexpr uint32_t COL_M = 256, COL_Y = 384, COL_A = 384;

// ---------------------------------------------------------------------------
// Accumulator units.  The fp32 TMEM accumulator is exact while every partial
// sum is an integer of magnitude <= 2^24.  With |a8| <= 128 a partial sum
// of w' * a8 over a set of weights is at most 128 * sum |w'| over them, so:
//   - a half superblock (K = 128) is always one unit for Q4_K
//     (128 * 945 * 128 < 2^24); for Q5_K when its rows' W1 (sum |w'|, from
//     the image's bounds plane) is <= 2^24 / 128, else two units of K = 64
//     (64 * 1953 * 128 < 2^24); for Q6_K when W1 allows it or every
//     |sub-scale| <= 32 (128 * 32 * 32 * 128 = 2^24), else two units of
//     K = 64 while every |sub-scale| <= 62, else four of K = 32 (split
//     planes of the same sign, 32 * 4096 * 128 = 2^24);
//   - a whole superblock is one unit when both halves are single units and
//     the rows' W1 over the superblock is <= 2^24 / 128 (the common case).
// Each unpack warp publishes, per half, a flag byte for its rows: bits 0..1
// the half's category (units 1, 2, 4), bit 2 (second half only) the whole-
// superblock bound, bit 3 (Q6_K) split planes.  The MMA issuer and the
// epilogue derive the same plan from these flags.
constexpr uint32_t W1_LIMIT = 1u << 17;  // 2^24 / 128
__host__ __device__ constexpr int units_of_cat(int cat) { return cat == 0 ? 1 : (cat == 1 ? 2 : 4); }

struct SbPlan {
    int cat[2];     // per half: 0, 1, 2
    bool split[2];  // Q6_K: two A planes in the half
    bool whole;     // one unit for the superblock
    int n;          // units of the superblock
};
// A half's flags: one byte per unpack warp (8 bytes; the bytes of absent
// warps hold FLAG_NEUTRAL), read as one 64-bit shared-memory load.
constexpr uint8_t FLAG_NEUTRAL = 4;
constexpr uint64_t BYTES_1 = 0x0101010101010101ull;
__device__ __forceinline__ uint64_t ld_flags(uint32_t saddr) {
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(saddr) : "memory");
    return v;
}
__device__ __forceinline__ int half_cat(uint64_t f) {
    return (f & (2 * BYTES_1)) ? 2 : ((f & BYTES_1) ? 1 : 0);
}
__device__ __forceinline__ bool half_split(uint64_t f) { return (f & (8 * BYTES_1)) != 0; }
// The plan of a superblock from its two halves' flags.
__device__ __forceinline__ SbPlan sb_plan(uint64_t f0, uint64_t f1) {
    SbPlan pl;
    pl.cat[0] = half_cat(f0);
    pl.cat[1] = half_cat(f1);
    pl.split[0] = half_split(f0);
    pl.split[1] = half_split(f1);
    pl.whole = pl.cat[0] == 0 && pl.cat[1] == 0 && (f1 & (4 * BYTES_1)) == 4 * BYTES_1;
    pl.n = pl.whole ? 1 : units_of_cat(pl.cat[0]) + units_of_cat(pl.cat[1]);
    return pl;
}
// An unpack warp's flag for half h: w1 = its rows' W1 bound of the half,
// w1sb of the superblock (h = 1), maxsc the largest |sub-scale| (Q6_K).
template <int F>
__device__ __forceinline__ int unit_flag(int h, uint32_t w1, uint32_t w1sb, int maxsc) {
    int cat = 0;
    if constexpr (F == FMT_Q5_K) cat = w1 <= W1_LIMIT ? 0 : 1;
    if constexpr (F == FMT_Q6_K) cat = (w1 <= W1_LIMIT || maxsc <= 32) ? 0 : (maxsc <= 62 ? 1 : 2);
    int f = cat;
    if (h == 1 && w1sb <= W1_LIMIT) f |= 4;
    if (F == FMT_Q6_K && maxsc > 62) f |= 8;
    return f;
}

struct GemmParams {
    const uint8_t *packed;
    uint64_t expert_bytes;
    int64_t N, K, nsb, M;
    const int32_t *offsets;  // grouped: [E+1]; dense: nullptr
    int64_t E;
    const float *d8t;        // workspace: d8 transposed [nsb][Mp]
    int64_t Mp;
    float *y;
    // debug: instead of y, the superblock integer sums, [M][N][nsb] each
    // (isum_out zero-filled before the launch; it is accumulated per unit pair)
    int32_t *isum_out, *msum_out;
    // dense: block b runs the steps [b * units / grid, (b + 1) * units / grid)
    // of the tiles x superblocks grid, in pieces of one tile each; a tile cut
    // between blocks is finished from their fp32 partial tiles (part: two
    // slots per block, [BT][BM] each) by the last of them to count itself in
    // tile_cnt (zeroed by the pre-pass)
    int64_t units;
    float *part;
    int *tile_cnt;
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
// the A operand.

// Q4_K/Q5_K, into TMEM: the row is the thread's lane, `a_tm` the TMEM address
// of the sub-tile (32 columns, two fp16 per column, the lower K in the low
// half).  Sub-tile = chunk c of the superblock (64 elements): elements
// 64c + l (low nibbles of qs[32c + l], sub-scale sc_2c) at K 0..31 and
// 64c + 32 + l (high nibbles, sc_2c+1) at K 32..63; Q5_K ORs bit 2c / 2c+1 of
// qh[l] in as value 16.  w' = q*sc is built exactly in fp16 as
// (1024 + q)*sc - 1024*sc (low) and (1024 + 16q)*(sc/16) - 64*sc (high).
template <int F>
__device__ __forceinline__ void unpack_q45(uint32_t a_tm, const uint32_t (&qs)[8], const uint32_t (&qh)[8], int c,
                                           int sc_lo, int sc_hi) {
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
                    // qh bytes 2pr, 2pr+1 in bytes 0 and 2 (bytes 1 and 3 from the zero operand)
                    const uint32_t hb = prmt(qh[2 * q + w], 0u, pr ? 0x4342u : 0x4140u);
                    const int b = 2 * c;  // low nibble's fifth bit
                    // bit b of each byte to bit 4 of its 16-bit lane: a rotation by
                    // 4 - b (the bits it wraps around fall outside the mask)
                    l |= __funnelshift_r(hb, hb, (uint32_t)(b - 4) & 31u) & 0x00100010u;
                    // high nibble's fifth bit (2c+1) lands on bit 8: value 256 = 16 * 16
                    h |= (hb << (7 - b)) & 0x01000100u;
                }
                lo[2 * w + pr] = h2_fma(l, s_lo, o_lo);
                hi[2 * w + pr] = h2_fma(h, s_hi, o_hi);
            }
        }
        tmem_st4(a_tm + 4 * q, lo[0], lo[1], lo[2], lo[3]);        // K 8q .. 8q+7
        tmem_st4(a_tm + 16 + 4 * q, hi[0], hi[1], hi[2], hi[3]);   // K 32 + 8q ..
    }
}

// Q6_K, into shared memory (128-byte swizzled K-major fp16 rows; `a_tile` is
// the sub-tile base, the row's 8 chunks of 8 fp16 at sw128_offset(r, 8q)):
// sub-tile j of half h holds groups t = 2j (K 0..31) and 2j+1 (K 32..63)
// of the half: element 128h + 32t + l is the low (t < 2) or high (t >= 2)
// nibble of ql[64h + 32(t&1) + l] with bits 2t..2t+1 of qh[32h + l] on top,
// sub-scale sc[8h + 2t + l/16] (byte 2(t - 2j) + l/16 of `scw`).  The 6-bit
// q of four elements is assembled in one word, then spread into fp16 lanes
// 1024 + q.  v = q - 32: P1 = v*sc = (1024 + q)*sc - 1056*sc in one fp16 FMA,
// exact for |sc| <= 62 (1056*sc and the result are exact fp16 integers); with
// `split` (some |sc| > 62), sc = sa + sb with sa = floor(sc / 2), sb = sc - sa
// (same sign, |sa|, |sb| <= 64): P1 = v*sa and P2 = v*sb, each an exact fp16
// integer (|.| <= 2048), of the same sign, summing to v*sc.  `zero2` writes
// zeros to this thread's P2 rows instead.
__device__ __forceinline__ void unpack_q6(uint32_t a_tile, uint32_t a2_tile, int r, const uint32_t (&ql)[16],
                                          const uint32_t (&qh)[8], uint32_t scw, int j, bool split, bool zero2) {
    const uint32_t off1056 = h2_splat(1056.0f);
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        const int t = 2 * j + tt;
        // the group's two sub-scales (l < 16, l >= 16): sc, -1056 * sc, and the halves sa, sb
        uint32_t s2v[2], c2v[2], sav[2], sbv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int scv = (int)(int8_t)((scw >> (8 * (2 * tt + u))) & 0xFF);
            const int sa = scv >> 1;
            s2v[u] = h2_splat((float)scv);
            c2v[u] = h2_splat(-1056.0f * (float)scv);
            sav[u] = h2_splat((float)sa);
            sbv[u] = h2_splat((float)(scv - sa));
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
                        const uint32_t v = h2_sub(x, off1056);                 // q - 32, exact
                        p1[2 * w + pr] = h2_mul(v, sav[q >> 1]);
                        p2[2 * w + pr] = h2_mul(v, sbv[q >> 1]);
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
// bnd: the row group's W1 bounds of the superblock's two halves.
struct RawQ4 { uint32_t qs[16]; uint4 hdr; uint2 bnd; };              // qs[64h .. 64h+64)
struct RawQ5 { uint32_t qs[16]; uint32_t qh[8]; uint4 hdr; uint2 bnd; };
struct RawQ6 { uint32_t ql[16]; uint32_t qh[8]; uint32_t sc[2]; uint32_t d; uint2 bnd; };  // ql/qh/sc of half h
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
    r.bnd = __ldg(reinterpret_cast<const uint2 *>(P.p4) + ch);
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
    r.bnd = __ldg(reinterpret_cast<const uint2 *>(P.p4) + ch);
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
    r.bnd = __ldg(reinterpret_cast<const uint2 *>(P.p4) + ch);
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

// Dense tile i: the token tiles of a weight row tile are adjacent, so
// consecutive tiles share that weight panel in L2.  The index arithmetic is
// 32-bit for Q4_K/Q5_K (the launcher takes at most INT32_MAX tiles) and
// 64-bit for Q6_K: measured per format on GB300 (27B Q4_K FFN 574 -> 587
// TOPS with 32 bits; the 4B Q6_K block-per-tile shapes 3-4 % slower).
template <int F>
__device__ __forceinline__ Tile tile_at(const GemmParams &p, int64_t i) {
    Tile t;
    t.e = 0;
    if constexpr (F == FMT_Q6_K) {
        const int t_tiles = (int)((p.M + BT - 1) / BT);
        t.n0 = (int)(i / t_tiles) * BM;
        t.t0 = (int)(i % t_tiles) * BT;
    } else {
        const uint32_t t_tiles = (uint32_t)((p.M + BT - 1) / BT), ii = (uint32_t)i;
        t.n0 = (int)(ii / t_tiles) * BM;
        t.t0 = (int)(ii % t_tiles) * BT;
    }
    t.t_end = (t.t0 + BT < p.M) ? t.t0 + BT : (int)p.M;
    finish_tile(t);
    return t;
}

// A block's work item: tile t, superblocks [sb0, sb1) of it (dense: one
// piece of the block's share of the steps; grouped: a whole list tile).
struct Piece {
    Tile t;
    int64_t tile;  // dense: the tile's index
    int sb0, sb1;
};
// first step of block b's share (dense)
__device__ __forceinline__ int64_t dense_step_of(int64_t b, int64_t units) { return b * units / (int64_t)gridDim.x; }
__device__ __forceinline__ int64_t dense_step(const GemmParams &p, int64_t b) { return dense_step_of(b, p.units); }
// The block's share as pieces, worked out once by one thread at the start
// (the 64-bit divisions stay out of every role's loop): plan[0] the first
// tile, [1] the last, [2] the first piece's first superblock, [3] the last
// piece's end, [4] the number of pieces.
constexpr int MISC_PLAN = 4;
__device__ __forceinline__ void dense_plan(const GemmParams &p, uint32_t *plan) {
    const int64_t u0 = dense_step(p, blockIdx.x), u1 = dense_step(p, blockIdx.x + 1);
    const int64_t i0 = u0 / p.nsb, i1 = u1 > u0 ? (u1 - 1) / p.nsb : i0;
    plan[0] = (uint32_t)i0;
    plan[1] = (uint32_t)i1;
    plan[2] = (uint32_t)(u0 - i0 * p.nsb);
    plan[3] = (uint32_t)(u1 - i1 * p.nsb);
    plan[4] = u0 < u1 ? (uint32_t)(i1 - i0 + 1) : 0u;
}
__device__ __forceinline__ int dense_pieces(const uint32_t *plan) { return (int)plan[4]; }
template <int F>
__device__ __forceinline__ Piece dense_piece(const GemmParams &p, const uint32_t *plan, int k) {
    const uint32_t i = plan[0] + (uint32_t)k;
    Piece q;
    q.t = tile_at<F>(p, i);
    q.tile = i;
    q.sb0 = k == 0 ? (int)plan[2] : 0;
    q.sb1 = i == plan[1] ? (int)plan[3] : (int)p.nsb;
    return q;
}
// the block whose share holds step x (dense)
__device__ __forceinline__ int64_t dense_block_of(int64_t x, int64_t units) {
    const int64_t B = gridDim.x;
    int64_t b = x * B / units;
    while (b + 1 < B && dense_step_of(b + 1, units) <= x) ++b;
    while (b > 0 && dense_step_of(b, units) > x) --b;
    return b;
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

// work item k of the block: grouped, list tile k; dense with the split-tile
// schedule (SK), piece k of the block's share; dense without it, the block's
// tile, whole
template <int F, bool G, bool SK>
__device__ __forceinline__ Piece work_piece(const GemmParams &p, const int4 *list, const uint32_t *plan, int k) {
    if constexpr (!G && SK) {
        return dense_piece<F>(p, plan, k);
    } else {
        Piece q;
        q.t = G ? list_tile(list, k) : tile_at<F>(p, blockIdx.x);
        q.tile = G ? -1 : (int64_t)blockIdx.x;
        q.sb0 = 0;
        q.sb1 = (int)p.nsb;
        return q;
    }
}
// dense: the block's work items
template <bool SK>
__device__ __forceinline__ int dense_items(const uint32_t *plan) {
    if constexpr (SK) return dense_pieces(plan);
    else return 1;
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

// ---------------------------------------------------------------------------
// Epilogue helpers.  TMEM addresses are of this warp's lane quadrant; a
// thread holds one weight row.

// Q4_K/Q5_K: y[64] (64 token columns, in registers) += d8 * (d * U - dmin *
// msum) for one unit U, CW (8 or 16) columns per TMEM load round trip, over
// the first nch such chunks (the tile's token columns; the rest are padding)
template <int CW, bool WM>
__device__ __forceinline__ void fold_unit_q45(float (&y)[64], uint32_t xu, uint32_t xm, float dd, float dm,
                                              const float *s_d8, int nch) {
#pragma unroll
    for (int cc = 0; cc < 64 / CW; ++cc) {
        if (cc >= nch) break;
        uint32_t vu[CW], vm[CW];
        if constexpr (CW == 16) {
            tmem_ld16(xu + 16 * cc, vu);
            if constexpr (WM) tmem_ld16(xm + 16 * cc, vm);
        } else {
            tmem_ld8(xu + 8 * cc, vu);
            if constexpr (WM) tmem_ld8(xm + 8 * cc, vm);
        }
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            const float tv = WM ? fmaf(-dm, __uint_as_float(vm[i]), dd * __uint_as_float(vu[i]))
                                : dd * __uint_as_float(vu[i]);
            y[CW * cc + i] = fmaf(s_d8[CW * cc + i], tv, y[CW * cc + i]);
        }
    }
}

// Q6_K: y (in TMEM at yt) += d8 * d * (Ua [+ Ub]) over nc chunks of 16
// columns; FIRST: y starts from zero
template <bool PAIR, bool FIRST>
__device__ __forceinline__ void fold_units_q6(uint32_t xa, uint32_t xb, uint32_t yt, int nc, float dd,
                                              const float *s_d8) {
    for (int c = 0; c < nc; ++c) {
        uint32_t va[16], vb[PAIR ? 16 : 1], vy[16];
        tmem_ld16(xa + 16 * c, va);
        if constexpr (PAIR) tmem_ld16(xb + 16 * c, vb);
        if constexpr (!FIRST) tmem_ld16(yt + 16 * c, vy);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float sum = __uint_as_float(va[i]);
            if constexpr (PAIR) sum += __uint_as_float(vb[i]);
            const float yo = FIRST ? 0.0f : __uint_as_float(vy[i]);
            vy[i] = __float_as_uint(fmaf(s_d8[16 * c + i] * dd, sum, yo));
        }
        tmem_st16(yt + 16 * c, vy);
    }
}

// Debug epilogue (kq_debug_gemm_partials): the units' exact integers added
// into isum, msum stored, for `ncols` token columns from tok0 (16 at a
// time); has_b: a second unit at xb, has_m: msum at xm.
__device__ __forceinline__ void debug_units(int32_t *isum_out, int32_t *msum_out, int64_t N, int64_t nsb, uint32_t xa,
                                            bool has_b, uint32_t xb, bool has_m, uint32_t xm, int ncols, int64_t tok0,
                                            int64_t t_end, int64_t n, int64_t sb) {
    for (int c = 0; c < ncols; c += 16) {
        uint32_t va[16], vb[16], vm[16];
        tmem_ld16(xa + c, va);
        if (has_b) tmem_ld16(xb + c, vb);
        if (has_m) tmem_ld16(xm + c, vm);
        tmem_wait_ld();
        if (n >= N) continue;
        for (int i = 0; i < 16; ++i) {
            const int64_t tt = tok0 + c + i;
            if (tt >= t_end) break;
            int iv = __float2int_rn(__uint_as_float(va[i]));
            if (has_b) iv += __float2int_rn(__uint_as_float(vb[i]));
            const int64_t o = (tt * N + n) * nsb + sb;
            atomicAdd(isum_out + o, iv);
            if (has_m) msum_out[o] = __float2int_rn(__uint_as_float(vm[i]));
        }
    }
}

// MMA issue of the K16 steps [S0, S1) of one half (A slot a_slot, B slot
// b_slot) into accumulator acc; `fresh`: the first step overwrites it.
// Straight-line: one tcgen05.mma per step and plane.  The two base
// descriptors are pinned in registers (the empty asm keeps the compiler from
// re-deriving them per step) and each step adds its compile-time offset to the
// 14-bit address field, which cannot carry: shared memory ends below 256 KB.
// A build that derived every step's descriptor from the slot address instead
// fed one step the operand address of the step before it (one K16 slice of
// the second half counted twice and the next one dropped, the same in every
// superblock), which the bit-exact partials tests caught.
template <int B_SUB, int S0, int S1, int PLANES>
__device__ __forceinline__ void issue_steps(uint32_t acc, uint32_t a_slot, uint32_t b_slot, bool fresh,
                                            uint32_t idesc) {
    uint64_t a0 = smem_desc(a_slot, 16, 1024, SWZ_128B), b0 = smem_desc(b_slot, 16, 1024, SWZ_128B);
    asm volatile("mov.b64 %0, %0;" : "+l"(a0));
    asm volatile("mov.b64 %0, %0;" : "+l"(b0));
#pragma unroll
    for (int st = S0; st < S1; ++st) {
        const int j = st >> 2, kk = st & 3;
        const uint64_t bd = b0 + (uint64_t)((j * B_SUB + 32 * kk) >> 4);
#pragma unroll
        for (int pl = 0; pl < PLANES; ++pl) {
            const uint64_t ad = a0 + (uint64_t)((pl * 32768 + j * 16384 + 32 * kk) >> 4);
            umma_f16(acc, ad, bd, idesc, (fresh && st == S0 && pl == 0) ? 0u : 1u);
        }
    }
}

// The same with A in TMEM (Q4_K/Q5_K): step st reads the 8 columns a_tm + 8st.
template <int B_SUB, int S0, int S1>
__device__ __forceinline__ void issue_steps_ts(uint32_t acc, uint32_t a_tm, uint32_t b_slot, bool fresh,
                                               uint32_t idesc) {
    uint64_t b0 = smem_desc(b_slot, 16, 1024, SWZ_128B);
    asm volatile("mov.b64 %0, %0;" : "+l"(b0));
    asm volatile("mov.b32 %0, %0;" : "+r"(a_tm));
#pragma unroll
    for (int st = S0; st < S1; ++st) {
        const int j = st >> 2, kk = st & 3;
        const uint64_t bd = b0 + (uint64_t)((j * B_SUB + 32 * kk) >> 4);
        umma_f16_ts(acc, a_tm + 8u * st, bd, idesc, (fresh && st == S0) ? 0u : 1u);
    }
}

// unit v of the U (1, 2 or 4) units a half is cut into: steps [8v/U, 8(v+1)/U)
template <int B_SUB, int PLANES>
__device__ __forceinline__ void issue_unit(int U, int v, uint32_t acc, uint32_t a_slot, uint32_t b_slot, bool fresh,
                                           uint32_t idesc) {
    if (U == 1) {
        issue_steps<B_SUB, 0, 8, PLANES>(acc, a_slot, b_slot, fresh, idesc);
    } else if (U == 2) {
        if (v == 0) issue_steps<B_SUB, 0, 4, PLANES>(acc, a_slot, b_slot, fresh, idesc);
        else issue_steps<B_SUB, 4, 8, PLANES>(acc, a_slot, b_slot, fresh, idesc);
    } else {
        switch (v) {
        case 0: issue_steps<B_SUB, 0, 2, PLANES>(acc, a_slot, b_slot, fresh, idesc); break;
        case 1: issue_steps<B_SUB, 2, 4, PLANES>(acc, a_slot, b_slot, fresh, idesc); break;
        case 2: issue_steps<B_SUB, 4, 6, PLANES>(acc, a_slot, b_slot, fresh, idesc); break;
        default: issue_steps<B_SUB, 6, 8, PLANES>(acc, a_slot, b_slot, fresh, idesc); break;
        }
    }
}
template <int B_SUB>
__device__ __forceinline__ void issue_unit_ts(int U, int v, uint32_t acc, uint32_t a_tm, uint32_t b_slot, bool fresh,
                                              uint32_t idesc) {
    if (U == 1) {
        issue_steps_ts<B_SUB, 0, 8>(acc, a_tm, b_slot, fresh, idesc);
    } else if (U == 2) {
        if (v == 0) issue_steps_ts<B_SUB, 0, 4>(acc, a_tm, b_slot, fresh, idesc);
        else issue_steps_ts<B_SUB, 4, 8>(acc, a_tm, b_slot, fresh, idesc);
    } else {
        switch (v) {
        case 0: issue_steps_ts<B_SUB, 0, 2>(acc, a_tm, b_slot, fresh, idesc); break;
        case 1: issue_steps_ts<B_SUB, 2, 4>(acc, a_tm, b_slot, fresh, idesc); break;
        case 2: issue_steps_ts<B_SUB, 4, 6>(acc, a_tm, b_slot, fresh, idesc); break;
        default: issue_steps_ts<B_SUB, 6, 8>(acc, a_tm, b_slot, fresh, idesc); break;
        }
    }
}

// Dense split tiles: this block's partial tile for its k-th piece (slot 0
// for its first piece, 1 for its last: the pieces between are whole tiles).
__device__ __forceinline__ float *own_slot(const GemmParams &p, int k) {
    return p.part + (size_t)(2 * blockIdx.x + (k == 0 ? 0 : 1)) * (BT * BM);
}

// After every epilogue thread has written its part of this block's partial
// tile for tile `tile`: the block counts itself in, and the last of the
// tile's blocks adds their partial tiles in block order (a fixed sum, so
// the result does not depend on timing) and writes this thread's row n of
// y, token columns [t0 + cbeg, t0 + cbeg + ncol) below t_end (`act`: the
// thread has such a row and columns).  The epilogue warps meet twice on the
// BAR_EPI mbarrier (bounded waits; its phase counted in *phase).  Out of
// line: it runs once per split tile, and inline its registers would crowd
// the epilogue's loop.  False on a timeout.
__device__ __noinline__ bool split_finish(float *part, int *tile_cnt, int64_t units, int64_t nsb, int64_t tile,
                                          float *y, int64_t N, int64_t n, int t0, int t_end, int cbeg, int ncol,
                                          bool act, bool leader, int lane, uint32_t *phase, uint64_t *bar,
                                          uint32_t *misc) {
    __threadfence();  // the partial sums are visible before the count
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[BAR_EPI]);
    bool w = mbar_wait(&bar[BAR_EPI], *phase & 1u);
    ++*phase;
    if (!__all_sync(0xFFFFFFFFu, w)) return false;
    const int64_t b_lo = dense_block_of(tile * nsb, units), b_hi = dense_block_of((tile + 1) * nsb - 1, units);
    if (leader) {
        const int before = atomicAdd(&tile_cnt[tile], 1);
        const bool is_last = before == (int)(b_hi - b_lo);
        if (is_last) tile_cnt[tile] = 0;  // every block of the tile has counted
        misc[2] = is_last ? 1u : 0u;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[BAR_EPI]);
    w = mbar_wait(&bar[BAR_EPI], *phase & 1u);
    ++*phase;
    if (!__all_sync(0xFFFFFFFFu, w)) return false;
    if (*reinterpret_cast<volatile uint32_t *>(&misc[2]) == 0u || !act) return true;
    __threadfence();  // the other blocks' partial sums are read after their counts
    for (int c = 0; c < ncol; c += 16) {
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int64_t b = b_lo; b <= b_hi; ++b) {
            // block b's slot for this tile: its first piece's when that piece is this tile
            const int which = dense_step_of(b, units) / nsb == tile ? 0 : 1;
            const float *src = part + (size_t)(2 * b + which) * (BT * BM) + (size_t)(cbeg + c) * BM + (n % BM);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] += __ldcg(src + i * BM);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t tt = (int64_t)t0 + cbeg + c + i;
            if (tt < t_end) y[tt * N + n] = acc[i];
        }
    }
    return true;
}

template <int F, bool G, bool DBG, bool SK>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a16, const __grid_constant__ CUtensorMap map_b16,
                const GemmParams p) {
    using C = Cfg<F>;
    constexpr int NU = n_units<F>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    float *s_d = reinterpret_cast<float *>(smem + C::OFF_SD);
    float *s_dmin = s_d + 2 * BM;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);  // [0] tmem base, [1] tile count
    // each unpack warp's unit flag byte, [superblock parity][half][8 warps]
    uint8_t *s_flag = reinterpret_cast<uint8_t *>(misc + 16);
    const uint32_t flag_sa = smem_u32(s_flag);  // the same, as a shared-memory address
    const uint32_t *s_plan = misc + MISC_PLAN;    // dense split-tile: the block's pieces
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
        // a half is full once every unpack warp has written its A rows and
        // the TMA thread's token tile has landed (its arrive carries the
        // byte count); empty once the MMAs that read it are complete
        for (int i = 0; i < C::NB; ++i) {
            mbar_init(&bar[BAR_FULL + i], n_unpack<F>() + 1);
            mbar_init(&bar[BAR_EMPTY + i], 1);
        }
        for (int i = 0; i < NU; ++i) {
            mbar_init(&bar[BAR_U_FULL + i], 1);
            mbar_init(&bar[BAR_U_EMPTY + i], n_epi<F>());
        }
        mbar_init(&bar[BAR_M_EMPTY], n_epi<F>());
        // every unpack warp arrives once the scales and both halves' unit
        // flags of the superblock are written
        mbar_init(&bar[BAR_SD_FULL + 0], n_unpack<F>());
        mbar_init(&bar[BAR_SD_FULL + 1], n_unpack<F>());
        mbar_init(&bar[BAR_SD_EMPTY + 0], n_epi<F>());
        mbar_init(&bar[BAR_SD_EMPTY + 1], n_epi<F>());
        mbar_init(&bar[BAR_MMA_DONE], 1);
        mbar_init(&bar[BAR_TILES], 1);
        mbar_init(&bar[BAR_EPI], n_epi<F>());  // the epilogue warps' split-tile handshake
        mbar_init(&bar[BAR_END], NTHREADS / 32);  // every warp is done with TMEM
        if constexpr (!G && SK) dense_plan(p, misc + MISC_PLAN);
        mbar_fence_init();
        for (int i = 0; i < 32; ++i) s_flag[i] = FLAG_NEUTRAL;
    }
    if (warp == W_MMA) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // TMEM columns: unit accumulator i at 128i (i < NU), msum at COL_M, A at COL_A (Q4_K/Q5_K), y at COL_Y (Q6_K).
    // The unit ring's slots and phases follow u, the block's count of units
    // over all tiles; the msum slot's phase the count of non-empty superblocks; the
    // SD barriers' the block's count g of superblock steps over all tiles.
    bool ok = true;

    if (warp == W_TMA) {
        // ------------------------------------------------ activation tiles
        griddep_wait();
        int ntiles = G ? 0 : dense_items<SK>(s_plan);
        if constexpr (G) {
            ntiles = build_tile_list(p, reinterpret_cast<int *>(smem + C::OFF_OFFS), s_list, lane);
            __threadfence_block();
            __syncwarp();
            if (lane == 0) {
                misc[1] = (uint32_t)ntiles;
                mbar_arrive(&bar[BAR_TILES]);
            }
        }
        // ring position of the half: slot and the parity of its round
        uint32_t slot = 0, round = 0, issued = 0;
        if (lane == 0) {
            tma_prefetch_desc(&map_a16);
            if (C::kMins) tma_prefetch_desc(&map_b16);
            if (ntiles > 0) prefetch_tile<F>(p, work_piece<F, G, SK>(p, s_list, s_plan, 0).t);
            for (int k = 0; k < ntiles && ok; ++k) {
                const Piece q = work_piece<F, G, SK>(p, s_list, s_plan, k);
                const Tile t = q.t;
                // the next tile's weights stream into L2 while this one runs
                if (k + 1 < ntiles) prefetch_tile<F>(p, work_piece<F, G, SK>(p, s_list, s_plan, k + 1).t);
                for (int64_t sb = q.sb0; sb < q.sb1 && ok; ++sb) {
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (!mbar_wait(&bar[BAR_EMPTY + slot], (round & 1u) ^ 1u)) { ok = false; break; }
                        if (t.ntok > 0) {
                            uint8_t *bs = smem + C::OFF_B + slot * C::B_SLOT;
                            // the token bsums (msum's operand) come with the second half,
                            // after whose units msum is issued
                            const bool mins = C::kMins && h == 1;
                            mbar_arrive_expect_tx(&bar[BAR_FULL + slot], 2 * C::B_SUB + (mins ? BT * 32 : 0));
                            const int k0 = (int)(sb * QK + 128 * h);
                            tma_load_2d(bs, &map_a16, k0, t.t0, &bar[BAR_FULL + slot]);
                            tma_load_2d(bs + C::B_SUB, &map_a16, k0 + 64, t.t0, &bar[BAR_FULL + slot]);
                            if (mins) tma_load_2d(bs + 2 * C::B_SUB, &map_b16, (int)(sb * 16), t.t0, &bar[BAR_FULL + slot]);
                            ++issued;
                        } else {
                            mbar_arrive(&bar[BAR_FULL + slot]);  // a tile without rows: nothing to load
                        }
                        if (++slot == C::NB) {
                            slot = 0;
                            ++round;
                        }
                    }
                }
            }
            if (!ok) {
                set_timeout();
                // let the copies already issued land before the block exits:
                // the MMA thread, also winding down, has stopped consuming,
                // so wait (bounded) for the last slots' phases
                for (int s = 0; s < C::NB && (uint32_t)s < issued; ++s) {
                    slot = slot == 0 ? C::NB - 1 : slot - 1;
                    if (slot == C::NB - 1) --round;
                    mbar_wait(&bar[BAR_FULL + slot], round & 1u, 20000000ull);
                }
            }
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------ MMA issue
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        const uint32_t amin = smem_u32(smem + C::OFF_AMIN);
        const uint32_t b_base = smem_u32(smem + C::OFF_B);
        // g: the block's superblock steps; slot/round: the ring position of the
        // half; u: units issued; mc: msum issues (32 bits: a block runs at
        // most TILE_CAP tiles of at most 2^22 superblocks)
        uint32_t g = 0, slot = 0, round = 0, u = 0, mc = 0;
        if (lane == 0) {
            int ntiles = G ? 0 : dense_items<SK>(s_plan);
            if constexpr (G) {
                ok = mbar_wait(&bar[BAR_TILES], 0);
                ntiles = ok ? (int)misc[1] : 0;
            }
            // unit v of U of half h (A: TMEM columns a_tm, or shared-memory slot
            // a_slot; B: slot b_slot) into accumulator acc (Q6_K split halves:
            // both planes per step)
            auto issue = [&](int U, int v, uint32_t acc, uint32_t a_slot, uint32_t a_tm, uint32_t b_slot, int planes,
                             bool fresh, uint32_t idesc) {
                if constexpr (C::kTmemA) issue_unit_ts<C::B_SUB>(U, v, acc, a_tm, b_slot, fresh, idesc);
                else if (planes == 2) issue_unit<C::B_SUB, 2>(U, v, acc, a_slot, b_slot, fresh, idesc);
                else issue_unit<C::B_SUB, 1>(U, v, acc, a_slot, b_slot, fresh, idesc);
            };
            for (int k = 0; k < ntiles && ok; ++k) {
                const Piece q = work_piece<F, G, SK>(p, s_list, s_plan, k);
                const Tile t = q.t;
                const uint32_t idesc = idesc_f16_f32(BM, t.n_mma > 0 ? t.n_mma : 16);
                for (int64_t sb = q.sb0; sb < q.sb1 && ok; ++sb, ++g) {
                    bool open = false;  // a unit begun in the first half, still accumulating
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t cur = slot, cur_par = round & 1u;
                        if (++slot == C::NB) {
                            slot = 0;
                            ++round;
                        }
                        // the half's A operand and token tile
                        if (!mbar_wait(&bar[BAR_FULL + cur], cur_par)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (t.ntok == 0) {  // a first tile without rows: release the half unread
                            mbar_arrive(&bar[BAR_EMPTY + cur]);
                            continue;
                        }
                        const uint32_t a_slot = a_base + h * C::A_SLOT;
                        const uint32_t a_tm = tmem + COL_A + 64 * (uint32_t)h;
                        const uint32_t b_slot = b_base + cur * C::B_SLOT;
                        // this half's flags are in (each unpack warp writes its byte before
                        // it arrives on the half's FULL)
                        const uint32_t fl = flag_sa + 16 * (uint32_t)(g & 1);
                        SbPlan pl;
                        if (h == 0) {
                            const uint64_t f0 = ld_flags(fl);
                            pl.cat[0] = half_cat(f0);
                            pl.split[0] = half_split(f0);
                            pl.whole = false;
                        } else {
                            pl = sb_plan(ld_flags(fl), ld_flags(fl + 8));
                        }
                        const int planes = (F == FMT_Q6_K && pl.split[h]) ? 2 : 1;
                        // msum, after the superblock's last unit and before that unit's
                        // commit (which then covers both; the epilogue folds msum with
                        // that unit): the sub-mins of the superblock's parity against the
                        // token bsums of this slot, into its one slot
                        auto issue_msum = [&]() -> bool {
                            if (!mbar_wait(&bar[BAR_M_EMPTY], (uint32_t)((mc & 1) ^ 1))) return false;
                            tc_fence_after();
                            const uint64_t ad = smem_desc(amin + (uint32_t)((g & 1) * C::AMIN_BYTES), 16, 256, SWZ_32B);
                            const uint64_t bd = smem_desc(b_slot + 2 * C::B_SUB, 16, 256, SWZ_32B);
                            umma_f16(tmem + COL_M, ad, bd, idesc, 0);
                            ++mc;
                            return true;
                        };
                        if (h == 1 && open && pl.whole) {
                            // the superblock is one unit: the second half goes on into it
                            issue(1, 0, tmem + 128 * (uint32_t)(u % NU), a_slot, a_tm, b_slot, planes, false, idesc);
                            if (C::kMins && !issue_msum()) {
                                ok = false;
                                break;
                            }
                            umma_commit(&bar[BAR_U_FULL + (int)(u % NU)]);
                            ++u;
                            open = false;
                        } else {
                            if (open) {  // the first half's unit ends there
                                umma_commit(&bar[BAR_U_FULL + (int)(u % NU)]);
                                ++u;
                                open = false;
                            }
                            const int U = units_of_cat(pl.cat[h]);
                            for (int v = 0; v < U && ok; ++v) {
                                const int us = (int)(u % NU);
                                if (!mbar_wait(&bar[BAR_U_EMPTY + us], (uint32_t)(((u / NU) & 1) ^ 1))) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                issue(U, v, tmem + 128 * (uint32_t)us, a_slot, a_tm, b_slot, planes, true, idesc);
                                if (h == 0 && U == 1) {
                                    open = true;  // committed with the second half, or before it
                                } else {
                                    if (C::kMins && h == 1 && v == U - 1 && !issue_msum()) {
                                        ok = false;
                                        break;
                                    }
                                    umma_commit(&bar[BAR_U_FULL + us]);
                                    ++u;
                                }
                            }
                        }
                        if (!ok) break;
                        umma_commit(&bar[BAR_EMPTY + cur]);  // frees the half's A and B slots
                    }
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
        // tile row: Q4_K/Q5_K write it into TMEM lane r, in the warp's quadrant
        const int r = C::kTmemA ? 32 * (warp & 3) + lane : 32 * (uw & 3) + lane;
        const int my_jj = uw >> 2;               // Q6_K: this thread's K sub-tile of each half
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        const uint32_t a_tm0 = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + COL_A;  // Q4_K/Q5_K A, half 0
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
        const uint8_t *cq = nullptr, *chd = nullptr, *cbd = nullptr;
        const uint32_t rbnd = smem_u32(smem + C::OFF_RBND);  // the W1 bounds ring, [RS][BM] x 8 B
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
            cbd = P.p4 + ch0 * BOUND_BYTES;
        };
        auto issue = [&](int cs) {
            if (c_on) {
                const int sb = hc >> 1, h = hc & 1, slot = cs % C::RS;
                const uint8_t *q = cq + (uint64_t)sb * 2048 + 256 * h;
#pragma unroll
                for (int i = 0; i < 4; ++i) cp_async16(slot_addr(slot, i), q + 512 * i);
                cp_async16(slot_addr(slot, 4), chd + (uint64_t)sb * 256);
                cp_async8(rbnd + (uint32_t)((slot * BM + r) * 8), cbd + (uint64_t)sb * BOUND_BYTES);
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
                uint2 bnd;
                asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(bnd.x), "=r"(bnd.y) : "r"(rbnd + (uint32_t)((slot * BM + r) * 8)));
                // A slot h: the MMAs of half 2 gg + h - 2 are complete
                const uint32_t hu = 2u * (uint32_t)gg + (uint32_t)h;
                bool w_ok = hu < 2 || mbar_wait(&bar[BAR_EMPTY + (hu - 2) % C::NB], ((hu - 2) / C::NB) & 1u);
                // the epilogue has read the scales of superblock gg - 2
                if (h == 0 && w_ok) w_ok = mbar_wait(&bar[BAR_SD_EMPTY + (gg & 1)], (uint32_t)(((gg >> 1) & 1) ^ 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this half's A columns are complete
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
                    unpack_q45<F>(a_tm0 + 64 * h + 32 * jj, qsc, qh0, cch, sc_lo, sc_hi);
                }
                if (h == 0) {
                    // sub-mins duplicated per 16: K i of the mins operand holds m_{i/2}
                    const uint32_t amin = smem_u32(smem + C::OFF_AMIN) + (uint32_t)((gg & 1) * C::AMIN_BYTES);
                    uint32_t mw[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mw[i] = h2_splat((float)byte_of(i < 4 ? sm.m_lo : sm.m_hi, i & 3));
                    sts128(amin + sw32_offset(r, 0), mw[0], mw[1], mw[2], mw[3]);
                    sts128(amin + sw32_offset(r, 8), mw[4], mw[5], mw[6], mw[7]);
                    s_d[(gg & 1) * BM + r] = half_lo(hdr.x);
                    s_dmin[(gg & 1) * BM + r] = half_hi(hdr.x);
                }
                {
                    const uint32_t w1 = __reduce_max_sync(0xFFFFFFFFu, h ? bnd.y : bnd.x);
                    const uint32_t w1sb = h ? __reduce_max_sync(0xFFFFFFFFu, bnd.x + bnd.y) : 0u;
                    if (lane == 0) s_flag[16 * (gg & 1) + 8 * h + uw] = (uint8_t)unit_flag<F>(h, w1, w1sb, 0);
                }
                tmem_wait_st();
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[BAR_FULL + hu % C::NB]);
                    // the scales and both halves' unit flags are written
                    if (h == 1) mbar_arrive(&bar[BAR_SD_FULL + (gg & 1)]);
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
        // the piece's half-stages [hs0, hs1) (grouped: the whole tile)
        int hs0 = 0, hs1 = nstage;
        int dn = 0;  // dense: the block's pieces
        if constexpr (!G) {
            dn = dense_items<SK>(s_plan);
            have = dn > 0;
            if (have) {
                const Piece q = work_piece<F, G, SK>(p, s_list, s_plan, 0);
                t = q.t;
                hs0 = 2 * q.sb0;
                hs1 = 2 * q.sb1;
            }
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
        if (have) load_raw(cur, make_planes(F, p.packed + (uint64_t)e_cur * p.expert_bytes, p.N, nsb), row, hs0 >> 1, nsb, 0);
        while (have && ok) {
            bool have_n = false;
            int e_nxt = e_cur, n0_nxt = 0;
            int hs0_n = 0, hs1_n = nstage;
            const Planes P = make_planes(F, p.packed + (uint64_t)e_cur * p.expert_bytes, p.N, nsb);
            for (int hs = hs0; hs < hs1; ++hs) {
                const int gg = g + ((hs - hs0) >> 1);  // the block's superblock step
                const int h = hs & 1;
                // the next half's bytes (the next piece's first half at the
                // end of a piece) are in flight while this one is converted
                if (hs + 1 < hs1) {
                    load_raw(nxt, P, row, (hs + 1) >> 1, nsb, (hs + 1) & 1);
                } else if constexpr (!G && SK) {
                    have_n = k + 1 < dn;
                    if (have_n) {
                        const Piece q = dense_piece<F>(p, s_plan, k + 1);
                        n0_nxt = q.t.n0;
                        hs0_n = 2 * q.sb0;
                        hs1_n = 2 * q.sb1;
                        const int rn = n0_nxt + r < p.N ? n0_nxt + r : (int)p.N - 1;
                        load_raw(nxt, P, rn, q.sb0, nsb, 0);
                    }
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
                        const Planes Q{P.p0 + delta, P.p1 + delta, P.p2 + delta, P.p3 + delta, P.p4 + delta};
                        const int rn = n0_nxt + r < p.N ? n0_nxt + r : (int)p.N - 1;
                        load_raw(nxt, Q, rn, 0, nsb, 0);
                    }
                }
                // A slot h: the MMAs of half 2 gg + h - 2 are complete
                const uint32_t hu = 2u * (uint32_t)gg + (uint32_t)h;
                bool w_ok = hu < 2 || mbar_wait(&bar[BAR_EMPTY + (hu - 2) % C::NB], ((hu - 2) / C::NB) & 1u);
                // the epilogue has read the scales (and Q6_K categories) of superblock gg - 2
                if (h == 0 && w_ok) w_ok = mbar_wait(&bar[BAR_SD_EMPTY + (gg & 1)], (uint32_t)(((gg >> 1) & 1) ^ 1));
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                if constexpr (C::kTmemA) tc_fence_after();  // the MMAs that read this half's A columns are complete
                const uint32_t a_slot = a_base + h * C::A_SLOT;
                float d = 0.0f, dmin = 0.0f;
                // this warp's unit flag for the half: its rows' W1 bounds and
                // (Q6_K) the largest |sub-scale| of its rows' K sub-tile
                const uint32_t w1 = __reduce_max_sync(0xFFFFFFFFu, h ? cur.bnd.y : cur.bnd.x);
                const uint32_t w1sb = h ? __reduce_max_sync(0xFFFFFFFFu, cur.bnd.x + cur.bnd.y) : 0u;
                if constexpr (F == FMT_Q6_K) {
                    const uint32_t scj = my_jj ? cur.sc[1] : cur.sc[0];
                    int amax = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int v = (int)(int8_t)((scj >> (8 * i)) & 0xFF);
                        amax = max(amax, v < 0 ? -v : v);
                    }
                    const int wmax = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)amax);
                    if (lane == 0) s_flag[16 * (gg & 1) + 8 * h + uw] = (uint8_t)unit_flag<F>(h, w1, w1sb, wmax);
                    const bool big = wmax > 62;
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
                        unpack_q45<F>(a_tm0 + 64 * h + 32 * jj, qsc, qh0, cch, sc_lo, sc_hi);
                    }
                    if (h == 0) {
                        // sub-mins duplicated per 16: K i of the mins operand holds m_{i/2}
                        const uint32_t amin = smem_u32(smem + C::OFF_AMIN) + (uint32_t)((gg & 1) * C::AMIN_BYTES);
                        uint32_t mw[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) mw[i] = h2_splat((float)byte_of(i < 4 ? sm.m_lo : sm.m_hi, i & 3));
                        sts128(amin + sw32_offset(r, 0), mw[0], mw[1], mw[2], mw[3]);
                        sts128(amin + sw32_offset(r, 8), mw[4], mw[5], mw[6], mw[7]);
                    }
                    d = half_lo(cur.hdr.x);
                    dmin = half_hi(cur.hdr.x);
                    if (lane == 0) s_flag[16 * (gg & 1) + 8 * h + uw] = (uint8_t)unit_flag<F>(h, w1, w1sb, 0);
                }
                if (h == 0 && my_jj == 0) {
                    s_d[(gg & 1) * BM + r] = d;
                    s_dmin[(gg & 1) * BM + r] = dmin;
                }
                if constexpr (C::kTmemA) {
                    tmem_wait_st();
                    tc_fence_before();
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[BAR_FULL + hu % C::NB]);
                    // the scales and both halves' unit flags are written
                    if (h == 1) mbar_arrive(&bar[BAR_SD_FULL + (gg & 1)]);
                }
                cur = nxt;
            }
            g += (hs1 - hs0) >> 1;
            ++k;
            have = have_n;
            e_cur = e_nxt;
            row = n0_nxt + r < p.N ? n0_nxt + r : (int)p.N - 1;
            hs0 = hs0_n;
            hs1 = hs1_n;
        }
        if (!ok && lane == 0) set_timeout();
        }
    } else if constexpr (F == FMT_Q6_K) {
        // ------------------------------------------------ epilogue, Q6_K
        // 4 warps, thread = weight row x every token column; y accumulates
        // in TMEM columns COL_Y.. (Q6_K has no mins), read back once at the
        // end of each tile.  TMEM is read 16 columns at a time.
        const int ew = warp - w_epi<F>();    // 0..3
        const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
        const int r = 32 * quad + lane;
        float *s_d8 = reinterpret_cast<float *>(smem + C::OFF_D8) + 128 * ew;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16);
        const uint32_t y_tm = lane_addr + COL_Y;
        constexpr bool dbg = DBG;
        griddep_wait();  // the scales are written by the kernels before this one
        int ntiles = G ? 0 : dense_items<SK>(s_plan);
        if constexpr (G) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0));
            ntiles = ok ? (int)misc[1] : 0;
        }
        int64_t g = 0, u = 0;
        uint32_t epi_phase = 0;
        for (int k = 0; k < ntiles && ok; ++k) {
            const Piece pc = work_piece<F, G, SK>(p, s_list, s_plan, k);
            const Tile t = pc.t;
            const int64_t n = t.n0 + r;
            const int nc = t.n_mma / 16;
            bool first = true;
            // the token scales d8 of the next superblock, loaded one superblock ahead
            float d8n[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t tc = t.t0 + 32 * q + lane;
                d8n[q] = tc < t.t_end ? __ldg(p.d8t + pc.sb0 * p.Mp + tc) : 0.0f;
            }
            for (int64_t sb = pc.sb0; sb < pc.sb1; ++sb) {
                const int64_t gg = g + sb - pc.sb0;
                const int b = (int)(gg & 1);
#pragma unroll
                for (int q = 0; q < 4; ++q) s_d8[32 * q + lane] = d8n[q];
                __syncwarp();
                if (sb + 1 < pc.sb1) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t tc = t.t0 + 32 * q + lane;
                        d8n[q] = tc < t.t_end ? __ldg(p.d8t + (sb + 1) * p.Mp + tc) : 0.0f;
                    }
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_SD_FULL + b], (uint32_t)((gg >> 1) & 1)))) {
                    ok = false;
                    break;
                }
                const float dd = s_d[b * BM + r];
                const int nu = sb_plan(ld_flags(flag_sa + 16 * b), ld_flags(flag_sa + 16 * b + 8)).n;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[BAR_SD_EMPTY + b]);
                if (t.ntok == 0) continue;
                if (nu == 1) {
                    // one unit for the superblock (the common case)
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_U_FULL + (int)(u % NU)], (uint32_t)((u / NU) & 1)))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xa = lane_addr + 128 * (uint32_t)(u % NU);
                    if constexpr (DBG) debug_units(p.isum_out, p.msum_out, p.N, nsb, xa, false, 0u, false, 0u, t.n_mma, t.t0, t.t_end, n, sb);
                    else if (first) fold_units_q6<false, true>(xa, 0u, y_tm, nc, dd, s_d8);
                    else fold_units_q6<false, false>(xa, 0u, y_tm, nc, dd, s_d8);
                    if (!dbg) tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[BAR_U_EMPTY + (int)(u % NU)]);
                    ++u;
                    first = false;
                    continue;
                }
                // several units, two at a time: y += d8 * d * (Ua + Ub)
                for (int left = nu; left > 0 && ok;) {
                    const int m = left >= 2 ? 2 : 1;
                    bool w_ok = mbar_wait(&bar[BAR_U_FULL + (int)(u % NU)], (uint32_t)((u / NU) & 1));
                    if (w_ok && m == 2) w_ok = mbar_wait(&bar[BAR_U_FULL + (int)((u + 1) % NU)], (uint32_t)(((u + 1) / NU) & 1));
                    if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xa = lane_addr + 128 * (uint32_t)(u % NU), xb = lane_addr + 128 * (uint32_t)((u + 1) % NU);
                    if constexpr (DBG) debug_units(p.isum_out, p.msum_out, p.N, nsb, xa, m == 2, xb, false, 0u, t.n_mma, t.t0, t.t_end, n, sb);
                    else if (m == 2 && first) fold_units_q6<true, true>(xa, xb, y_tm, nc, dd, s_d8);
                    else if (m == 2) fold_units_q6<true, false>(xa, xb, y_tm, nc, dd, s_d8);
                    else if (first) fold_units_q6<false, true>(xa, xb, y_tm, nc, dd, s_d8);
                    else fold_units_q6<false, false>(xa, xb, y_tm, nc, dd, s_d8);
                    if (!dbg) tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bar[BAR_U_EMPTY + (int)(u % NU)]);
                        if (m == 2) mbar_arrive(&bar[BAR_U_EMPTY + (int)((u + 1) % NU)]);
                    }
                    u += m;
                    left -= m;
                    first = false;
                }
                if (!ok) break;
            }
            if (!ok) break;
            if (!dbg && t.ntok > 0) {
                tc_fence_after();
                const bool whole = G || !SK || (pc.sb0 == 0 && pc.sb1 == (int)nsb);
                float *mine = own_slot(p, k);
                for (int c = 0; c < nc; ++c) {
                    uint32_t vy[16];
                    tmem_ld16(y_tm + 16 * c, vy);
                    tmem_wait_ld();
                    if (!whole) {
                        // a tile split between blocks: this block's partial sums
#pragma unroll
                        for (int i = 0; i < 16; ++i) mine[(16 * c + i) * BM + r] = __uint_as_float(vy[i]);
                    } else if (n < p.N) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int64_t tt = t.t0 + 16 * c + i;
                            if (tt < t.t_end) p.y[tt * p.N + n] = __uint_as_float(vy[i]);
                        }
                    }
                }
                if (!whole && !split_finish(p.part, p.tile_cnt, p.units, nsb, pc.tile, p.y, p.N, n, t.t0, t.t_end, 0,
                                            16 * nc, n < p.N, ew == 0 && lane == 0, lane, &epi_phase, bar, misc)) {
                    ok = false;
                    break;
                }
            }
            g += pc.sb1 - pc.sb0;
        }
        if (!ok && lane == 0) set_timeout();
    } else {
        // ------------------------------------------------ epilogue, Q4_K / Q5_K
        // 8 warps, thread = weight row x 64 token columns, y in registers.
        // Each unit is folded as it lands, the first of a superblock with
        // msum: y += d8 * (d * U0 - dmin * msum), then y += d8 * d * Uk.
        const int ew = warp - w_epi<F>();    // 0..7
        const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
        const int ch = ew >> 2;              // token columns 64*ch .. +63
        const int r = 32 * quad + lane;
        float *s_d8 = reinterpret_cast<float *>(smem + C::OFF_D8) + 64 * ew;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quad) << 16) + 64 * ch;
        griddep_wait();  // the scales are written by the kernels before this one
        int ntiles = G ? 0 : dense_items<SK>(s_plan);
        if constexpr (G) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_TILES], 0));
            ntiles = ok ? (int)misc[1] : 0;
        }
        // 32-bit counters: a block runs at most TILE_CAP tiles of at most 2^22 superblocks
        uint32_t g = 0, u = 0, epi_phase = 0;
        for (int k = 0; k < ntiles && ok; ++k) {
            const Piece pc = work_piece<F, G, SK>(p, s_list, s_plan, k);
            const Tile t = pc.t;
            const int n = t.n0 + r;
            float y[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) y[i] = 0.0f;
            const bool cols = 64 * ch < t.n_mma;
            // this warp's 8-column chunks holding tokens of the tile
            const int nch = cols ? (t.n_mma - 64 * ch >= 64 ? 8 : (t.n_mma - 64 * ch + 7) / 8) : 0;
            // this warp's 64 token scales d8 of the next superblock, loaded one superblock ahead
            const int tc = t.t0 + 64 * ch + lane;
            const float *d8col = p.d8t + tc;
            float d8n0 = tc < t.t_end ? __ldg(d8col + (int64_t)pc.sb0 * p.Mp) : 0.0f;
            float d8n1 = (tc + 32) < t.t_end ? __ldg(d8col + (int64_t)pc.sb0 * p.Mp + 32) : 0.0f;
            for (int sb = pc.sb0; sb < pc.sb1; ++sb) {
                const uint32_t gg = g + (uint32_t)(sb - pc.sb0);
                const int b = (int)(gg & 1);
                s_d8[lane] = d8n0;
                s_d8[lane + 32] = d8n1;
                __syncwarp();
                if (sb + 1 < pc.sb1) {
                    const float *d8p = d8col + (int64_t)(sb + 1) * p.Mp;
                    d8n0 = tc < t.t_end ? __ldg(d8p) : 0.0f;
                    d8n1 = (tc + 32) < t.t_end ? __ldg(d8p + 32) : 0.0f;
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[BAR_SD_FULL + b], (uint32_t)((gg >> 1) & 1)))) {
                    ok = false;
                    break;
                }
                const float dd = s_d[b * BM + r], dm = s_dmin[b * BM + r];
                const int nu = sb_plan(ld_flags(flag_sa + 16 * b), ld_flags(flag_sa + 16 * b + 8)).n;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[BAR_SD_EMPTY + b]);
                if (t.ntok == 0) continue;
                // the superblock's units, folded as they land; msum, issued
                // after the last unit into its one slot and covered by that
                // unit's commit, is folded with it (the units before it never
                // wait for it)
                const uint32_t xm = lane_addr + COL_M;
#pragma unroll 1
                for (int v = 0; v < nu; ++v, ++u) {
                    const bool last = v == nu - 1;
                    bool w_ok = mbar_wait(&bar[BAR_U_FULL + (int)(u % NU)], (u / NU) & 1);
                    if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xu = lane_addr + 128 * (u % NU);
                    if (cols) {
                        // 8 columns a TMEM round trip: with y[64] and the loop's
                        // state live, 16 would spill
                        if constexpr (DBG) debug_units(p.isum_out, p.msum_out, p.N, nsb, xu, false, 0u, last, xm, 64, t.t0 + 64 * ch, t.t_end, n, sb);
                        else if (last) fold_unit_q45<8, true>(y, xu, xm, dd, dm, s_d8, nch);
                        else fold_unit_q45<8, false>(y, xu, xm, dd, 0.0f, s_d8, nch);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bar[BAR_U_EMPTY + (int)(u % NU)]);
                        if (last) mbar_arrive(&bar[BAR_M_EMPTY]);
                    }
                }
                if (!ok) break;
            }
            if (!ok) break;
            if constexpr (!DBG) {
                // a whole tile goes to y; a tile split between blocks to this
                // block's partial slot, finished by the last of its blocks
                const bool whole = G || !SK || (pc.sb0 == 0 && pc.sb1 == (int)nsb);
                const int c0 = t.t0 + 64 * ch;
                const int lim = whole ? t.t_end - c0 : 64;
                float *yp = whole ? p.y + (int64_t)c0 * p.N + n : own_slot(p, k) + 64 * ch * BM + r;
                const int64_t ys = whole ? p.N : BM;
                if (cols && (n < p.N || !whole)) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (i < lim) yp[(int64_t)i * ys] = y[i];
                }
                if (!whole && !split_finish(p.part, p.tile_cnt, p.units, nsb, pc.tile, p.y, p.N, n, t.t0, t.t_end,
                                            64 * ch, 64, n < p.N && cols, ew == 0 && lane == 0, lane, &epi_phase,
                                            bar, misc)) {
                    ok = false;
                    break;
                }
            }
            g += (uint32_t)(pc.sb1 - pc.sb0);
        }
        if (!ok && lane == 0) set_timeout();
    }

    // TMEM is released once every warp is done with it.  An explicit
    // mbarrier, not __syncthreads: the roles reach the end at different
    // times on diverged lanes (the TMA and MMA roles run on lane 0), and a
    // block barrier reached that way was measured to let the MMA warp pass
    // while the epilogue warps were still at work.
    __syncwarp();
    tc_fence_before();
    if (lane == 0) mbar_arrive(&bar[BAR_END]);
    if (warp == W_MMA) {
        if (!mbar_wait(&bar[BAR_END], 0) && lane == 0) set_timeout();
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
                                                        __half *__restrict__ b16, float *__restrict__ d8t,
                                                        int *__restrict__ tile_cnt, int64_t n_cnt) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 quants
    // the GEMM's split-tile counters start from zero (the image has at least as many threads)
    if (i < n_cnt) tile_cnt[i] = 0;
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

// The workspace: the activation image (a16, b16, d8t: all a launch needs),
// then, for the dense split-tile schedule, two fp32 partial tiles per SM and
// a counter per tile.
struct WsLayout {
    uint64_t a16, b16, d8t, total;
    uint64_t part, cnt, total_split;
    int64_t Mp, tiles;
};

static int device_sms() {
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

static WsLayout ws_layout(int64_t M, int64_t N, int64_t K) {
    WsLayout w;
    w.Mp = (M + 3) & ~int64_t(3);
    w.a16 = 0;
    w.b16 = align256((uint64_t)M * K * 2);
    w.d8t = w.b16 + align256((uint64_t)M * (K / 16) * 2);
    w.total = w.d8t + align256((uint64_t)(K / QK) * w.Mp * 4);
    w.tiles = ((N + BM - 1) / BM) * ((M + BT - 1) / BT);
    w.part = w.total;
    w.cnt = w.part + (uint64_t)2 * device_sms() * BT * BM * 4;
    w.total_split = w.cnt + align256((uint64_t)w.tiles * 4);
    return w;
}

// M below which the CUDA-core token-group kernel is used instead

size_t gemm_workspace_bytes(int, int64_t M, int64_t N, int64_t K) {
    if (M < GEMM_TC_MIN_M) return 0;
    return (size_t)ws_layout(M, N, K).total_split;
}

size_t gemm_workspace_min_bytes(int, int64_t M, int64_t N, int64_t K) {
    if (M < GEMM_TC_MIN_M) return 0;
    return (size_t)ws_layout(M, N, K).total;
}

template <int F>
static cudaError_t launch_gemm_f(const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, const int32_t *offsets,
                                 int64_t E, uint64_t expert_bytes, float *y, uint8_t *ws, size_t ws_bytes,
                                 cudaStream_t s, int32_t *isum_out = nullptr, int32_t *msum_out = nullptr) {
    using Cf = Cfg<F>;
    const WsLayout L = ws_layout(M, N, K);
    __half *a16 = reinterpret_cast<__half *>(ws + L.a16);
    __half *b16 = reinterpret_cast<__half *>(ws + L.b16);
    float *d8t = reinterpret_cast<float *>(ws + L.d8t);
    // dense: the split-tile schedule (one block per SM, each an even share of
    // the tiles x superblocks steps) where a block per tile would leave the
    // last wave of tiles mostly empty and every block still gets 16
    // superblock steps or more (fewer: its start-up and the partial tiles'
    // handoff cost more than the wave saves; measured on GB300), and the
    // workspace has its room
    bool split = false;
    if (!offsets && ws_bytes >= L.total_split) {
        const int64_t n_sm = device_sms(), nsb = K / QK;
        const int64_t waves = (L.tiles + n_sm - 1) / n_sm;
        const bool ragged = 4 * L.tiles < 3 * waves * n_sm;  // the tiles fill under 3/4 of their waves
        split = (ragged && L.tiles * nsb >= 16 * n_sm) || (launch_flags() & LAUNCH_GEMM_SPLIT);
    }
    int *tile_cnt = split ? reinterpret_cast<int *>(ws + L.cnt) : nullptr;
    const int64_t n_cnt = split ? L.tiles : 0;
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, act_image_kernel, a.qs, a.bsums, a.d, M, K, L.Mp, a16, b16, d8t,
                                           tile_cnt, n_cnt);
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
        const void *fns[6] = {(const void *)gemm_kernel<F, false, false, false>,
                              (const void *)gemm_kernel<F, false, false, true>,
                              (const void *)gemm_kernel<F, true, false, false>,
                              (const void *)gemm_kernel<F, false, true, false>,
                              (const void *)gemm_kernel<F, false, true, true>,
                              (const void *)gemm_kernel<F, true, true, false>};
        for (const void *fn : fns) {
            const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
            if (e != cudaSuccess) return e;
        }
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
    p.isum_out = isum_out;
    p.msum_out = msum_out;
    p.part = split ? reinterpret_cast<float *>(ws + L.part) : nullptr;
    p.tile_cnt = tile_cnt;
    if (isum_out) {
        const size_t bytes = (size_t)M * (size_t)N * (size_t)(K / QK) * sizeof(int32_t);
        cudaError_t e = cudaMemsetAsync(isum_out, 0, bytes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(msum_out, 0, bytes, s);
        if (e != cudaSuccess) return e;
    }
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
    if (!offsets) {
        p.units = tiles * p.nsb;
        if (split) {
            const int64_t n_sm = device_sms();
            blocks = p.units < n_sm ? p.units : n_sm;
        }
    }
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
    if (isum_out) {
        if (offsets) return cudaLaunchKernelEx(&cfg, gemm_kernel<F, true, true, false>, ma, mb, p);
        if (split) return cudaLaunchKernelEx(&cfg, gemm_kernel<F, false, true, true>, ma, mb, p);
        return cudaLaunchKernelEx(&cfg, gemm_kernel<F, false, true, false>, ma, mb, p);
    }
    if (offsets) return cudaLaunchKernelEx(&cfg, gemm_kernel<F, true, false, false>, ma, mb, p);
    if (split) return cudaLaunchKernelEx(&cfg, gemm_kernel<F, false, false, true>, ma, mb, p);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<F, false, false, false>, ma, mb, p);
}

cudaError_t launch_gemm_tc(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M, const int32_t *offsets,
                           int64_t E, uint64_t expert_bytes, float *y, void *workspace, size_t workspace_bytes,
                           cudaStream_t s) {
    if (M < GEMM_TC_MIN_M || !workspace) return cudaErrorNotSupported;
    if (workspace_bytes < ws_layout(M, N, K).total) return cudaErrorInvalidValue;
    if (M > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX / 2) return cudaErrorNotSupported;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t wb = workspace_bytes;
    if (f == FMT_Q4_K) return launch_gemm_f<FMT_Q4_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, wb, s);
    if (f == FMT_Q5_K) return launch_gemm_f<FMT_Q5_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, wb, s);
    return launch_gemm_f<FMT_Q6_K>(packed, N, K, a, M, offsets, E, expert_bytes, y, ws, wb, s);
}

cudaError_t launch_gemm_tc_partials(int f, const void *packed, int64_t N, int64_t K, Q8K a, int64_t M,
                                    const int32_t *offsets, int64_t E, uint64_t expert_bytes, int32_t *isum,
                                    int32_t *msum, void *workspace, size_t workspace_bytes, cudaStream_t s) {
    if (M < GEMM_TC_MIN_M || !workspace) return cudaErrorNotSupported;
    if (workspace_bytes < ws_layout(M, N, K).total) return cudaErrorInvalidValue;
    if (M > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX / 2) return cudaErrorNotSupported;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t wb = workspace_bytes;
    if (f == FMT_Q4_K)
        return launch_gemm_f<FMT_Q4_K>(packed, N, K, a, M, offsets, E, expert_bytes, nullptr, ws, wb, s, isum, msum);
    if (f == FMT_Q5_K)
        return launch_gemm_f<FMT_Q5_K>(packed, N, K, a, M, offsets, E, expert_bytes, nullptr, ws, wb, s, isum, msum);
    return launch_gemm_f<FMT_Q6_K>(packed, N, K, a, M, offsets, E, expert_bytes, nullptr, ws, wb, s, isum, msum);
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
