// dh_coarse_tc8.cu -- kernels (2)+(3), tcgen05 path with 8-bit operands: coarse pass on the
// 5th-generation tensor cores (kind::f8f6f4, A from tensor memory) and the fused block
// top-KCAND epilogue.
//
// radiance_drafthead.py, _draft_head_int2 and _emit.  The page's kernel feeds its dot product
// with the bf16 bit pattern 1 + v/4 and collapses the scale and zero into two accumulator
// operations per group.  This kernel computes the same group term with exact 8-bit operands:
//   * weight: the e4m3 byte patterns 0..15 are exactly p 2^-9, so the 2-bit code of a plane
//     masked in place is an exact e4m3 weight: v 2^-9 for planes 0 and 2 (mask 0x03), 4 v 2^-9
//     for planes 1 and 3 (mask 0x0C), planes 2-3 after a 4-bit shift.  One AND (plus one
//     shift) turns a 32-bit word of packed bytes into four weights of one plane, in k order;
//   * x: every row is scaled by a power of two 2^e (max |x 2^e| in [128, 256)) and written as
//     T e4m3 terms, x 2^e ~ t1 + w2 t2 (+ w3 t3), each term the rounded residual of the ones
//     before at its own power-of-two scale (per-row weights w2, w3; dh_prep.cu).  The terms are
//     stacked along the MMA's N dimension (rows t MP + m) and recombined in fp32 in the
//     epilogue.  Two terms represent every element of an ordinary row exactly; a launch whose
//     rows need the third term (the staging kernel measures each row's two-term error) runs the
//     T = 3 instance of this kernel, the T = 2 instance returning at once, and vice versa;
//   * per group g (128 consecutive k of one plane q), with p = sum_t w_t D_t the recombined
//     partial, sum_k x_k v_k = 2^9 p / f (f = 1 for even q, 4 for odd q), and the page's
//     group term S sum_k x_k (1 + v_k/4) - ZS xs = (S/4) sum_k x_k v_k + (S - ZS) xs, so
//         c[m, n] = 2^-e * sum_g ( (2^7/f) S[n,g] p + (S[n,g] - ZS[n,g]) xs'[m,g] )
//     with xs' the group sums of the represented x (in the scaled units): the scale and zero
//     are applied to the fp32 partial of every group, never to the weight.
//
// Roles (24 or 20 warps, one CTA per SM, persistent over 128-row vocabulary tiles).  The unit of
// handoff is a span (N = 32: the four planes of 512 k) or half a span (larger N: planes 2u,
// 2u+1); unit q uses tensor-memory slot q % 2 (an A buffer and one accumulator per group).
// Issuing a tcgen05.mma holds the issuing warp for many cycles, so each plane has its own issuer
// warp: the four issuers of a span work at once, each on its own SM sub-partition, and each of
// them takes every unit that holds its plane, in order (every barrier's phases are awaited in
// order).  With one unit per span two sets of dequant warps share each span's A buffer, which
// halves the time a slot waits for its weights.
//   warp 0        TMA: per span one [128 rows x 128 B] box of packed codes (two for the 4-bit
//                 head) and four [128 k x N] boxes of the staged x terms (128-byte swizzle)
//                 into a stage ring; per tile a bulk copy of the tile's S and ZS rows
//                 (contiguous in memory) into a double-buffered shared copy for the epilogue
//   warps 1-3 and the one after the epilogue   MMA issuers of planes 0..3, a whole warp each
//                 (one elected lane issues): per unit 4 x tcgen05.mma kind::f8f6f4 (M = 128,
//                 K = 32) of their plane, one commit for the unit's accumulators and one for
//                 the stage
//   warps 4-11    dequant, two sets of four warps (one set where every launch body has two
//                 units per span): one TMEM lane (= one vocabulary row) per thread; with two
//                 sets, set c writes k half c of every plane (2-bit layouts) or planes 2c,
//                 2c + 1 (4-bit head); a single set every plane (tcgen05.st, one wait per unit)
//   next 8 warps  epilogue, two halves of four warps (one per TMEM lane quarter): half h folds
//                 planes 2h, 2h+1 of every span -- tcgen05.ld of the partials, recombination of
//                 the terms, scale/zero fold into fp32 registers -- and at the tile end writes its
//                 half of the coarse values; the selection warp adds the halves
//   next 2 warps  block top-KCAND of the previous tile (overlaps the current one): two lanes
//                 per (batch column, block) pair each keep an insertion list of the best 8 of
//                 their 32 rows, then merge
//   last warp     idle: it completes the last warpgroup, so that each warpgroup can set its own
//                 register budget (setmaxnreg: the TMA / issuer and issuer / selection / idle
//                 warpgroups give registers to the epilogue's)
// Every handoff is an mbarrier; every wait is bounded.
//
// The 4-bit head (BITS = 4, half split, bias 16; _quantize_head_now's 4-bit variant) runs the
// same pipeline: a nibble masked in place is the exact e4m3 weight v 2^-9 (v in 0..15), and two
// 128-byte boxes of a row (packed bytes 256 span ..) carry four groups -- low and high nibbles
// of each box -- so one span is again four planes of 128 k, sixteen MMAs and four groups, with
// NG = H / 512 spans per row.  The fold becomes (2^9 / 16) S p = 32 S p for every plane.
#include "dh_common.cuh"
#include "dh_internal.h"
#include "dh_tcgen05.cuh"

#include <climits>
#include <type_traits>

namespace dh {

namespace {

constexpr int kTileRows = 128;

constexpr int kTmemCols = 512;
constexpr int kPkBytes = kTileRows * kSpanBytes; // 16 KB packed box per span
constexpr int kSmemLimit8 = 232448;
// The tile's coarse values for the selection warps: one 64-value block per (batch column,
// block) pair, pairs kRedPitch floats apart (16-byte aligned, bank-conflict free per lane).
constexpr int kRedPitch = 68;
// Warp roles: 0 TMA, 1-3 the MMA issuers of planes 0-2, 4-7 the first dequant set (one warp per
// TMEM lane quarter), then, for launches with one unit per span, the second dequant set (8-11);
// then the epilogue (two halves of four warps), the issuer of plane 3 and the two selection
// warps.
// The four issuers sit on the four SM sub-partitions (warp % 4).  Launches that never use the
// second dequant set leave it out, for registers.
constexpr int kWarpTma = 0, kWarpDq0 = 4;
constexpr int kDqWarps = 4; // warps of one dequant set
constexpr int kEpWarps = 8; // two halves of four
constexpr int kIssuers = 4; // one MMA issuer warp per plane
template <bool kTwoSets> struct Roles {
    static constexpr int kEp0 = kTwoSets ? 12 : 8;           // first epilogue warp
    static constexpr int kSel0 = kEp0 + kEpWarps + 1;        // the two selection warps
    static constexpr int kSel1 = kEp0 + kEpWarps + 2;
    // + the plane-3 issuer, the selection warps and one idle warp: whole warpgroups, so that
    // every warpgroup can set its own register budget
    static constexpr int kWarps = kEp0 + kEpWarps + 4;
    static constexpr int kThreads = 32 * kWarps;
    // registers a thread: at launch (the kernel's count, checked on the host), then per
    // warpgroup -- the TMA / issuer and the issuer / selection warpgroups give registers to
    // the epilogue's; the budgets add up to the launch's exactly
    static constexpr int kRegsLaunch = kTwoSets ? 80 : 96;
    // light warpgroups: 48 in 24-warp launches, 64 in 20-warp ones (each measured faster)
    static constexpr int kRegsLight = kTwoSets ? 48 : 64;
    static constexpr int kRegsDq = kTwoSets ? 80 : 96;
    static constexpr int kRegsEp = (kRegsLaunch * (kWarps / 4) - 2 * kRegsLight -
                                    (kTwoSets ? 2 : 1) * kRegsDq) / 2;
    static_assert(kWarps % 4 == 0, "whole warpgroups");
    // the dequant branch sets no budget: its warpgroups keep the launch's, and only the light
    // and epilogue branches move registers (a setmaxnreg.inc that asks for more than the decs
    // free waits forever)
    static_assert(kRegsDq == kRegsLaunch, "the dequant warpgroups keep the launch budget");
    static_assert(2 * (kRegsLaunch - kRegsLight) == 2 * (kRegsEp - kRegsLaunch),
                  "the epilogue takes exactly what the light warpgroups free");
    static_assert(2 * kRegsLight + (kTwoSets ? 2 : 1) * kRegsDq + 2 * kRegsEp ==
                      kRegsLaunch * (kWarps / 4), "register budgets must add up");
    __device__ static int issuer_plane(int warp)
    {
        return (warp >= 1 && warp <= 3) ? warp - 1 : (warp == kEp0 + kEpWarps ? 3 : -1);
    }
};

// Batch rows per launch MP in {16, 32}; x in T in {2, 3} e4m3 terms; MMA N = T * MP.
// The unit of handoff is a whole span at N = 32 (kU = 1: 4 planes, 16 MMAs) and half a span
// otherwise (kU = 2: planes 2u, 2u+1, 8 MMAs).  Tensor memory holds two unit slots, each an A
// buffer (32 columns of e4m3 per plane) and one N-column fp32 accumulator per group of the
// unit's planes; unit q uses slot q % 2.  Groups of 64 (kPackG64, MP = 16 only) put two
// accumulators on each plane.
template <int MP, int PACK, int T_> struct Cfg8 {
    static constexpr int T = T_;
    static constexpr int kPkBoxes = PACK == kPackHalf4 ? 2 : 1; // packed boxes per span
    static constexpr int N = MP * T;
    static constexpr int G = PACK == kPackG64 ? 64 : 128;   // weight group size
    static constexpr int kGPP = 128 / G;                    // groups per plane of a span
    static constexpr int kU = (MP == 16 && G == 128 && T == 2) ? 1 : 2; // units per span
    // two dequant sets, each a k half of every plane (2-bit layouts) or one packed box (4-bit
    // head), for the whole-span units of 16-row launches (for 32-row launches the second set
    // measured slower)
    static constexpr int kDqSets = kU == 1 ? 2 : 1;
    static constexpr int kPP = 4 / kU;                      // planes per unit
    static constexpr uint32_t kACols = 32 * kPP;
    static constexpr uint32_t kSlotCols = kACols + kPP * kGPP * N; // one accumulator per group
    static constexpr int K = 2;                             // unit slots
    static constexpr uint32_t kXBytes = N * 512;            // 4 planes x 128 k x N rows
    static constexpr uint32_t kStage = kPkBoxes * kPkBytes + kXBytes; // multiple of 1024
    static_assert(K * kSlotCols <= kTmemCols, "two unit slots must fit");
    static_assert(N % 16 == 0 && N <= 256, "MMA N out of range");
};

struct Tc8Params {
    const uint16_t *S;
    const uint16_t *ZS;
    const float *xs2;       // [MP][NGt] group sums of the 2-term representation (scaled units)
    const float *xs3;       // [MP][NGt] group sums of the 3-term representation
    const float *row_f;     // [3][kTc8MaxMP] per batch row: 2^-e, weights w2 and w3
    const int *row_terms;   // [MP] terms each row needs (2 or 3)
    int V, H, m0, mrows, kcand, ntiles, nstage2, nstage3; // stage counts of the two bodies
    long long ncand;
    float *cand_val;
    int32_t *cand_idx;
    float *coarse;
    int *timeout_flag;
};

// L2 prefetch of one [128 rows x 128 B] box of a 2-D tensor map (x a multiple of 16 bytes),
// and of a contiguous byte range (address and size multiples of 16).
__device__ __forceinline__ void prefetch_l2_box(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void prefetch_l2_bytes(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// kind::f8f6f4 instruction descriptor: D f32, A e4m3, B e4m3, both K-major, M = 128, N.
__host__ __device__ constexpr uint32_t make_idesc_f8(int N)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

// e4m3 weights of plane P from a word of four packed bytes (four consecutive k): the codes
// masked in place, v 2^-9 (even P) or 4 v 2^-9 (odd P), exact e4m3 values
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::
                     "r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                 "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

template <int P>
__device__ __forceinline__ uint32_t deq4_e4m3(uint32_t w)
{
    return (P >= 2 ? (w >> 4) : w) & ((P & 1) ? 0x0C0C0C0Cu : 0x03030303u);
}

// The 4-bit head: the low / high nibble of each byte, v 2^-9 with v in 0..15 (e4m3 bytes 0..15
// are exactly p 2^-9: subnormals up to 7, then 2^-6 (1 + m/8) = (8 + m) 2^-9).
__device__ __forceinline__ uint32_t deq_nib_lo(uint32_t w) { return w & 0x0F0F0F0Fu; }
__device__ __forceinline__ uint32_t deq_nib_hi(uint32_t w) { return (w >> 4) & 0x0F0F0F0Fu; }

// The contiguous-4 layout (the page's packing ablation): the eight words w[8p .. 8p+7] of a
// span are group p's 128 codes, byte j holding k = 4j .. 4j+3.  The four fields of every byte
// masked to the low bits (v 2^-9) and transposed 4 x 4 by byte permutes give four words of
// e4m3 weights in k order: the price of the layout is this transpose (15 operations per
// 16 weights against 4 for the quarter split).
__device__ __forceinline__ void deq_c4(uint32_t w, uint32_t (&o)[4])
{
    const uint32_t p0 = w & 0x03030303u, p1 = (w >> 2) & 0x03030303u;
    const uint32_t p2 = (w >> 4) & 0x03030303u, p3 = (w >> 6) & 0x03030303u;
    const uint32_t t0 = __byte_perm(p0, p1, 0x5140), t1 = __byte_perm(p0, p1, 0x7362);
    const uint32_t t2 = __byte_perm(p2, p3, 0x5140), t3 = __byte_perm(p2, p3, 0x7362);
    o[0] = __byte_perm(t0, t2, 0x5410);
    o[1] = __byte_perm(t0, t2, 0x7632);
    o[2] = __byte_perm(t1, t3, 0x5410);
    o[3] = __byte_perm(t1, t3, 0x7632);
}

// Weight group (index into a row's H/128 groups, = first k / 128) of plane `plane` of span
// `span` (NG = H / 512 spans per row).  Quarter split: one 128-byte box per span, plane p at
// k = p H/4 + 128 span.  Half split (4 bits): two 128-byte boxes per span (packed bytes
// 256 span ..), plane p = 2 box + half at k = half H/2 + 128 (2 span + box).  Contiguous-4:
// the span's 512 consecutive k, plane p = group 4 span + p.
template <int PACK>
__device__ __forceinline__ int plane_group(int plane, int span, int NG)
{
    if constexpr (PACK == kPackHalf4) return (plane & 1) * 2 * NG + 2 * span + (plane >> 1);
    else if constexpr (PACK == kPackContig2) return 4 * span + plane;
    else return plane * NG + span;
}

// Block top-KCAND of up to 4 (batch column, block) pairs at once.  Lane l holds rows l and
// l + 32 of each pair's 64-row block as order keys (0 = no row); one round takes the largest
// key by redux.sync, equal values go to the lower row.
template <int NB>
__device__ __forceinline__ void select_pairs(uint32_t (&k0)[NB], uint32_t (&k1)[NB],
                                             const int (&base_row)[NB], float *const (&oval)[NB],
                                             int32_t *const (&oidx)[NB], int kcand, int lane)
{
    for (int r = 0; r < kcand; ++r) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t km = __reduce_max_sync(0xffffffffu, k0[b] > k1[b] ? k0[b] : k1[b]);
            const unsigned b0 = __ballot_sync(0xffffffffu, k0[b] == km && km != 0u);
            const unsigned b1 = __ballot_sync(0xffffffffu, k1[b] == km && km != 0u);
            const int row = b0 ? (__ffs(b0) - 1) : (b1 ? 32 + __ffs(b1) - 1 : -1);
            if (row == lane) k0[b] = 0u;
            if (row == lane + 32) k1[b] = 0u;
            if (lane == 0 && oval[b] != nullptr) {
                oval[b][r] = row >= 0 ? f32_from_order_key(km) : -INFINITY;
                oidx[b][r] = row >= 0 ? base_row[b] + row : -1;
            }
        }
    }
}

// (va, ra) ranks above (vb, rb): larger value, equal values to the lower row (an empty slot,
// row -1, loses every tie).
__device__ __forceinline__ bool ranks_above(float va, int ra, float vb, int rb)
{
    return va > vb || (va == vb && static_cast<uint32_t>(ra) < static_cast<uint32_t>(rb));
}

__device__ __forceinline__ void cmp_swap(float (&v)[8], int (&r)[8], int a, int b)
{
    const bool sw = ranks_above(v[b], r[b], v[a], r[a]);
    const float va = v[a], vb = v[b];
    const int ra = r[a], rb = r[b];
    v[a] = sw ? vb : va;
    v[b] = sw ? va : vb;
    r[a] = sw ? rb : ra;
    r[b] = sw ? ra : rb;
}

// Block top-KCAND for KCAND <= 8, two lanes per (batch column, block) pair: lane 2i + h keeps the
// best 8 of rows 32h .. 32h + 31 of its pair's block (insertion, as select_lane8), then lane 2i
// merges the two lists: the best 8 of the 16 are the better of list[k] and partner[7 - k]
// (a bitonic sequence), sorted by a bitonic merge.  Every lane of the warp takes part (shuffles);
// `live` is false for lanes whose pair is past the batch or the head.
__device__ __forceinline__ void select_pair2(bool live, const float *vals0, const float *vals1,
                                             int base_row, int V, int kcand, float *oval,
                                             int32_t *oidx, float *coarse, int lane)
{
    const int h = lane & 1;
    float v[8];
    int r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = -INFINITY;
        r[k] = -1;
    }
    if (live) {
#pragma unroll 2
        for (int j4 = 0; j4 < 8; ++j4) {
            const float4 u0 = reinterpret_cast<const float4 *>(vals0 + 32 * h)[j4];
            const float4 u1 = reinterpret_cast<const float4 *>(vals1 + 32 * h)[j4];
            const float uu[4] = {u0.x + u1.x, u0.y + u1.y, u0.z + u1.z, u0.w + u1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float xv = uu[e];
                const int row = base_row + 32 * h + 4 * j4 + e;
                if (coarse && row < V) coarse[row] = xv;
                bool c[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) c[k] = xv > v[k];
#pragma unroll
                for (int k = 7; k > 0; --k) {
                    v[k] = c[k] ? (c[k - 1] ? v[k - 1] : xv) : v[k];
                    r[k] = c[k] ? (c[k - 1] ? r[k - 1] : row) : r[k];
                }
                v[0] = c[0] ? xv : v[0];
                r[0] = c[0] ? row : r[0];
            }
        }
    }
    float pv[8];
    int pr[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        pv[k] = __shfl_xor_sync(0xffffffffu, v[k], 1);
        pr[k] = __shfl_xor_sync(0xffffffffu, r[k], 1);
    }
    if (!live || h != 0) return;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (ranks_above(pv[7 - k], pr[7 - k], v[k], r[k])) {
            v[k] = pv[7 - k];
            r[k] = pr[7 - k];
        }
    }
#pragma unroll
    for (int s = 4; s > 0; s >>= 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if ((k & s) == 0) cmp_swap(v, r, k, k + s);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < kcand) {
            oval[k] = v[k];
            oidx[k] = r[k];
        }
}

// Two dequant sets exactly when the two-term body has one unit per span.
template <int MP, int PACK> constexpr bool two_sets() { return Cfg8<MP, PACK, 2>::kDqSets == 2; }

// The kernel body for a launch whose rows take TT x terms (see Cfg8).
template <int MP, int PACK, int TT>
__device__ __forceinline__ void coarse_tc8_body(const CUtensorMap &tm_packed, const CUtensorMap &tm_x,
                                                const Tc8Params &prm, int nstage,
                                                uint8_t *smem_raw)
{
    using C = Cfg8<MP, PACK, TT>;
    constexpr int BITS = PACK == kPackHalf4 ? 4 : 2;
    constexpr int G = C::G, kGPP = C::kGPP;
    constexpr int kBoxes = C::kPkBoxes;
    constexpr int N = C::N, T = C::T, K = C::K, kU = C::kU, kPP = C::kPP;
    constexpr int kGU = kPP * kGPP;         // weight groups (accumulators) of a unit
    using R = Roles<two_sets<MP, PACK>()>;
    constexpr int kDqSets = C::kDqSets; // dequant warp sets (split each span's planes)
    static_assert(kDqSets == 1 || two_sets<MP, PACK>(), "a second dequant set needs its warps");
    constexpr int kWarpEp0 = R::kEp0;
    constexpr uint32_t kSlotCols = C::kSlotCols, kACols = C::kACols;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = prm.H / 512, NGt = prm.H / G;
    const uint32_t sz_bytes = static_cast<uint32_t>(kTileRows) * NGt * 2; // S (or ZS) of a tile

    // ---- shared memory ------------------------------------------------------------------
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t *const stages = smem_raw + pad;                                   // nstage x kStage
    uint8_t *const szbuf = stages + static_cast<size_t>(nstage) * C::kStage; // [2][S, ZS] tiles
    float *const red = reinterpret_cast<float *>(szbuf + 4 * static_cast<size_t>(sz_bytes));
    constexpr int kRedHalf = MP * 2 * kRedPitch; // floats of one epilogue half's tile values
    float *const xs_s = red + 2 * kRedHalf;                                   // [NGt][MP]
    float *const inv_s = xs_s + NGt * MP;                                     // [MP] 2^-e
    float *const tw_s = inv_s + MP;                                           // [2][MP] w2, w3
    uint64_t *const bars = reinterpret_cast<uint64_t *>(tw_s + 2 * MP);
    uint64_t *const full = bars;              // [nstage] TMA -> dequant, MMA
    uint64_t *const empty = full + nstage;    // [nstage] dequant (4 warps) + issuers -> TMA
    uint64_t *const a_full = empty + nstage;  // [K]      dequant (4 warps) -> MMA, per unit
    uint64_t *const d_full = a_full + K;      // [K]      MMA -> epilogue + dequant, per unit
    uint64_t *const d_empty = d_full + K;     // [K]      epilogue -> MMA, per unit
    uint64_t *const fin = d_empty + K;        // [4]      MMA drain before teardown
    uint64_t *const red_full = fin + kIssuers; // [1]     epilogue (8 warps) -> selection
    uint64_t *const red_free = red_full + 1;  // [1]      selection -> epilogue: `red` free
    uint64_t *const sz_full = red_free + 1;   // [2]      bulk copy -> epilogue: S, ZS of a tile
    uint64_t *const sz_empty = sz_full + 2;   // [2]      epilogue (8 warps) -> bulk copy
    uint64_t *const xs_full = sz_empty + 2;   // [1]      epilogue (8 warps): xs, 2^-e, weights
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(xs_full + 1);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_packed);
        prefetch_tensormap(&tm_x);
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kDqSets * kDqWarps + kIssuers); // dequant warps, issuers
        }
        for (int i = 0; i < K; ++i) {
            mbar_init(&a_full[i], kDqSets * kDqWarps);
            mbar_init(&d_full[i], kPP);     // one commit per plane of the unit
            mbar_init(&d_empty[i], kU == 1 ? 8 : 4); // the epilogue warps reading the unit
        }
        for (int i = 0; i < kIssuers; ++i) mbar_init(&fin[i], 1);
        mbar_init(red_full, kEpWarps);
        mbar_init(red_free, 2); // both selection warps
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sz_full[i], 1);
            mbar_init(&sz_empty[i], kEpWarps);
        }
        mbar_init(xs_full, kEpWarps);
        fence_barrier_init();
    }
    // (the group sums, 2^-e and the term weights are read by the epilogue only: its warps load
    // them, so that their global-memory latency stays off the start of the weight stream)
    if (warp == kWarpTma) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int first_tile = blockIdx.x, tile_step = gridDim.x;
    bool failed = false;

    // Register budgets per warpgroup, set at the top of each role's branch (every warp of a
    // warpgroup sets the same value): the TMA / issuer and the issuer / selection / idle
    // warpgroups drop to kRegsLight, the epilogue's two rise to kRegsEp.
    if (warp == kWarpTma) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsLight));
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            uint32_t st = 0, ph = 0, it = 0; // stage ring position and its phase parity
            for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step, ++it) {
                // the tile's S and ZS rows (contiguous in memory) into buffer it % 2, free once
                // the epilogue finished tile it - 2; a partial last tile is read from global
                // memory by the epilogue instead (an arrival without data keeps the phases)
                const uint32_t b = it & 1u;
                if (!mbar_wait_bounded(&sz_empty[b], ((it >> 1) & 1u) ^ 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                if ((tile + 1) * kTileRows <= prm.V) {
                    uint8_t *const sz = szbuf + static_cast<size_t>(b) * 2 * sz_bytes;
                    const size_t off = static_cast<size_t>(tile) * kTileRows * NGt;
                    mbar_arrive_expect_tx(&sz_full[b], 2 * sz_bytes);
                    bulk_load(sz, prm.S + off, sz_bytes, &sz_full[b]);
                    bulk_load(sz + sz_bytes, prm.ZS + off, sz_bytes, &sz_full[b]);
                } else {
                    mbar_arrive(&sz_full[b]);
                }
                for (int span = 0; span < NG; ++span) {
                    if (!mbar_wait_bounded(&empty[st], ph ^ 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    uint8_t *const stage = stages + static_cast<size_t>(st) * C::kStage;
                    mbar_arrive_expect_tx(&full[st], C::kStage);
#pragma unroll
                    for (int bx = 0; bx < kBoxes; ++bx)
                        tma_load_2d_hint(stage + bx * kPkBytes, &tm_packed,
                                         (kBoxes * span + bx) * kSpanBytes, tile * kTileRows,
                                         &full[st], policy);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d(stage + kBoxes * kPkBytes + q * (N * 128), &tm_x,
                                    plane_group<PACK>(q, span, NG) * kGroup, 0, &full[st]);
                    if (++st == static_cast<uint32_t>(nstage)) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (R::issuer_plane(warp) >= 0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsLight));
        // ---------------- MMA issuers: one warp per plane, every unit holding that plane ------
        // The whole warp runs the loop (warp-uniform operands); one elected lane issues.
        constexpr uint32_t idesc = make_idesc_f8(N);
        const int plane = R::issuer_plane(warp);
        const int u = plane / kPP, g = plane % kPP; // the plane's unit in a span, and its place
        uint32_t st = 0, ph = 0, q = u;             // stage ring position, parity; unit index
        for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step) {
            for (int span = 0; span < NG && !failed; ++span, q += kU) {
                const uint32_t slot = q % K, use = q / K;
                if (!warp_wait(&full[st], ph, prm.timeout_flag) ||
                    !warp_wait(&a_full[slot], use & 1u, prm.timeout_flag) ||
                    !warp_wait(&d_empty[slot], (use & 1u) ^ 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_tmem = tmem + slot * kSlotCols;
                const uint32_t d_tmem = a_tmem + kACols;
                // the descriptor's address field counts 16-byte units
                const uint64_t qdesc =
                    sw128_desc(smem_u32(stages + static_cast<size_t>(st) * C::kStage +
                                        kBoxes * kPkBytes)) +
                    static_cast<uint64_t>(plane * (N * 128) / 16);
                // K = 32 per MMA: 128 / G groups of the plane, 4 / (128 / G) MMAs each into
                // the group's own accumulator
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    mma_ts_f8_elect(d_tmem + (g * kGPP + i / (4 / kGPP)) * N, a_tmem + g * 32 + i * 8,
                                    qdesc + static_cast<uint64_t>(i * 2), idesc,
                                    (i % (4 / kGPP)) ? 1u : 0u);
                mma_commit_elect(&d_full[slot]);
                mma_commit_elect(&empty[st]);
                if (++st == static_cast<uint32_t>(nstage)) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
        mma_commit_elect(&fin[plane]);
        warp_wait(&fin[plane], 0, prm.timeout_flag);
    } else if (warp >= kWarpDq0 && warp < kWarpDq0 + kDqWarps * kDqSets) {
        // ---------------- dequant: one TMEM lane (= tile row) per thread ------------------------
        // With one unit per span two sets of four warps share every span.  2-bit layouts: set c
        // writes k half c (64 k) of every plane and reads only that half of the packed row; the
        // 4-bit head: set c writes planes 2c, 2c + 1, the two nibbles of packed box c.  A single
        // set writes every plane.
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        auto run = [&](auto set_c) {
            constexpr int SET = decltype(set_c)::value;
            constexpr bool kSplitK = kDqSets == 2 && BITS == 2;
            constexpr bool kSplitP = kDqSets == 2 && BITS == 4;
            constexpr int hf0 = kSplitK ? SET : 0, hf1 = kSplitK ? SET + 1 : 2;
            constexpr int pp0 = kSplitP ? 2 * SET : 0, pp1 = kSplitP ? 2 * SET + 2 : kPP;
            uint32_t s = 0, st = 0, ph = 0; // span count, stage ring position and parity
            for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step) {
                for (int span = 0; span < NG; ++span, ++s) {
                    if (!warp_wait(&full[st], ph, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    const uint32_t pk =
                        smem_u32(stages + static_cast<size_t>(st) * C::kStage) + row * kSpanBytes;
                    uint32_t w[32];
                    // this thread's row of packed box bx (128-byte swizzle): the 16-byte chunks
                    // holding this warp's k halves (chunk c is words 4c .. 4c + 3)
                    auto load_box = [&](int bx) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int hc = PACK == kPackContig2 ? (c & 1) : (c >> 2);
                            if (hc < hf0 || hc >= hf1) continue;
                            const uint32_t addr = pk + bx * kPkBytes + ((c ^ (row & 7)) << 4);
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]),
                                           "=r"(w[4 * c + 3])
                                         : "r"(addr));
                        }
                    };
                    if constexpr (BITS == 2) {
                        // every plane of this warp's share is in these words: the stage goes back
                        load_box(0);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[st]);
                    }
                    // the span's units: their planes into the A buffer of slot q % K, free once
                    // that slot's previous unit (q - K) has been accumulated
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const uint32_t q = kU * s + u, slot = q % K, use = q / K;
                        if (use > 0 &&
                            !warp_wait(&d_full[slot], (use - 1) & 1u, prm.timeout_flag)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t abuf = tmem + lane_base + slot * kSlotCols;
                        // this warp's planes of the unit, two at a time, in halves of 16 columns
                        // (64 k; a tcgen05.st reads its registers at issue: r0 and r1 are free
                        // again after it)
#pragma unroll
                        for (int pp = pp0; pp < pp1; pp += 2) {
                            const int plane = kPP * u + pp;
                            // planes 2 bx, 2 bx + 1 of the 4-bit head: the nibbles of box bx
                            if constexpr (BITS == 4) load_box(plane >> 1);
#pragma unroll
                            for (int hf = hf0; hf < hf1; ++hf) {
                                uint32_t r0[16], r1[16];
                                if constexpr (BITS == 4) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        r0[i] = deq_nib_lo(w[16 * hf + i]);
                                        r1[i] = deq_nib_hi(w[16 * hf + i]);
                                    }
                                } else if constexpr (PACK == kPackContig2) {
                                    // planes p, p + 1 are words 8p .. 8p + 15; half hf of plane
                                    // p is words 8p + 4 hf ..
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        uint32_t o0[4], o1[4];
                                        deq_c4(w[8 * plane + 4 * hf + i], o0);
                                        deq_c4(w[8 * plane + 8 + 4 * hf + i], o1);
#pragma unroll
                                        for (int b = 0; b < 4; ++b) {
                                            r0[4 * i + b] = o0[b];
                                            r1[4 * i + b] = o1[b];
                                        }
                                    }
                                } else if (plane == 0) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        r0[i] = deq4_e4m3<0>(w[16 * hf + i]);
                                        r1[i] = deq4_e4m3<1>(w[16 * hf + i]);
                                    }
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        r0[i] = deq4_e4m3<2>(w[16 * hf + i]);
                                        r1[i] = deq4_e4m3<3>(w[16 * hf + i]);
                                    }
                                }
                                tmem_st_x16(abuf + pp * 32 + 16 * hf, r0);
                                tmem_st_x16(abuf + pp * 32 + 32 + 16 * hf, r1);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&a_full[slot]);
                    }
                    if (failed) break;
                    if constexpr (BITS == 4) {
                        // this warp's boxes have been read into registers
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[st]);
                    }
                    if (++st == static_cast<uint32_t>(nstage)) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
        };
        if constexpr (kDqSets == 2) {
            if ((warp - kWarpDq0) >> 2) run(std::integral_constant<int, 1>{});
            else run(std::integral_constant<int, 0>{});
        } else {
            run(std::integral_constant<int, 0>{});
        }
    } else if (warp >= kWarpEp0 && warp < kWarpEp0 + kEpWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R::kRegsEp));
        // ---------------- epilogue: two halves of four warps, each two groups of every span ---
        {
            // the batch rows' group sums (scaled units), 2^-e and term weights, shared by the
            // eight epilogue warps (written by all of them, read after every one has arrived)
            const int et = static_cast<int>(threadIdx.x) - 32 * kWarpEp0;
            const float *const xsrc = T == 3 ? prm.xs3 : prm.xs2;
            for (int i = et; i < NGt * MP; i += 32 * kEpWarps) {
                const int g = i / MP, m = i - g * MP;
                xs_s[i] = xsrc[static_cast<long long>(m) * NGt + g];
            }
            for (int i = et; i < MP; i += 32 * kEpWarps) {
                inv_s[i] = prm.row_f[i];
                tw_s[i] = prm.row_f[kTc8MaxMP + i];
                tw_s[MP + i] = prm.row_f[2 * kTc8MaxMP + i];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xs_full);
            if (!warp_wait(xs_full, 0, prm.timeout_flag)) failed = true;
        }
        const int h = (warp - kWarpEp0) >> 2; // planes 2h, 2h + 1
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        constexpr int NGH = 2 * kGPP; // groups of a half in one span
        constexpr int CH = MP / 16;   // 16-column chunks of one term of one group
        uint32_t t = 0, it = 0;
        for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step, ++it) {
            const int grow = tile * kTileRows + row;
            const bool row_ok = grow < prm.V;
            const bool full_tile = (tile + 1) * kTileRows <= prm.V;
            const uint32_t b = it & 1u;
            if (!warp_wait(&sz_full[b], (it >> 1) & 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            const uint16_t *const sS = reinterpret_cast<const uint16_t *>(
                szbuf + static_cast<size_t>(b) * 2 * sz_bytes) + row * NGt;
            const uint16_t *const sZ = sS + sz_bytes / 2;
            const uint16_t *const gS = prm.S + static_cast<long long>(row_ok ? grow : 0) * NGt;
            const uint16_t *const gZ = prm.ZS + static_cast<long long>(row_ok ? grow : 0) * NGt;
            // the row's coarse values for batch rows 2i, 2i + 1 (packed fp32 pairs: one FFMA2
            // folds two rows)
            float2 acc2[MP / 2];
#pragma unroll
            for (int i = 0; i < MP / 2; ++i) acc2[i] = make_float2(0.f, 0.f);
            for (int span = 0; span < NG; ++span, t += 4) {
                // this half's groups: planes 2h, 2h+1, kGPP groups each
                float s2[NGH], sz[NGH];
#pragma unroll
                for (int gl = 0; gl < NGH; ++gl) {
                    const int plane = 2 * h + gl / kGPP;
                    const int gi = plane_group<PACK>(plane, span, NG) * kGPP + gl % kGPP;
                    uint16_t sb = 0, zb = 0;
                    if (full_tile) {
                        sb = sS[gi];
                        zb = sZ[gi];
                    } else if (row_ok) {
                        sb = __ldg(gS + gi);
                        zb = __ldg(gZ + gi);
                    }
                    const float sv = bf16_bits_to_f32(sb), zv = bf16_bits_to_f32(zb);
                    // (S / B) sum x v with the MMA's sum of x v 2^-9 (quarter split, B = 4: odd
                    // planes carry 4 v 2^-9, even planes v 2^-9; contiguous-4, B = 4: every
                    // plane v 2^-9; 4 bits, B = 16: v 2^-9)
                    const bool four_v = PACK != kPackHalf4 && PACK != kPackContig2 && (plane & 1);
                    s2[gl] = (BITS == 4 ? 32.0f : (four_v ? 32.0f : 128.0f)) * sv;
                    sz[gl] = sv - zv;
                }
                // the unit holding this half's two groups (planes 2h, 2h+1) of the span
                const uint32_t q = kU * (t / 4) + (kU == 1 ? 0 : h), slot = q % K, use = q / K;
                if (!warp_wait(&d_full[slot], use & 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                // the half's first accumulator within the unit
                const uint32_t dcol = tmem + lane_base + slot * kSlotCols + kACols +
                                      (kU == 1 ? 2 * h * kGPP : 0) * N;
                // the half's NGH * CH chunks, one per tcgen05 wait (T * 16 registers, as packed
                // pairs of batch rows)
#pragma unroll
                for (int k = 0; k < NGH * CH; ++k) {
                    const int gl = k / CH, c = k % CH;
                    uint64_t u[T][8];
                    if constexpr (T == 3) tmem_ld_terms3(dcol + gl * N + c * 16, MP, u);
                    else tmem_ld_terms2(dcol + gl * N + c * 16, MP, u);
                    if (k == NGH * CH - 1) {
                        // every partial of the unit is in registers: the slot goes back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_empty[slot]);
                    }
                    const int gi = plane_group<PACK>(2 * h + gl / kGPP, span, NG) * kGPP + gl % kGPP;
                    const float4 *xg = reinterpret_cast<const float4 *>(xs_s + gi * MP);
                    const float2 s2v = make_float2(s2[gl], s2[gl]), szv = make_float2(sz[gl], sz[gl]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 x4 = xg[c * 4 + j];
                        const float4 a4 = reinterpret_cast<const float4 *>(tw_s)[c * 4 + j];
                        const float2 xv[2] = {make_float2(x4.x, x4.y), make_float2(x4.z, x4.w)};
                        const float2 w2[2] = {make_float2(a4.x, a4.y), make_float2(a4.z, a4.w)};
                        float2 w3[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                        if constexpr (T == 3) {
                            const float4 b4 = reinterpret_cast<const float4 *>(tw_s + MP)[c * 4 + j];
                            w3[0] = make_float2(b4.x, b4.y);
                            w3[1] = make_float2(b4.z, b4.w);
                        }
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            // batch rows m, m + 1: the terms weighted by their powers of two
                            // (exact), then the scale and zero fold, two rows per instruction
                            const int e = 2 * j + i; // pair within the chunk
                            float2 p = __ffma2_rn(w2[i], pair_f2(u[1][e]), pair_f2(u[0][e]));
                            if constexpr (T == 3) p = __ffma2_rn(w3[i], pair_f2(u[2][e]), p);
                            const int mp = c * 8 + e;
                            acc2[mp] = __ffma2_rn(s2v, p, __ffma2_rn(szv, xv[i], acc2[mp]));
                        }
                    }
                }
            }
            if (failed) break;
            // every read of the tile's S / ZS buffer is done
            __syncwarp();
            if (lane == 0) mbar_arrive(&sz_empty[b]);
            // the selection warp is done with the previous tile's values
            if (!warp_wait(red_free, (it & 1u) ^ 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            float *const rh = red + h * kRedHalf + (row >> 6) * kRedPitch + (row & 63);
#pragma unroll
            for (int i = 0; i < MP / 2; ++i) {
                rh[4 * i * kRedPitch] = row_ok ? acc2[i].x * inv_s[2 * i] : -INFINITY;
                rh[(4 * i + 2) * kRedPitch] = row_ok ? acc2[i].y * inv_s[2 * i + 1] : -INFINITY;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_full);
        }
    } else if (warp == R::kSel0 || warp == R::kSel1) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsLight));
        // ---------------- block top-KCAND: pair = (batch column m, block b of the tile) ------
        // the tile's coarse values are the sums of the two epilogue halves (both -inf past V)
        const int npairs = 2 * prm.mrows;
        const int sw = warp == R::kSel0 ? 0 : 1;
        uint32_t it = 0;
        for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step, ++it) {
            if (!warp_wait(red_full, it & 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            if (prm.kcand <= 8) {
                // two lanes per pair: selection warp sw takes pairs 16 sw .. 16 sw + 15 of
                // every 32
                for (int p0 = 0; p0 < npairs; p0 += 32) {
                    const int pidx = p0 + 16 * sw + (lane >> 1);
                    const int m = pidx >> 1, blk = tile * 2 + (pidx & 1);
                    const bool live = pidx < npairs && static_cast<long long>(blk) * kBlockN < prm.V;
                    const long long off = static_cast<long long>(prm.m0 + m) * prm.ncand +
                                          static_cast<long long>(blk) * prm.kcand;
                    float *const cdbg = (prm.coarse && live)
                                            ? prm.coarse + static_cast<long long>(prm.m0 + m) * prm.V
                                            : nullptr;
                    const int pp = live ? pidx : 0;
                    select_pair2(live, red + pp * kRedPitch, red + kRedHalf + pp * kRedPitch,
                                 blk * kBlockN, prm.V, prm.kcand, live ? prm.cand_val + off : nullptr,
                                 live ? prm.cand_idx + off : nullptr, cdbg, lane);
                }
            } else if (sw == 0) {
                // larger KCAND: four pairs at a time, one warp-wide round per entry
                for (int p0 = 0; p0 < npairs; p0 += 4) {
                    uint32_t k0[4], k1[4];
                    int base_row[4];
                    float *oval[4];
                    int32_t *oidx[4];
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        const int pidx = p0 + bb;
                        const int m = pidx >> 1, blk = tile * 2 + (pidx & 1);
                        const bool live = pidx < npairs &&
                                          static_cast<long long>(blk) * kBlockN < prm.V;
                        const int g0 = blk * kBlockN + lane;
                        const float *pv = red + (live ? pidx : 0) * kRedPitch;
                        const float c0 = pv[lane] + pv[kRedHalf + lane];
                        const float c1 = pv[lane + 32] + pv[kRedHalf + lane + 32];
                        k0[bb] = (live && g0 < prm.V) ? f32_order_key(c0) : 0u;
                        k1[bb] = (live && g0 + 32 < prm.V) ? f32_order_key(c1) : 0u;
                        if (prm.coarse && live) {
                            float *const cd = prm.coarse + static_cast<long long>(prm.m0 + m) * prm.V;
                            if (g0 < prm.V) cd[g0] = c0;
                            if (g0 + 32 < prm.V) cd[g0 + 32] = c1;
                        }
                        base_row[bb] = blk * kBlockN;
                        const long long off = static_cast<long long>(prm.m0 + m) * prm.ncand +
                                              static_cast<long long>(blk) * prm.kcand;
                        oval[bb] = live ? prm.cand_val + off : nullptr;
                        oidx[bb] = live ? prm.cand_idx + off : nullptr;
                    }
                    select_pairs<4>(k0, k1, base_row, oval, oidx, prm.kcand, lane);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_free);
        }
    } else if (warp == R::kWarps - 1) {
        // the idle warp that completes the last warpgroup gives its registers up too
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsLight));
    }

    // ---- teardown: every role is done (or gave up); release tensor memory ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the selection may be scheduled (it waits for this grid before it reads the candidates)
    pdl_trigger();
    if (warp == kWarpTma) tmem_dealloc(tmem, kTmemCols);
}

// One launch covers both term counts: the launch's count is the most any of its rows needs.
template <int MP, int PACK>
__global__ void __launch_bounds__(Roles<two_sets<MP, PACK>()>::kThreads, 1)
    coarse_tc8_kernel(const __grid_constant__ CUtensorMap tm_packed,
                      const __grid_constant__ CUtensorMap tm_x2,
                      const __grid_constant__ CUtensorMap tm_x3, const Tc8Params prm)
{
    extern __shared__ uint8_t smem_raw[];
    // before the x staging is known to be done: the weights are the caller's, so the first
    // two spans of this CTA's first tile and the tile's S / ZS rows can already move to L2
    if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < prm.ntiles) {
        constexpr int kBoxes = PACK == kPackHalf4 ? 2 : 1;
        const int tile = blockIdx.x;
        prefetch_tensormap(&tm_packed);
#pragma unroll
        for (int b = 0; b < 2 * kBoxes; ++b) prefetch_l2_box(&tm_packed, b * kSpanBytes, tile * kTileRows);
        const int NGt = prm.H / (PACK == kPackG64 ? 64 : 128);
        if ((tile + 1) * kTileRows <= prm.V) {
            const size_t off = static_cast<size_t>(tile) * kTileRows * NGt;
            const uint32_t bytes = static_cast<uint32_t>(kTileRows) * NGt * 2;
            prefetch_l2_bytes(prm.S + off, bytes);
            prefetch_l2_bytes(prm.ZS + off, bytes);
        }
    }
    // launched while the x staging may still run: everything below reads its output
    pdl_wait();
    int need = 2;
    for (int m = 0; m < MP; ++m) need = max(need, prm.row_terms[m]);
    if (need == 3) coarse_tc8_body<MP, PACK, 3>(tm_packed, tm_x3, prm, prm.nstage3, smem_raw);
    else coarse_tc8_body<MP, PACK, 2>(tm_packed, tm_x2, prm, prm.nstage2, smem_raw);
}

// Dynamic shared memory besides the stages: alignment slack, the double-buffered S/ZS tile
// copies, the two epilogue halves' tile values, xs, 2^-e and the term weights, barriers.
size_t tc8_fixed_smem(int MP, int H, int G)
{
    const int NGt = H / G;
    return 1024 + 4 * static_cast<size_t>(kTileRows) * NGt * 2 +
           2 * static_cast<size_t>(MP) * 2 * kRedPitch * 4 + static_cast<size_t>(NGt) * MP * 4 +
           3 * MP * 4 + 64 * 8 + 32;
}

// Stage count of a body: as many as fit (at most 6).
template <int MP, int PACK, int TT>
int tc8_stages(int H)
{
    using C = Cfg8<MP, PACK, TT>;
    const size_t fixed = tc8_fixed_smem(MP, H, C::G);
    long long n = (kSmemLimit8 - static_cast<long long>(fixed)) / C::kStage;
    if (n > 6) n = 6;
    return static_cast<int>(n);
}

template <int MP, int PACK>
cudaError_t launch_cfg(const CUtensorMap &tm_packed, const uint8_t *xt8_chunk,
                       const Tc8Params &base, cudaStream_t stream)
{
    // the staged x of the launch: [3 MP rows, H] bytes; a box is a plane's 128 k of the
    // first T terms (T MP rows)
    CUtensorMap tm_x[2];
    for (int t = 0; t < 2; ++t) {
        CUresult r = encode_tensor_map_2d(&tm_x[t], CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                          const_cast<uint8_t *>(xt8_chunk), base.H,
                                          static_cast<uint64_t>(kTc8Terms) * MP, base.H, 128,
                                          (2 + t) * MP, CU_TENSOR_MAP_SWIZZLE_128B);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    const int n2 = tc8_stages<MP, PACK, 2>(base.H), n3 = tc8_stages<MP, PACK, 3>(base.H);
    if (n2 < 2 || n3 < 2) return cudaErrorInvalidConfiguration;
    const size_t s2 = tc8_fixed_smem(MP, base.H, Cfg8<MP, PACK, 2>::G) +
                      static_cast<size_t>(n2) * Cfg8<MP, PACK, 2>::kStage;
    const size_t s3 = tc8_fixed_smem(MP, base.H, Cfg8<MP, PACK, 3>::G) +
                      static_cast<size_t>(n3) * Cfg8<MP, PACK, 3>::kStage;
    const size_t smem = s2 > s3 ? s2 : s3;
    // the shared-memory limit is a per-device attribute: raised once on every device
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        // the warpgroups' register budgets (setmaxnreg) add up to the launch's registers a
        // thread times its threads: a kernel built with another count could wait forever for
        // registers in setmaxnreg.inc, so it is not launched
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, coarse_tc8_kernel<MP, PACK>);
        if (err != cudaSuccess) return err;
        if (fa.numRegs != Roles<two_sets<MP, PACK>()>::kRegsLaunch)
            return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(coarse_tc8_kernel<MP, PACK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit8);
    });
    if (e != cudaSuccess) return e;
    Tc8Params prm = base;
    prm.nstage2 = n2;
    prm.nstage3 = n3;
    const int sms = device_sm_count();
    const int grid = prm.ntiles < sms ? prm.ntiles : sms;
    constexpr int kThreads = Roles<two_sets<MP, PACK>()>::kThreads;
    return launch_pdl(coarse_tc8_kernel<MP, PACK>, dim3(grid), dim3(kThreads), smem, stream,
                      tm_packed, tm_x[0], tm_x[1], prm);
}

template <int PACK>
bool fits(int MP, int H)
{
    if (MP == 16) return tc8_stages<16, PACK, 2>(H) >= 2 && tc8_stages<16, PACK, 3>(H) >= 2;
    if constexpr (PACK == kPackG64) return false; // groups of 64: 16-row launches only
    else return tc8_stages<32, PACK, 2>(H) >= 2 && tc8_stages<32, PACK, 3>(H) >= 2;
}

} // namespace

int tc8_max_rows(int pack, int H)
{
    // groups of 64 need two accumulators per plane; the 4-bit head's 32 KB packed boxes leave
    // no room for two stages of 32 rows in three terms; 2-bit rows wider than a 32-row launch's
    // shared memory holds run in 16-row launches too
    if (pack == kPackG64 || pack == kPackHalf4) return 16;
    return fits<kPackQuarter2>(32, H) && fits<kPackContig2>(32, H) ? 32 : 16;
}

int tc8_chunks(int M, int pack, int H)
{
    const int r = tc8_max_rows(pack, H);
    return (M + r - 1) / r;
}

Tc8Chunk tc8_chunk(int M, int c, int pack, int H)
{
    const int r = tc8_max_rows(pack, H);
    Tc8Chunk k;
    k.m0 = c * r;
    k.rows = M - k.m0 < r ? M - k.m0 : r;
    k.MP = k.rows <= 16 ? 16 : 32;
    // launches before c are full (r rows, MP = r)
    k.x_off = static_cast<size_t>(c) * kTc8Terms * r * H;
    return k;
}

size_t tc8_x_bytes(int M, int H)
{
    size_t most = 0;
    const int packs[2] = {kPackQuarter2, kPackHalf4};
    for (int pack : packs) {
        const int n = tc8_chunks(M, pack, H);
        const Tc8Chunk last = tc8_chunk(M, n - 1, pack, H);
        const size_t b = last.x_off + static_cast<size_t>(kTc8Terms) * last.MP * H;
        if (b > most) most = b;
    }
    return most;
}

bool tc8_supported(int M, int H, int bits, int group)
{
    // the x staging keeps a row in registers: H <= 16384
    if (M < 1 || M > kMaxM || H % 512 != 0 || H > 16384) return false;
    if (bits != 2 && bits != 4) return false;
    // groups of 64 need two accumulators per plane: only the 16-row launch
    if (group != 128 && (group != 64 || bits != 2 || M > 16)) return false;
    const int pack = bits == 4 ? kPackHalf4 : (group == 64 ? kPackG64 : kPackQuarter2);
    for (int c = 0; c < tc8_chunks(M, pack, H); ++c) {
        const int MP = tc8_chunk(M, c, pack, H).MP;
        bool ok;
        if (pack == kPackHalf4) ok = fits<kPackHalf4>(MP, H);
        else if (pack == kPackG64) ok = fits<kPackG64>(MP, H);
        else ok = fits<kPackQuarter2>(MP, H) && fits<kPackContig2>(MP, H);
        if (!ok) return false;
    }
    return true;
}

cudaError_t launch_coarse_tc8(const CoarseArgs &a, const Tc8Workspace &w, cudaStream_t stream)
{
    CUtensorMap tm_packed;
    const int bits = a.pack == kPackHalf4 ? 4 : 2;
    const int row_bytes = a.H * bits / 8; // packed bytes per row
    CUresult r = encode_tensor_map_2d(&tm_packed, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                      const_cast<uint8_t *>(a.packed), row_bytes, a.V, row_bytes,
                                      kSpanBytes, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (!tc8_supported(a.M, a.H, bits, a.pack == kPackG64 ? 64 : 128))
        return cudaErrorInvalidConfiguration;
    Tc8Params base;
    base.S = a.S;
    base.ZS = a.ZS;
    base.V = a.V;
    base.H = a.H;
    base.kcand = a.kcand;
    base.ntiles = (a.V + kTileRows - 1) / kTileRows;
    base.ncand = static_cast<long long>((a.V + kBlockN - 1) / kBlockN) * a.kcand;
    base.cand_val = a.cand_val;
    base.cand_idx = a.cand_idx;
    base.coarse = a.coarse;
    base.timeout_flag = a.timeout_flag;
    base.nstage2 = base.nstage3 = 2;
    for (int c = 0; c < tc8_chunks(a.M, a.pack, a.H); ++c) {
        const Tc8Chunk k = tc8_chunk(a.M, c, a.pack, a.H);
        const float *const small = w.small + static_cast<size_t>(c) * tc8_small_floats(a.H);
        base.m0 = k.m0;
        base.mrows = k.rows;
        base.xs2 = small;
        base.xs3 = small + static_cast<size_t>(kTc8MaxMP) * (a.H / 64);
        base.row_f = small + 2 * static_cast<size_t>(kTc8MaxMP) * (a.H / 64);
        base.row_terms = reinterpret_cast<const int *>(base.row_f + 3 * kTc8MaxMP);
        const uint8_t *xt = w.xt8 + k.x_off;
        cudaError_t e;
        if (a.pack == kPackHalf4) {
            if (k.MP == 16) e = launch_cfg<16, kPackHalf4>(tm_packed, xt, base, stream);
            else e = launch_cfg<32, kPackHalf4>(tm_packed, xt, base, stream);
        } else if (a.pack == kPackG64) {
            e = launch_cfg<16, kPackG64>(tm_packed, xt, base, stream); // M <= 16 (checked)
        } else if (a.pack == kPackContig2) {
            if (k.MP == 16) e = launch_cfg<16, kPackContig2>(tm_packed, xt, base, stream);
            else e = launch_cfg<32, kPackContig2>(tm_packed, xt, base, stream);
        } else {
            if (k.MP == 16) e = launch_cfg<16, kPackQuarter2>(tm_packed, xt, base, stream);
            else e = launch_cfg<32, kPackQuarter2>(tm_packed, xt, base, stream);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace dh
