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
//     T e4m3 terms, x 2^e ~ t1 + w2 t2 + w3 t3, each term the rounded residual of the ones
//     before at its own power-of-two scale (per row weights w2, w3; dh_prep.cu); the terms are
//     stacked along the MMA's N dimension (rows t MP + m) and recombined in fp32 in the
//     epilogue.  Two terms represent every element of an ordinary row exactly, the third
//     covers rows with a wide dynamic range; the staging kernel measures the two-term error of
//     every row and a launch uses the third term when any row needs it;
//   * per group g (128 consecutive k of one plane q), with p = sum_t w_t D_t the recombined
//     partial, sum_k x_k v_k = 2^9 p / f (f = 1 for even q, 4 for odd q), and the page's
//     group term S sum_k x_k (1 + v_k/4) - ZS xs = (S/4) sum_k x_k v_k + (S - ZS) xs, so
//         c[m, n] = 2^-e * sum_g ( (2^7/f) S[n,g] p + (S[n,g] - ZS[n,g]) xs'[m,g] )
//     with xs' the group sums of the represented x (in the scaled units): the scale and zero
//     are applied to the fp32 partial of every group, never to the weight.
//
// The unit of MMA work is one plane of one span (128 k of 128 vocabulary rows: one weight
// group, two for groups of 64): four tcgen05.mma of K = 32 into the unit's accumulator, then
// one commit to the unit's tensor-memory slot (accumulator ready, A buffer free) and one to its
// x stage.  A thread issuing tcgen05.mma is held for ~100 cycles per instruction whatever the
// shape (~700 cycles per unit with its waits and commits), so the units are spread over I
// issuer warps: unit q goes to issuer q mod I, tensor-memory slot q mod K and x stage q mod nx,
// with K and nx multiples of I.  Every slot and x stage then belongs to one issuer, which
// waits on the phases of its barriers strictly in order (a parity wait is only exact when the
// phase before the awaited one has completed).
//
// Roles (28 warps, one CTA per SM, persistent over 128-row vocabulary tiles taken round-robin):
//   warp 0        TMA: per span one [128 rows x 128 B] box of packed codes (two for the 4-bit
//                 head) into a ring of packed stages; per tile a bulk copy of the tile's S and
//                 ZS rows (contiguous in memory) into a double-buffered shared copy
//   warp 1        TMA: per unit the unit's 128 k of the staged x terms ([T MP rows x 128 B],
//                 128-byte swizzle) into a ring of x stages
//   warp 2        block top-KCAND of the previous tile (overlaps the current one)
//   warps 3..3+I  MMA issuers (lane 0)
//   warps 8-11    dequant: one TMEM lane (= one vocabulary row) per thread; reads the span's
//                 packed bytes once, then writes each plane into its unit's A buffer
//                 (tcgen05.st) as soon as that slot's previous unit has completed
//   warps 12-27   epilogue, four sets of four warps (one per TMEM lane quarter): set cp folds
//                 every unit for batch columns [cp MP/4, (cp + 1) MP/4) -- tcgen05.ld of the
//                 terms, recombination, scale and zero fold into fp32 registers -- and at the
//                 tile end writes those columns of the tile's coarse values
// Every handoff is an mbarrier; every wait is bounded.
//
// The 4-bit head (BITS = 4, half split, bias 16; _quantize_head_now's 4-bit variant) runs the
// same pipeline: a nibble masked in place is the exact e4m3 weight v 2^-9 (v in 0..15), and two
// 128-byte boxes of a row (packed bytes 256 span ..) carry four groups -- low and high nibbles
// of each box -- so one span is again four planes of 128 k, with NG = H / 512 spans per row.
// The fold becomes (2^9 / 16) S p = 32 S p for every plane.
#include "dh_common.cuh"
#include "dh_internal.h"
#include "dh_tcgen05.cuh"

#include <climits>

namespace dh {

namespace {

constexpr int kTileRows = 128;
constexpr int kTmemCols = 512;
constexpr int kPkBytes = kTileRows * kSpanBytes; // 16 KB packed box per span
constexpr int kSmemLimit8 = 232448;
// The tile's coarse values for the selection warp: one 64-value block per (batch column,
// block) pair, pairs kRedPitch floats apart (16-byte aligned, bank-conflict free per lane).
constexpr int kRedPitch = 68;

// warp roles
constexpr int kWarpPk = 0, kWarpX = 1, kWarpSel = 2, kWarpIss0 = 3, kMaxIssuers = 5;
constexpr int kWarpDq0 = 8, kDqWarps = 4;
constexpr int kWarpEp0 = 12, kEpWarps = 16;
constexpr int kWarps = kWarpEp0 + kEpWarps; // 28
constexpr int kThreads = kWarps * 32;       // 896

template <int MP, int PACK> struct Cfg8 {
    static constexpr int kBoxes = PACK == kPackHalf4 ? 2 : 1; // packed boxes per span
    static constexpr int G = PACK == kPackG64 ? 64 : 128;     // weight group size
    static constexpr int GPU = 128 / G;                       // groups (accumulators) per unit
    static constexpr int NT = kTc8Terms * MP;                 // accumulator columns, all terms
    static constexpr uint32_t kSlotCols = 32 + GPU * NT;      // A buffer + accumulators
    static constexpr int kSlotsFit = static_cast<int>(kTmemCols / kSlotCols);
    // issuer warps, and tensor-memory slots: a multiple of them, so that each slot (and each x
    // stage) belongs to one issuer, which waits on its barriers' phases in order
    static constexpr int I = kSlotsFit < kMaxIssuers ? kSlotsFit : kMaxIssuers;
    static constexpr int K = (kSlotsFit / I) * I;
    static constexpr int CW = MP / 4;                         // columns per epilogue thread
    // units read per tensor-memory round trip by one epilogue warp (register budget)
    static constexpr int kPerUnit = GPU * kTc8Terms * CW;     // values loaded per unit
    static constexpr int UPR = kPerUnit <= 24 ? 2 : 1;
    static constexpr uint32_t kXTile = static_cast<uint32_t>(NT) * 128; // one x stage
    static constexpr uint32_t kPkStage = kBoxes * kPkBytes;
    static_assert(K >= 2 && K % I == 0, "tensor-memory slots: at least two, a multiple of I");
    static_assert(MP % 16 == 0 && 2 * MP <= 256 && NT <= 256, "MMA N out of range");
    static_assert(CW == 4 || CW == 8 || CW == 16, "epilogue column part of 4, 8 or 16");
    static_assert(kXTile % 1024 == 0 && kPkStage % 1024 == 0, "stages keep 1024-byte alignment");
};

struct Tc8Params {
    const uint16_t *S;
    const uint16_t *ZS;
    const float *xs2;       // [MP][NGt] sums of the 2-term representation (scaled units)
    const float *xs3;       // [MP][NGt] sums of the 3-term representation
    const float *row_f;     // [3][kTc8MaxMP] per batch row: 2^-e, weights of terms 2 and 3
    const int *row_terms;   // [MP] terms each row needs (2 or 3)
    int V, H, m0, mrows, kcand, ntiles, npk, nx;
    long long ncand;
    float *cand_val;
    int32_t *cand_idx;
    float *coarse;
    int *timeout_flag;
};

// kind::f8f6f4 instruction descriptor: D f32, A e4m3, B e4m3, both K-major, M = 128, N.
__host__ __device__ constexpr uint32_t make_idesc_f8(int N)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

template <int CW>
__device__ __forceinline__ void tmem_ld_cw(uint32_t taddr, float (&v)[CW])
{
    if constexpr (CW == 4) tmem_ld_x4(taddr, v);
    else if constexpr (CW == 8) tmem_ld_x8(taddr, v);
    else tmem_ld_x16(taddr, v);
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::
                     "r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                 "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

// e4m3 weights of plane P from a word of four packed bytes (four consecutive k): the codes
// masked in place, v 2^-9 (even P) or 4 v 2^-9 (odd P), exact e4m3 values
__device__ __forceinline__ uint32_t deq4_e4m3(uint32_t w, int P)
{
    return (P >= 2 ? (w >> 4) : w) & ((P & 1) ? 0x0C0C0C0Cu : 0x03030303u);
}

// The 4-bit head: the low / high nibble of each byte, v 2^-9 with v in 0..15 (e4m3 bytes 0..15
// are exactly p 2^-9: subnormals up to 7, then 2^-6 (1 + m/8) = (8 + m) 2^-9).
__device__ __forceinline__ uint32_t deq_nib(uint32_t w, int hi)
{
    return (hi ? (w >> 4) : w) & 0x0F0F0F0Fu;
}

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

// Block top-KCAND for KCAND <= 8, one lane per (batch column, block) pair: the lane walks the
// block's 64 values in row order and keeps the 8 best in a descending list.  A value enters
// only where it is strictly greater, so equal values keep the lower row first; rows past the
// head hold -inf and never enter, leaving (-inf, -1) in unfilled slots.  With `coarse` set it
// also writes the block's coarse values (rows below V).
__device__ __forceinline__ void select_lane8(const float *pair, int base_row, int V, int kcand,
                                             float *oval, int32_t *oidx, float *coarse)
{
    float v[8];
    int r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = -INFINITY;
        r[k] = -1;
    }
#pragma unroll 2
    for (int j4 = 0; j4 < kBlockN / 4; ++j4) {
        const float4 u = reinterpret_cast<const float4 *>(pair)[j4];
        const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float xv = uu[e];
            const int row = base_row + 4 * j4 + e;
            if (coarse && row < V) coarse[row] = xv;
            bool c[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) c[k] = xv > v[k];
            // the list is descending, so c is false up to the insertion point, true after it
#pragma unroll
            for (int k = 7; k > 0; --k) {
                v[k] = c[k] ? (c[k - 1] ? v[k - 1] : xv) : v[k];
                r[k] = c[k] ? (c[k - 1] ? r[k - 1] : row) : r[k];
            }
            v[0] = c[0] ? xv : v[0];
            r[0] = c[0] ? row : r[0];
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < kcand) {
            oval[k] = v[k];
            oidx[k] = r[k];
        }
}

// Shared-memory plan of one launch configuration.
struct Smem8 {
    uint32_t pk, x, sz, red, xs, inv, bars, total;
    int npk, nx;
};

__host__ __device__ inline uint32_t sz_tile_bytes(int H, int G)
{
    return static_cast<uint32_t>(kTileRows) * (H / G) * 2; // S (or ZS) of one tile
}

template <int MP, int PACK>
__host__ __device__ inline Smem8 smem_plan(int H, int npk, int nx)
{
    using C = Cfg8<MP, PACK>;
    Smem8 p;
    p.npk = npk;
    p.nx = nx;
    p.pk = 0; // offsets from the 1024-aligned base
    p.x = p.pk + static_cast<uint32_t>(npk) * C::kPkStage;
    p.sz = p.x + static_cast<uint32_t>(nx) * C::kXTile;
    p.red = p.sz + 4 * sz_tile_bytes(H, C::G);
    p.xs = p.red + static_cast<uint32_t>(MP) * 2 * kRedPitch * 4;
    p.inv = p.xs + static_cast<uint32_t>(H / C::G) * MP * 4;
    p.bars = (p.inv + 3 * MP * 4 + 4 + 7u) & ~7u; // 2^-e, term weights, the launch's term count
    const uint32_t nbars = 2 * npk + 2 * nx + 3 * C::K + 4 + 2 + C::I;
    // + the tensor-memory address word, + slack for the 1024-byte alignment of the base (no
    // static shared memory: the dynamic size may then take the whole per-block limit)
    p.total = p.bars + nbars * 8 + 8 + 1024;
    return p;
}

template <int MP, int PACK>
__global__ void __launch_bounds__(kThreads, 1)
    coarse_tc8_kernel(const __grid_constant__ CUtensorMap tm_packed,
                      const __grid_constant__ CUtensorMap tm_x, const Tc8Params prm)
{
    using C = Cfg8<MP, PACK>;
    constexpr int BITS = PACK == kPackHalf4 ? 4 : 2;
    constexpr int G = C::G, GPU = C::GPU, NT = C::NT, K = C::K, I = C::I;
    constexpr int CW = C::CW, UPR = C::UPR, kBoxes = C::kBoxes;
    constexpr uint32_t kSlotCols = C::kSlotCols;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = prm.H / 512, NGt = prm.H / G;
    const int npk = prm.npk, nx = prm.nx;
    const Smem8 L = smem_plan<MP, PACK>(prm.H, npk, nx);
    const uint32_t sz_bytes = sz_tile_bytes(prm.H, G);

    // ---- shared memory ------------------------------------------------------------------
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *const base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *const pkring = base + L.pk;
    uint8_t *const xring = base + L.x;
    uint8_t *const szbuf = base + L.sz;
    float *const red = reinterpret_cast<float *>(base + L.red);
    float *const xs_s = reinterpret_cast<float *>(base + L.xs); // [NGt][MP]
    float *const inv_s = reinterpret_cast<float *>(base + L.inv); // [MP] 2^-e
    float *const tw_s = inv_s + MP;                               // [2][MP] term weights
    int *const nterms_s = reinterpret_cast<int *>(tw_s + 2 * MP);
    uint64_t *const bars = reinterpret_cast<uint64_t *>(base + L.bars);
    uint64_t *const pk_full = bars;              // [npk] TMA -> dequant
    uint64_t *const pk_empty = pk_full + npk;    // [npk] dequant (4 warps) -> TMA
    uint64_t *const x_full = pk_empty + npk;     // [nx]  TMA -> issuer
    uint64_t *const x_empty = x_full + nx;       // [nx]  MMA commit -> TMA
    uint64_t *const a_full = x_empty + nx;       // [K]   dequant (4 warps) -> issuer
    uint64_t *const d_full = a_full + K;         // [K]   MMA commit -> epilogue, dequant
    uint64_t *const d_empty = d_full + K;        // [K]   epilogue (16 warps) -> issuer
    uint64_t *const sz_full = d_empty + K;       // [2]   bulk copy -> epilogue
    uint64_t *const sz_empty = sz_full + 2;      // [2]   epilogue (16 warps) -> bulk copy
    uint64_t *const red_full = sz_empty + 2;     // [1]   epilogue (16 warps) -> selection
    uint64_t *const red_free = red_full + 1;     // [1]   selection -> epilogue
    uint64_t *const fin = red_free + 1;          // [I]   issuer drain before teardown
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(fin + I);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_packed);
        prefetch_tensormap(&tm_x);
        for (int i = 0; i < npk; ++i) {
            mbar_init(&pk_full[i], 1);
            mbar_init(&pk_empty[i], kDqWarps);
        }
        for (int i = 0; i < nx; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < K; ++i) {
            mbar_init(&a_full[i], kDqWarps);
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kEpWarps); // every epilogue warp reads every unit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sz_full[i], 1);
            mbar_init(&sz_empty[i], kEpWarps);
        }
        mbar_init(red_full, kEpWarps);
        mbar_init(red_free, 1);
        for (int i = 0; i < I; ++i) mbar_init(&fin[i], 1);
        fence_barrier_init();
    }
    // the launch's term count: the most any of its rows needs
    if (warp == 0) {
        int t = 2;
        for (int m = lane; m < MP; m += 32) t = max(t, prm.row_terms[m]);
        t = __reduce_max_sync(0xffffffffu, t);
        if (lane == 0) *nterms_s = t > 2 ? 3 : 2;
    }
    __syncthreads();
    const int T = *nterms_s;
    const float *const xsrc = T == 3 ? prm.xs3 : prm.xs2;
    for (int i = threadIdx.x; i < NGt * MP; i += blockDim.x) {
        const int g = i / MP, m = i - g * MP;
        xs_s[i] = xsrc[static_cast<long long>(m) * NGt + g];
    }
    for (int i = threadIdx.x; i < MP; i += blockDim.x) {
        inv_s[i] = prm.row_f[i];
        tw_s[i] = prm.row_f[kTc8MaxMP + i];
        tw_s[MP + i] = prm.row_f[2 * kTc8MaxMP + i];
    }
    if (warp == kWarpPk) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int first_tile = blockIdx.x, tile_step = gridDim.x;
    const int my_tiles = first_tile < prm.ntiles ? (prm.ntiles - 1 - first_tile) / tile_step + 1 : 0;
    const int units = my_tiles * NG * 4; // this CTA's units, in order
    bool failed = false;

    if (warp == kWarpPk) {
        // ---------------- TMA: packed codes and S / ZS ----------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            uint32_t s = 0;
            for (int it = 0; it < my_tiles && !failed; ++it) {
                const int tile = first_tile + it * tile_step;
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
                for (int span = 0; span < NG; ++span, ++s) {
                    const uint32_t st = s % npk;
                    if (!mbar_wait_bounded(&pk_empty[st], ((s / npk) & 1u) ^ 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    uint8_t *const stage = pkring + static_cast<size_t>(st) * C::kPkStage;
                    mbar_arrive_expect_tx(&pk_full[st], C::kPkStage);
#pragma unroll
                    for (int bx = 0; bx < kBoxes; ++bx)
                        tma_load_2d_hint(stage + bx * kPkBytes, &tm_packed,
                                         (kBoxes * span + bx) * kSpanBytes, tile * kTileRows,
                                         &pk_full[st], policy);
                }
            }
        }
    } else if (warp == kWarpX) {
        // ---------------- TMA: the staged x terms of every unit ----------------
        if (lane == 0) {
            const uint32_t xbytes = static_cast<uint32_t>(T) * MP * 128;
            for (int q = 0; q < units && !failed; ++q) {
                const int span = (q >> 2) % NG, plane = q & 3;
                const uint32_t st = q % nx;
                if (!mbar_wait_bounded(&x_empty[st], ((q / nx) & 1u) ^ 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                uint8_t *const stage = xring + static_cast<size_t>(st) * C::kXTile;
                const int k0 = plane_group<PACK>(plane, span, NG) * kGroup;
                mbar_arrive_expect_tx(&x_full[st], xbytes);
                for (int t = 0; t < T; ++t)
                    tma_load_2d(stage + t * (MP * 128), &tm_x, k0, t * MP, &x_full[st]);
            }
        }
    } else if (warp >= kWarpIss0 && warp < kWarpIss0 + I) {
        // ---------------- MMA issuers: unit q goes to issuer q % I, slot q % K ----------------
        if (lane == 0) {
            const int me = warp - kWarpIss0;
            const uint32_t idesc = make_idesc_f8(T * MP);
            for (int q = me; q < units && !failed; q += I) {
                const uint32_t slot = q % K, use = q / K, st = q % nx;
                if (!mbar_wait_bounded(&x_full[st], (q / nx) & 1u, prm.timeout_flag) ||
                    !mbar_wait_bounded(&a_full[slot], use & 1u, prm.timeout_flag) ||
                    !mbar_wait_bounded(&d_empty[slot], (use & 1u) ^ 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_tmem = tmem + slot * kSlotCols;
                const uint32_t d_tmem = a_tmem + 32;
                const uint64_t xdesc =
                    sw128_desc(smem_u32(xring + static_cast<size_t>(st) * C::kXTile));
                // K = 32 per MMA (32 bytes of the swizzled rows: +2 in the descriptor's 16-byte
                // address units); groups of 64 put MMAs 0-1 and 2-3 in their own accumulators
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    mma_ts_f8(d_tmem + (i / (4 / GPU)) * NT, a_tmem + i * 8,
                              xdesc + static_cast<uint64_t>(i * 2), idesc,
                              (i % (4 / GPU)) ? 1u : 0u);
                mma_commit(&d_full[slot]);
                mma_commit(&x_empty[st]);
            }
            mma_commit(&fin[me]);
            mbar_wait_bounded(&fin[me], 0, prm.timeout_flag);
        }
    } else if (warp >= kWarpDq0 && warp < kWarpDq0 + kDqWarps) {
        // ---------------- dequant: one TMEM lane (= tile row) per thread ----------------
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        int q = 0;
        for (int sidx = 0; sidx < my_tiles * NG && !failed; ++sidx) {
            const uint32_t st = sidx % npk;
            if (!warp_wait(&pk_full[st], (sidx / npk) & 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            const uint32_t pk = smem_u32(pkring + static_cast<size_t>(st) * C::kPkStage) +
                                row * kSpanBytes;
            uint32_t w[32];
            // this thread's row of packed box bx (128-byte swizzle)
            auto load_box = [&](int bx) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = pk + bx * kPkBytes + ((c ^ (row & 7)) << 4);
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]),
                                   "=r"(w[4 * c + 3])
                                 : "r"(addr));
                }
            };
            load_box(0);
            if constexpr (BITS == 2) {
                // every plane of the span is in these 32 words: the stage goes back now
                __syncwarp();
                if (lane == 0) mbar_arrive(&pk_empty[st]);
            }
#pragma unroll 1
            for (int plane = 0; plane < 4; ++plane, ++q) {
                if (BITS == 4 && plane == 2) {
                    // planes 2 bx, 2 bx + 1 are the two nibbles of box bx
                    load_box(1);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&pk_empty[st]);
                }
                const uint32_t slot = q % K, use = q / K;
                // the slot's A buffer is free once its previous unit's MMAs have completed
                if (use > 0 && !warp_wait(&d_full[slot], (use - 1) & 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t abuf = tmem + lane_base + slot * kSlotCols;
                // two halves of 16 columns (64 k) each
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t r[16];
                    if constexpr (BITS == 4) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = deq_nib(w[16 * hf + i], plane & 1);
                    } else if constexpr (PACK == kPackContig2) {
                        // plane p is words 8p .. 8p + 7; half hf is words 8p + 4 hf ..
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t o[4];
                            deq_c4(w[8 * plane + 4 * hf + i], o);
#pragma unroll
                            for (int b = 0; b < 4; ++b) r[4 * i + b] = o[b];
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = deq4_e4m3(w[16 * hf + i], plane);
                    }
                    tmem_st_x16(abuf + 16 * hf, r);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[slot]);
            }
        }
    } else if (warp >= kWarpEp0) {
        // ---------------- epilogue: set cp = batch columns [cp CW, cp CW + CW) ----------------
        const int cp = (warp - kWarpEp0) >> 2;
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        for (int it = 0; it < my_tiles && !failed; ++it) {
            const int tile = first_tile + it * tile_step;
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
            float acc[CW];
#pragma unroll
            for (int j = 0; j < CW; ++j) acc[j] = 0.f;
            for (int span = 0; span < NG && !failed; ++span) {
#pragma unroll 1
                for (int p0 = 0; p0 < 4; p0 += UPR) {
                    // the units of planes p0 .. p0 + UPR - 1 of the span
                    float v[UPR][GPU][kTc8Terms][CW];
                    const int q0 = (it * NG + span) * 4 + p0;
#pragma unroll
                    for (int u = 0; u < UPR; ++u) {
                        const uint32_t slot = (q0 + u) % K, use = (q0 + u) / K;
                        if (!warp_wait(&d_full[slot], use & 1u, prm.timeout_flag)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t dcol = tmem + lane_base + slot * kSlotCols + 32 + cp * CW;
#pragma unroll
                        for (int a = 0; a < GPU; ++a)
#pragma unroll
                            for (int t = 0; t < kTc8Terms; ++t)
                                if (t < T) tmem_ld_cw<CW>(dcol + a * NT + t * MP, v[u][a][t]);
                    }
                    if (failed) break;
                    tmem_wait_ld();
                    // every partial of these units is in registers: their slots go back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
#pragma unroll
                        for (int u = 0; u < UPR; ++u) mbar_arrive(&d_empty[(q0 + u) % K]);
#pragma unroll
                    for (int u = 0; u < UPR; ++u) {
                        const int plane = p0 + u;
#pragma unroll
                        for (int a = 0; a < GPU; ++a) {
                            const int gi = plane_group<PACK>(plane, span, NG) * GPU + a;
                            uint16_t sb = 0, zb = 0;
                            if (full_tile) {
                                sb = sS[gi];
                                zb = sZ[gi];
                            } else if (row_ok) {
                                sb = __ldg(gS + gi);
                                zb = __ldg(gZ + gi);
                            }
                            const float sv = bf16_bits_to_f32(sb), zv = bf16_bits_to_f32(zb);
                            // (S / B) sum x v with the MMA's sum of x v 2^-9 (quarter split,
                            // B = 4: odd planes carry 4 v 2^-9, even planes v 2^-9;
                            // contiguous-4, B = 4: every plane v 2^-9; 4 bits, B = 16: v 2^-9)
                            const bool four_v = PACK != kPackHalf4 && PACK != kPackContig2 && (plane & 1);
                            const float s2 = (BITS == 4 ? 32.0f : (four_v ? 32.0f : 128.0f)) * sv;
                            const float sz = sv - zv;
                            const float *const xg = xs_s + gi * MP + cp * CW;
                            const float *const w2 = tw_s + cp * CW, *const w3 = w2 + MP;
#pragma unroll
                            for (int j = 0; j < CW; ++j) {
                                // the row's terms, weighted by their powers of two (exact)
                                float r = fmaf(sz, xg[j], acc[j]);
                                r = fmaf(s2, v[u][a][0][j], r);
                                r = fmaf(s2 * w2[j], v[u][a][1][j], r);
                                if (T == 3) r = fmaf(s2 * w3[j], v[u][a][2][j], r);
                                acc[j] = r;
                            }
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
            float *const rh = red + (row >> 6) * kRedPitch + (row & 63);
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const int m = cp * CW + j;
                rh[2 * m * kRedPitch] = row_ok ? acc[j] * inv_s[m] : -INFINITY;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_full);
        }
    } else if (warp == kWarpSel) {
        // ---------------- block top-KCAND: pair = (batch column m, block b of the tile) ------
        const int npairs = 2 * prm.mrows;
        for (int it = 0; it < my_tiles && !failed; ++it) {
            const int tile = first_tile + it * tile_step;
            if (!warp_wait(red_full, it & 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            if (prm.kcand <= 8) {
                // one lane per pair
                for (int pidx = lane; pidx < npairs; pidx += 32) {
                    const int m = pidx >> 1, blk = tile * 2 + (pidx & 1);
                    if (static_cast<long long>(blk) * kBlockN < prm.V) {
                        const long long off = static_cast<long long>(prm.m0 + m) * prm.ncand +
                                              static_cast<long long>(blk) * prm.kcand;
                        float *const cdbg =
                            prm.coarse ? prm.coarse + static_cast<long long>(prm.m0 + m) * prm.V
                                       : nullptr;
                        select_lane8(red + pidx * kRedPitch, blk * kBlockN, prm.V, prm.kcand,
                                     prm.cand_val + off, prm.cand_idx + off, cdbg);
                    }
                }
            } else {
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
                        const float c0 = pv[lane];
                        const float c1 = pv[lane + 32];
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
    }

    // ---- teardown: every role is done (or gave up); release tensor memory ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpPk) tmem_dealloc(tmem, kTmemCols);
}

// Stage counts for a launch configuration: x stages a multiple of the issuer count (each
// issuer owns nx / I of them, two where they fit, so that an issuer's next x tile is in flight
// while it works), then as many packed stages as fit (two to eight); false if nothing fits.
template <int MP, int PACK>
bool pick_stages(int H, int *npk, int *nx)
{
    using C = Cfg8<MP, PACK>;
    for (int per = 2; per >= 1; --per) {
        const int x = per * C::I;
        for (int p = 8; p >= 2; --p) {
            if (smem_plan<MP, PACK>(H, p, x).total <= static_cast<uint32_t>(kSmemLimit8)) {
                *npk = p;
                *nx = x;
                return true;
            }
        }
    }
    return false;
}

template <int MP, int PACK>
cudaError_t launch_cfg(const CUtensorMap &tm_packed, const uint8_t *xt8_chunk,
                       const Tc8Params &base, cudaStream_t stream)
{
    CUtensorMap tm_x;
    // the staged x of the launch: [3 MP rows, H] bytes; a box is one term's MP rows x 128 k
    CUresult r = encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                      const_cast<uint8_t *>(xt8_chunk), base.H,
                                      static_cast<uint64_t>(kTc8Terms) * MP, base.H, 128, MP,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    int npk = 0, nx = 0;
    if (!pick_stages<MP, PACK>(base.H, &npk, &nx)) return cudaErrorInvalidConfiguration;
    const uint32_t smem = smem_plan<MP, PACK>(base.H, npk, nx).total;
    // the shared-memory limit is a per-device attribute: raised once on every device
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        return cudaFuncSetAttribute(coarse_tc8_kernel<MP, PACK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit8);
    });
    if (e != cudaSuccess) return e;
    Tc8Params prm = base;
    prm.npk = npk;
    prm.nx = nx;
    const int sms = device_sm_count();
    const int grid = prm.ntiles < sms ? prm.ntiles : sms;
    coarse_tc8_kernel<MP, PACK><<<grid, kThreads, smem, stream>>>(tm_packed, tm_x, prm);
    return cudaGetLastError();
}

template <int PACK>
bool fits_all(int H)
{
    int p, x;
    if constexpr (PACK == kPackG64) return pick_stages<16, PACK>(H, &p, &x);
    else if constexpr (PACK == kPackQuarter2)
        return pick_stages<16, PACK>(H, &p, &x) && pick_stages<32, PACK>(H, &p, &x) &&
               pick_stages<64, PACK>(H, &p, &x);
    else return pick_stages<16, PACK>(H, &p, &x) && pick_stages<32, PACK>(H, &p, &x);
}

} // namespace

int tc8_max_rows(int pack)
{
    if (pack == kPackG64) return 16;
    if (pack == kPackQuarter2) return 64;
    return 32; // the 4-bit head and the contiguous-4 layout
}

int tc8_chunks(int M, int pack)
{
    const int r = tc8_max_rows(pack);
    return (M + r - 1) / r;
}

Tc8Chunk tc8_chunk(int M, int c, int pack, int H)
{
    const int r = tc8_max_rows(pack);
    Tc8Chunk k;
    k.m0 = c * r;
    k.rows = M - k.m0 < r ? M - k.m0 : r;
    k.MP = k.rows <= 16 ? 16 : (k.rows <= 32 ? 32 : 64);
    // launches before c are full (r rows, MP = r)
    k.x_off = static_cast<size_t>(c) * kTc8Terms * r * H;
    return k;
}

size_t tc8_x_bytes(int M, int H)
{
    size_t most = 0;
    const int packs[3] = {kPackQuarter2, kPackHalf4, kPackG64};
    for (int pack : packs) {
        const int n = tc8_chunks(M, pack);
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
    if (bits == 4) return group == 128 && fits_all<kPackHalf4>(H);
    if (group == 64) return M <= 16 && fits_all<kPackG64>(H);
    if (group != 128) return false;
    return fits_all<kPackQuarter2>(H) && fits_all<kPackContig2>(H);
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
    const int G = a.pack == kPackG64 ? 64 : 128;
    const int NGt = a.H / G;
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
    base.npk = base.nx = 2;
    for (int c = 0; c < tc8_chunks(a.M, a.pack); ++c) {
        const Tc8Chunk k = tc8_chunk(a.M, c, a.pack, a.H);
        float *const small = w.small + static_cast<size_t>(c) * tc8_small_floats(a.H);
        base.m0 = k.m0;
        base.mrows = k.rows;
        base.xs2 = small;
        base.xs3 = small + static_cast<size_t>(kTc8MaxMP) * (a.H / 64);
        base.row_f = small + 2 * static_cast<size_t>(kTc8MaxMP) * (a.H / 64);
        base.row_terms = reinterpret_cast<const int *>(base.row_f + 3 * kTc8MaxMP);
        (void)NGt;
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
            else if (k.MP == 32) e = launch_cfg<32, kPackQuarter2>(tm_packed, xt, base, stream);
            else e = launch_cfg<64, kPackQuarter2>(tm_packed, xt, base, stream);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace dh
