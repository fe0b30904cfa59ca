// dh_quantize.cu -- kernel (1): quantise and pack the head to 2 (or 4) bits.
//
// radiance_drafthead.py, _quantize_head_now (GROUP = 128): per (row, group of 128 consecutive
// k), in IEEE fp32, with L = 2^BITS - 1 levels and bias B = 2^BITS,
//     lo, hi = min, max;  sc = max((hi - lo) / L, 1e-8);  zp = clamp(rne(-lo / sc), 0, L)
//     q_k = clamp(rne(w_k / sc + zp), 0, L);  S = bf16(B sc);  ZS = bf16(B sc + zp sc)
// BITS = 2 (the default head): quarter split, byte j of a row holds
// q[j] | q[Q+j] << 2 | q[2Q+j] << 4 | q[3Q+j] << 6 (Q = H/4).  BITS = 4 (the page's 4-bit
// variant): half split, byte j holds q[j] | q[H/2+j] << 4.
//
// Every arithmetic step uses the explicitly rounded intrinsics (no contraction into FMA),
// division is correctly rounded, rintf rounds half to even: the result is bit-exact with the
// definition.  The per-weight division is replaced by a product with the group's reciprocal
// wherever that provably gives the same code (quant_pair), because a correctly rounded
// division per weight -- a reciprocal on the SM's few special-function units, a rounding and a
// float-to-int conversion -- bound the kernel far below the HBM rate (2 bytes read per weight,
// BITS/8 + 1/32 written).
//
// An fp8 head (kernel (1) with the e4m3 input): row n's weights are the fp32 products
// e4m3(b) * wsc[n] (radiance_drafthead.py, _quantize_head_now, the fp8 weight pre-scaled by its
// per-row scale before the group statistics), each rounded once; the steps above then run on
// those values.
//
// Work unit: one warp per (row n, two spans) with groups of 128 (one span with groups of 64),
// where span s is packed bytes [128 s, 128 s + 128) of the row -- one group per plane p
// (P = 8 / BITS planes): group p NS + s, NS = H / (128 P) spans per row.  Lane l owns packed
// bytes 4l .. 4l+3 of each span, i.e. four consecutive weights of each of the span's groups, so
// the packed words it writes need nothing from other lanes.
#include "dh_common.cuh"
#include "dh_internal.h"

#include <type_traits>

namespace dh {

// min / max over aligned groups of L lanes (L = 32: the warp)
template <int L>
__device__ __forceinline__ float lanes_min(float v)
{
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int L>
__device__ __forceinline__ float lanes_max(float v)
{
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The group's scale and zero point, as defined (both correctly rounded divisions).
struct GroupParams {
    float sc, zp;
};

__device__ __forceinline__ GroupParams group_params(float lo, float hi, float L)
{
    const float sc = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), L), 1e-8f);
    const float zp = fminf(fmaxf(rintf(__fdiv_rn(-lo, sc)), 0.0f), L);
    return {sc, zp};
}

// The defining code of one weight: clamp(rne(fl32(fl32(w / sc) + zp)), 0, L).
__device__ __forceinline__ uint32_t code_by_definition(float w, GroupParams g, float L)
{
    const float re = rintf(__fadd_rn(__fdiv_rn(w, g.sc), g.zp));
    return static_cast<uint32_t>(fminf(fmaxf(re, 0.0f), L));
}

// The fast codes of a pair of weights of one group, added into a packed word.
//
// With ra = fl32(fl32(1 / sc) fl32(1 / L)) and zb = fl32(zp fl32(1 / L)) (once per group),
// y = fl32(w ra + zb) is the code's argument divided by L, clamped to [0, 1] by the FMA's
// saturation (the code's own clamp: clamping to integer ends commutes with rounding to the
// nearest integer).  Against the defining t* = fl32(fl32(w / sc) + zp), L y is off by at most
// 2^-24 (6 |w / sc| + 4 zp) (four roundings on the w / sc term and three on zp in L y, two and
// one in t*).  Where t* lies within one unit of a rounding boundary of [0, L], t* and zp both
// lie in [0, L], so |w / sc| <= L and the difference is below 10 L 2^-24 <= 2^-16 for L <= 15.
// So where L y lies farther than 2^-16 from every half-integer, rne(L y) is the defining code;
// the pair falls back to the definition otherwise (about one weight in a thousand: with bf16
// weights, sc = (hi - lo) / L often has few significant bits, and exact ties are common).
//
// rne(L y) comes from one FMA onto -1.5 2^23, whose bits are those of -1.5 2^23 plus the code in
// the low mantissa bits; the word adds those bits at each code's position, and the caller
// removes the constant part once per word (mod 2^32 the magic's bits and the codes add
// independently, and the codes' fields do not overlap).  The rounding of L y and its distance to
// the integer run on the paired fp32 units.
constexpr float kQMagic = 12582912.0f;           // 1.5 2^23
constexpr uint32_t kQMagicNegBits = 0xCB400000u; // the bits of -1.5 2^23
constexpr float kQThreshold = 0.5f - 0x1p-16f;   // |L y - rne(L y)| at or above: near a boundary

// The magic's bits summed over n fields at positions 0, step, 2 step, ...
__host__ __device__ constexpr uint32_t magic_bits_sum(int n, int step)
{
    uint32_t c = 0;
    for (int i = 0; i < n; ++i) c += kQMagicNegBits << (i * step);
    return c;
}

__device__ __forceinline__ float fma_sat(float a, float b, float c)
{
    float r;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The correction that turns a pair's fast codes (magic bits b0, b1 at s0, s1) into the defining
// ones; out of line, so that the rare path costs the unrolled loop no code space.
__device__ __noinline__ uint32_t pair_by_definition(float w0, float w1, float lo, float hi, float L,
                                                    uint32_t b0, uint32_t b1, int s0, int s1)
{
    const GroupParams g = group_params(lo, hi, L);
    return ((code_by_definition(w0, g, L) - (b0 - kQMagicNegBits)) << s0) +
           ((code_by_definition(w1, g, L) - (b1 - kQMagicNegBits)) << s1);
}

template <int BITS>
__device__ __forceinline__ void quant_pair(float w0, float w1, float ra, float zb, float lo,
                                           float hi, int s0, int s1, uint32_t &word)
{
    constexpr float L = static_cast<float>((1 << BITS) - 1);
    const float2 y = make_float2(fma_sat(w0, ra, zb), fma_sat(w1, ra, zb));
    const float2 m = __ffma2_rn(y, make_float2(-L, -L), make_float2(-kQMagic, -kQMagic));
    const float2 nr = __fadd2_rn(m, make_float2(kQMagic, kQMagic)); // -rne(L y), exact
    const float2 d = __ffma2_rn(y, make_float2(L, L), nr);         // L y - rne(L y)
    const uint32_t b0 = __float_as_uint(m.x), b1 = __float_as_uint(m.y);
    word += b0 << s0;
    word += b1 << s1;
    if (__builtin_expect(fmaxf(fabsf(d.x), fabsf(d.y)) >= kQThreshold, 0))
        word += pair_by_definition(w0, w1, lo, hi, L, b0, b1, s0, s1);
}

// The same for four weights of one group at bit positions s0, s0 + step, s0 + 2 step, s0 + 3
// step, with one boundary test for the four (two pairs on the paired units).
__device__ __noinline__ uint32_t quad_by_definition(float w0, float w1, float w2, float w3, float lo,
                                                    float hi, float L, uint32_t b0, uint32_t b1,
                                                    uint32_t b2, uint32_t b3, int s0, int step)
{
    const GroupParams g = group_params(lo, hi, L);
    return ((code_by_definition(w0, g, L) - (b0 - kQMagicNegBits)) << s0) +
           ((code_by_definition(w1, g, L) - (b1 - kQMagicNegBits)) << (s0 + step)) +
           ((code_by_definition(w2, g, L) - (b2 - kQMagicNegBits)) << (s0 + 2 * step)) +
           ((code_by_definition(w3, g, L) - (b3 - kQMagicNegBits)) << (s0 + 3 * step));
}

// Returns true when one of the four lies within the margin of a rounding boundary; the caller
// then adds quad_by_definition's correction (with the group's extrema).
template <int BITS>
__device__ __forceinline__ bool quant_quad(const float (&w)[4], float ra, float zb, int s0, int step,
                                           uint32_t &word, uint32_t (&b)[4])
{
    constexpr float L = static_cast<float>((1 << BITS) - 1);
    const float2 ya = make_float2(fma_sat(w[0], ra, zb), fma_sat(w[1], ra, zb));
    const float2 yb = make_float2(fma_sat(w[2], ra, zb), fma_sat(w[3], ra, zb));
    const float2 ma = __ffma2_rn(ya, make_float2(-L, -L), make_float2(-kQMagic, -kQMagic));
    const float2 mb = __ffma2_rn(yb, make_float2(-L, -L), make_float2(-kQMagic, -kQMagic));
    const float2 da = __ffma2_rn(ya, make_float2(L, L), __fadd2_rn(ma, make_float2(kQMagic, kQMagic)));
    const float2 db = __ffma2_rn(yb, make_float2(L, L), __fadd2_rn(mb, make_float2(kQMagic, kQMagic)));
    b[0] = __float_as_uint(ma.x);
    b[1] = __float_as_uint(ma.y);
    b[2] = __float_as_uint(mb.x);
    b[3] = __float_as_uint(mb.y);
#pragma unroll
    for (int i = 0; i < 4; ++i) word += b[i] << (s0 + i * step);
    const float dm = fmaxf(fmaxf(fabsf(da.x), fabsf(da.y)), fmaxf(fabsf(db.x), fabsf(db.y)));
    return __builtin_expect(dm >= kQThreshold, 0);
}

// The fast path's per-group constants ra, zb.
template <int BITS>
__device__ __forceinline__ float2 fast_params(GroupParams g)
{
    constexpr float kInvL = 1.0f / static_cast<float>((1 << BITS) - 1); // fl32(1 / L)
    return make_float2(__fmul_rn(__frcp_rn(g.sc), kInvL), __fmul_rn(g.zp, kInvL));
}

// Bytes 0 and 1 of v, two e4m3 codes, as fp32: the conversion unit's e4m3 -> f16 pair (every
// finite e4m3 value is an f16 value), then f16 -> f32; both exact.  (Placing the code's fields
// in an fp32 word and scaling by 2^120, also exact, measured slower: the integer pipe is the
// busier one here.)
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t v)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(h2) : "r"(v));
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

// Element-wise minimum / maximum of two bf16 pairs (each result is one of its inputs; the sign
// of a zero result may differ from fminf's, which changes no code, S or ZS: the extrema enter
// only as hi - lo and -lo / sc, rounded to an integer and clamped at 0).
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// min / max over the whole warp in one instruction each (groups of 128: every lane holds four
// weights of each group of the span)
__device__ __forceinline__ float warp_min_f32(float v)
{
    float r;
    asm("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float warp_max_f32(float v)
{
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// kFp8: W holds e4m3 bytes and wsc the per-row fp32 scales; otherwise W holds bf16.
// G: the group size, 128 (the head) or 64 (the page's group-size ablation: each plane's 128 k
// of a span are two groups, lanes 0-15 and 16-31).
template <bool kFp8, int BITS, int G>
__global__ void __launch_bounds__(256, 3) quantize_kernel(const void *__restrict__ Wv,
                                                       const float *__restrict__ wsc,
                                                       uint8_t *__restrict__ packed,
                                                       uint16_t *__restrict__ S,
                                                       uint16_t *__restrict__ ZS, int V, int H)
{
    constexpr int P = 8 / BITS;                          // planes (codes per byte)
    constexpr float L = static_cast<float>((1 << BITS) - 1);
    constexpr float B = static_cast<float>(1 << BITS);
    // spans per work item: two with groups of 128 (the per-group work -- extrema, scale and
    // zero point, fast constants, the S / ZS stores -- is then shared by 8 groups' lanes at
    // once), one with groups of 64
    constexpr int SPI = G == 128 ? 2 : 1;
    constexpr int NGI = SPI * P; // groups of 128 k per item
    const int lane = threadIdx.x & 31;
    const int PS = H / P;       // k stride between planes = packed bytes per row
    const int NS = PS / 128;    // spans per row
    const int NSI = (NS + SPI - 1) / SPI; // items per row (the last may hold one span)
    const int NGt = H / G;      // groups per row
    // the extrema of the item's groups, for the rare codes taken by their definition
    __shared__ float lohi_s[8][2 * NGI];
    float *const lohi = lohi_s[threadIdx.x >> 5];
    // work items (n, si) = warp w, w + nwarps, ...: the position advances by (dn, ds) with no
    // division in the loop, and the next item's weights are in flight while this one is
    // quantised (2 KB per warp); the two items' registers alternate, the loop body unrolled
    // twice
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    const int dn = nwarps / NSI, ds = nwarps - dn * NSI;
    const int w0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    using Raw = typename std::conditional<kFp8, uint32_t, uint2>::type;
    // an item's weights and, for the fp8 head, its row scale
    auto load = [&](int rn, int ri, Raw (&raw)[SPI][P], float &rsc) {
        if (rn >= V) return;
        if constexpr (kFp8) rsc = __ldg(wsc + rn);
#pragma unroll
        for (int j = 0; j < SPI; ++j) {
            const int rs = SPI * ri + j;
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (rs >= NS) { // the row's last item holds one span: the other reads as zero
                    raw[j][p] = Raw{};
                } else if constexpr (kFp8) {
                    const uint8_t *row = static_cast<const uint8_t *>(Wv) + static_cast<long long>(rn) * H;
                    raw[j][p] = __ldg(reinterpret_cast<const uint32_t *>(row + p * PS + 128 * rs + 4 * lane));
                } else {
                    const uint16_t *row = static_cast<const uint16_t *>(Wv) + static_cast<long long>(rn) * H;
                    raw[j][p] = __ldg(reinterpret_cast<const uint2 *>(row + p * PS + 128 * rs + 4 * lane));
                }
            }
        }
    };
    auto advance = [&](int &an, int &ai, int fn, int fi) {
        an = fn + dn;
        ai = fi + ds;
        if (ai >= NSI) {
            ai -= NSI;
            ++an;
        }
    };
    // one item: lane l holds four weights of each plane of each span, k = p PS + 128 s + 4 l + i
    auto process = [&](const Raw (&raw)[SPI][P], float rs, int n, int si) {
        const int nsp = min(SPI, NS - SPI * si); // spans in this item (warp-uniform)
        // the fp8 head's weights are decoded once and kept; bf16 weights are re-read from the
        // raw words where they are used (one shift or mask each), which keeps the register
        // count within three blocks per SM without spills
        float wv8[kFp8 ? SPI : 1][kFp8 ? P : 1][4];
        if constexpr (kFp8) {
#pragma unroll
            for (int j = 0; j < SPI; ++j)
#pragma unroll
                for (int p = 0; p < P; ++p)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const float2 v =
                            __fmul2_rn(e4m3x2_to_f32x2(raw[j][p] >> (8 * i)), make_float2(rs, rs));
                        wv8[j][p][i] = v.x;
                        wv8[j][p][i + 1] = v.y;
                    }
        }
        auto weights = [&](int j, int p, float (&w)[4]) {
            if constexpr (kFp8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) w[i] = wv8[j][p][i];
            } else {
                w[0] = __uint_as_float(raw[j][p].x << 16);
                w[1] = __uint_as_float(raw[j][p].x & 0xFFFF0000u);
                w[2] = __uint_as_float(raw[j][p].y << 16);
                w[3] = __uint_as_float(raw[j][p].y & 0xFFFF0000u);
            }
        };
        uint32_t word[SPI];
#pragma unroll
        for (int j = 0; j < SPI; ++j) word[j] = 0;
        if constexpr (G == 128) {
            // every group covers the whole warp: one reduction instruction per extremum, then
            // lane l computes the scale, zero point and fast constants of group l % NGI (span
            // (l / P) % SPI, plane l % P) once and the others fetch them
            const int gl = lane & (NGI - 1);
            float glo = 0.f, ghi = 0.f;
#pragma unroll
            for (int j = 0; j < SPI; ++j)
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    float tmin, tmax; // the lane's four weights' extrema
                    if constexpr (kFp8 || BITS == 4) { // (the packed form measured slower here)
                        float w[4];
                        weights(j, p, w);
                        tmin = fminf(fminf(w[0], w[1]), fminf(w[2], w[3]));
                        tmax = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
                    } else {
                        // on the packed bf16 pairs first (exact selections), then the halves
                        const uint32_t mn = bf16x2_min(raw[j][p].x, raw[j][p].y);
                        const uint32_t mx = bf16x2_max(raw[j][p].x, raw[j][p].y);
                        tmin = fminf(__uint_as_float(mn << 16), __uint_as_float(mn & 0xFFFF0000u));
                        tmax = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u));
                    }
                    const float lo = warp_min_f32(tmin);
                    const float hi = warp_max_f32(tmax);
                    if (gl == j * P + p) {
                        glo = lo;
                        ghi = hi;
                    }
                }
            if (lane < NGI) {
                lohi[2 * lane] = glo;
                lohi[2 * lane + 1] = ghi;
            }
            const GroupParams gg = group_params(glo, ghi, L);
            const float2 gf = fast_params<BITS>(gg);
            if (lane < NGI && gl / P < nsp) {
                const float sb = __fmul_rn(B, gg.sc);
                const long long gi = static_cast<long long>(gl % P) * NS + SPI * si + gl / P;
                S[static_cast<long long>(n) * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(sb));
                ZS[static_cast<long long>(n) * NGt + gi] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(sb, __fmul_rn(gg.zp, gg.sc))));
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < SPI; ++j)
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int g = j * P + p;
                    const float ra = __shfl_sync(0xffffffffu, gf.x, g);
                    const float zb = __shfl_sync(0xffffffffu, gf.y, g);
                    float w[4];
                    weights(j, p, w);
                    uint32_t bq[4];
                    if (quant_quad<BITS>(w, ra, zb, BITS * p, 8, word[j], bq))
                        word[j] += quad_by_definition(w[0], w[1], w[2], w[3], lohi[2 * g],
                                                      lohi[2 * g + 1], L, bq[0], bq[1], bq[2],
                                                      bq[3], BITS * p, 8);
                }
        } else {
            const int s = si; // one span per item
#pragma unroll
            for (int p = 0; p < P; ++p) {
                float w[4];
                weights(0, p, w);
                const float lo = lanes_min<G / 4>(fminf(fminf(w[0], w[1]), fminf(w[2], w[3])));
                const float hi = lanes_max<G / 4>(fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3])));
                const GroupParams g = group_params(lo, hi, L);
                const float2 f = fast_params<BITS>(g);
                uint32_t bq[4];
                if (quant_quad<BITS>(w, f.x, f.y, BITS * p, 8, word[0], bq))
                    word[0] += quad_by_definition(w[0], w[1], w[2], w[3], lo, hi, L, bq[0], bq[1],
                                                  bq[2], bq[3], BITS * p, 8);
                if ((lane & (G / 4 - 1)) == p) {
                    const float sb = __fmul_rn(B, g.sc);
                    const long long gi = (static_cast<long long>(p) * NS + s) * (128 / G) +
                                         lane / (G / 4);
                    S[static_cast<long long>(n) * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(sb));
                    ZS[static_cast<long long>(n) * NGt + gi] =
                        __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(sb, __fmul_rn(g.zp, g.sc))));
                }
            }
        }
        // a word's fields are at 8 i + BITS p: every multiple of BITS below 32
        constexpr uint32_t kFix = magic_bits_sum(32 / BITS, BITS);
#pragma unroll
        for (int j = 0; j < SPI; ++j)
            if (j < nsp)
                reinterpret_cast<uint32_t *>(packed + static_cast<long long>(n) * PS +
                                             128 * (SPI * si + j))[lane] = word[j] - kFix;
        __syncwarp(); // the extrema scratch is reused by the next item
    };
    Raw r0[SPI][P], r1[SPI][P];
    float f0 = 0.0f, f1 = 0.0f;
    int n0 = w0 / NSI, i0 = w0 - (w0 / NSI) * NSI, n1, i1;
    load(n0, i0, r0, f0);
    // items only grow along the walk: once one is past the head, so are the rest
    for (;;) {
        if (n0 >= V) break;
        advance(n1, i1, n0, i0);
        load(n1, i1, r1, f1);
        process(r0, f0, n0, i0);
        if (n1 >= V) break;
        advance(n0, i0, n1, i1);
        load(n0, i0, r0, f0);
        process(r1, f1, n1, i1);
    }
}

// The contiguous-4 layout of the 2-bit head (the page's packing ablation: byte j holds
// k = 4j .. 4j+3, code of k = 4j + f in bits 2f .. 2f+1).  Same group steps as above.  Work
// unit: one warp per (row n, span s) of 128 packed bytes = k in [512 s, 512 s + 512) = groups
// 4s .. 4s+3; lane l owns bytes 4l .. 4l+3 (k = 512 s + 16 l .. + 15), so each group is eight
// lanes and its min / max reduce over those eight.
__global__ void __launch_bounds__(256) quantize_c4_kernel(const uint16_t *__restrict__ W,
                                                          uint8_t *__restrict__ packed,
                                                          uint16_t *__restrict__ S,
                                                          uint16_t *__restrict__ ZS, int V, int H)
{
    const int lane = threadIdx.x & 31;
    const int Q = H / 4, NS = Q / 128, NGt = H / kGroup;
    const long long total = static_cast<long long>(V) * NS;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long item = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) +
                          (threadIdx.x >> 5);
         item < total; item += nwarps) {
        const long long n = item / NS;
        const int s = static_cast<int>(item - n * NS);
        const uint4 *src = reinterpret_cast<const uint4 *>(W + n * H + 512 * s + 16 * lane);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        const uint32_t raw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float w[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w[2 * i] = __uint_as_float(raw[i] << 16);
            w[2 * i + 1] = __uint_as_float(raw[i] & 0xFFFF0000u);
        }
        float lo = w[0], hi = w[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            lo = fminf(lo, w[i]);
            hi = fmaxf(hi, w[i]);
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const GroupParams g = group_params(lo, hi, 3.0f);
        const float2 f = fast_params<2>(g);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 16; i += 2) quant_pair<2>(w[i], w[i + 1], f.x, f.y, lo, hi, 2 * i, 2 * i + 2, word);
        constexpr uint32_t kFix = magic_bits_sum(16, 2);
        word -= kFix;
        if ((lane & 7) == 0) {
            const float s4 = __fmul_rn(4.0f, g.sc);
            const long long gi = 4LL * s + (lane >> 3);
            S[n * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(s4));
            ZS[n * NGt + gi] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(s4, __fmul_rn(g.zp, g.sc))));
        }
        reinterpret_cast<uint32_t *>(packed + n * Q + 128 * s)[lane] = word;
    }
}

cudaError_t launch_quantize_c4(const uint16_t *W, int V, int H, uint8_t *packed, uint16_t *S,
                               uint16_t *ZS, cudaStream_t stream)
{
    const long long total = static_cast<long long>(V) * (H / 512);
    long long blocks = (total + 7) / 8;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    quantize_c4_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(W, packed, S, ZS, V, H);
    return cudaGetLastError();
}

// One resident wave: as many blocks as fit on every SM at once (the work loop strides over the
// items), so that no block waits for a second round while others have finished.
template <bool kFp8, int BITS, int G>
cudaError_t launch_quantize_cfg(const void *W, const float *wsc, int V, int H, uint8_t *packed,
                                uint16_t *S, uint16_t *ZS, cudaStream_t stream)
{
    const int ns = H / (128 * (8 / BITS));                    // spans per row
    const long long total = static_cast<long long>(V) * (G == 128 ? (ns + 1) / 2 : ns); // items
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, quantize_kernel<kFp8, BITS, G>, 256, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    long long blocks = (total + 7) / 8;
    const long long cap = static_cast<long long>(device_sm_count()) * per_sm;
    if (blocks > cap) blocks = cap;
    quantize_kernel<kFp8, BITS, G><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        W, wsc, packed, S, ZS, V, H);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const void *W, const float *wsc, int V, int H, int bits, int group,
                            uint8_t *packed, uint16_t *S, uint16_t *ZS, cudaStream_t stream)
{
    if (bits == 4) {
        if (wsc) return launch_quantize_cfg<true, 4, 128>(W, wsc, V, H, packed, S, ZS, stream);
        return launch_quantize_cfg<false, 4, 128>(W, nullptr, V, H, packed, S, ZS, stream);
    }
    if (group == 64) // the 2-bit bf16 head with groups of 64
        return launch_quantize_cfg<false, 2, 64>(W, nullptr, V, H, packed, S, ZS, stream);
    if (wsc) return launch_quantize_cfg<true, 2, 128>(W, wsc, V, H, packed, S, ZS, stream);
    return launch_quantize_cfg<false, 2, 128>(W, nullptr, V, H, packed, S, ZS, stream);
}

} // namespace dh
