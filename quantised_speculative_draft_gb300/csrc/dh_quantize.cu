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
// wherever that provably gives the same code (quant_code), because a correctly rounded
// division per weight -- a reciprocal on the SM's few special-function units, a rounding and a
// float-to-int conversion -- bound the kernel far below the HBM rate (2 bytes read per weight,
// BITS/8 + 1/32 written).
//
// An fp8 head (kernel (1) with the e4m3 input): row n's weights are the fp32 products
// e4m3(b) * wsc[n] (radiance_drafthead.py, _quantize_head_now, the fp8 weight pre-scaled by its
// per-row scale before the group statistics), each rounded once; the steps above then run on
// those values.
//
// Work unit: one warp per (row n, span s), where span s is packed bytes [128 s, 128 s + 128)
// of the row -- one group per plane p (P = 8 / BITS planes): group p NS + s, NS = H / (128 P)
// spans per row.  Lane l owns packed bytes 4l .. 4l+3 of the span, i.e. four consecutive
// weights of each of the span's groups, so the packed word it writes needs nothing from other
// lanes.
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

// The code q = clamp(rne(fl32(fl32(w / sc) + zp)), 0, L) of one weight, without a division in the
// common case.  With rcp = fl32(1 / sc), t = fma(w, rcp, zp) (one rounding) differs from the
// defining t* = fl32(fl32(w / sc) + zp) by less than 2^-24 (4 |t| + 4 L + 4) (the reciprocal's
// and the quotient's roundings of |w / sc| <= |t| + L, the sums' of |t|), below the margin
// 2^-21 (|t| + 16) for L <= 15; so where t lies farther than the margin from every
// half-integer, rne(t) = rne(t*) and the cheap code is the exact one.  t is clamped to [0, L]
// first (the code's own clamp: no boundary is left at the ends, and a clamped t sits half a
// unit from the nearest one), then rounded to an integer by adding 1.5 2^23 (round to nearest
// even on the unit grid), whose bits give the code.  Within the margin the defining division
// decides (a few weights in ten thousand).
__device__ __forceinline__ uint32_t quant_code(float w, float sc, float rcp, float zp, float L)
{
    constexpr float kMagic = 12582912.0f; // 1.5 2^23
    const float tc = fminf(fmaxf(__fmaf_rn(w, rcp, zp), 0.0f), L);
    const float sm = __fadd_rn(tc, kMagic);
    const float r = __fsub_rn(sm, kMagic);
    uint32_t q = static_cast<uint32_t>(__float_as_int(sm) - __float_as_int(kMagic));
    // distance to the nearest half-integer: | |tc - r| - 1/2 |
    if (fabsf(__fsub_rn(fabsf(__fsub_rn(tc, r)), 0.5f)) <= __fmaf_rn(tc, 0x1p-21f, 0x1p-17f)) {
        const float re = rintf(__fadd_rn(__fdiv_rn(w, sc), zp));
        q = static_cast<uint32_t>(fminf(fmaxf(re, 0.0f), L));
    }
    return q;
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
__global__ void __launch_bounds__(256) quantize_kernel(const void *__restrict__ Wv,
                                                       const float *__restrict__ wsc,
                                                       uint8_t *__restrict__ packed,
                                                       uint16_t *__restrict__ S,
                                                       uint16_t *__restrict__ ZS, int V, int H)
{
    constexpr int P = 8 / BITS;                          // planes (codes per byte)
    constexpr float L = static_cast<float>((1 << BITS) - 1);
    constexpr float B = static_cast<float>(1 << BITS);
    const int lane = threadIdx.x & 31;
    const int PS = H / P;       // k stride between planes = packed bytes per row
    const int NS = PS / 128;    // spans per row
    const int NGt = H / G;      // groups per row
    // work items (n, s) = warp w, w + nwarps, ...: the position advances by (dn, ds) with no
    // division in the loop, and the next two items' weights are in flight while this one is
    // quantised (2 KB per warp: enough loads outstanding to cover the HBM latency)
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    const int dn = nwarps / NS, ds = nwarps - dn * NS;
    const int w0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    int n = w0 / NS, s = w0 - (w0 / NS) * NS;
    using Raw = typename std::conditional<kFp8, uint32_t, uint2>::type;
    auto load = [&](int rn, int rs, Raw (&raw)[P]) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if constexpr (kFp8) {
                const uint8_t *row = static_cast<const uint8_t *>(Wv) + static_cast<long long>(rn) * H;
                raw[p] = __ldg(reinterpret_cast<const uint32_t *>(row + p * PS + 128 * rs + 4 * lane));
            } else {
                const uint16_t *row = static_cast<const uint16_t *>(Wv) + static_cast<long long>(rn) * H;
                raw[p] = __ldg(reinterpret_cast<const uint2 *>(row + p * PS + 128 * rs + 4 * lane));
            }
        }
    };
    auto advance = [&](int &an, int &as) {
        an += dn;
        as += ds;
        if (as >= NS) {
            as -= NS;
            ++an;
        }
    };
    Raw raw[P], next[P];
    if (n < V) load(n, s, raw);
    int nn = n, ns = s;
    advance(nn, ns);
    if (nn < V) load(nn, ns, next);
    while (n < V) {
        int n2 = nn, s2 = ns;
        advance(n2, s2);
        Raw next2[P];
        if (n2 < V) load(n2, s2, next2);
        // four weights of each plane: k = p*PS + 128 s + 4 lane + i
        float wv[P][4];
        if constexpr (kFp8) {
            const float rs = __ldg(wsc + n);
#pragma unroll
            for (int p = 0; p < P; ++p)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    wv[p][i] = __fmul_rn(e4m3_to_f32(raw[p] >> (8 * i)), rs);
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                wv[p][0] = __uint_as_float(raw[p].x << 16);
                wv[p][1] = __uint_as_float(raw[p].x & 0xFFFF0000u);
                wv[p][2] = __uint_as_float(raw[p].y << 16);
                wv[p][3] = __uint_as_float(raw[p].y & 0xFFFF0000u);
            }
        }
        uint32_t word = 0;
        if constexpr (G == 128) {
            // the span's P groups each cover the whole warp: one reduction instruction per
            // extremum, then lane l computes the scale, zero point and reciprocal of group
            // l % P once (not every lane every group) and the others fetch them
            float lo[P], hi[P];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float *w = wv[p];
                lo[p] = warp_min_f32(fminf(fminf(w[0], w[1]), fminf(w[2], w[3])));
                hi[p] = warp_max_f32(fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3])));
            }
            const int gp = lane & (P - 1);
            float glo = lo[0], ghi = hi[0];
#pragma unroll
            for (int p = 1; p < P; ++p)
                if (gp == p) {
                    glo = lo[p];
                    ghi = hi[p];
                }
            const float gsc = fmaxf(__fdiv_rn(__fsub_rn(ghi, glo), L), 1e-8f);
            const float gzp = fminf(fmaxf(rintf(__fdiv_rn(-glo, gsc)), 0.0f), L);
            const float grcp = __frcp_rn(gsc);
            if (lane < P) {
                const float sb = __fmul_rn(B, gsc);
                const long long gi = static_cast<long long>(lane) * NS + s;
                S[static_cast<long long>(n) * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(sb));
                ZS[static_cast<long long>(n) * NGt + gi] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(sb, __fmul_rn(gzp, gsc))));
            }
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float sc = __shfl_sync(0xffffffffu, gsc, p);
                const float zp = __shfl_sync(0xffffffffu, gzp, p);
                const float rcp = __shfl_sync(0xffffffffu, grcp, p);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    word |= quant_code(wv[p][i], sc, rcp, zp, L) << (8 * i + BITS * p);
            }
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float *w = wv[p];
                float lo = fminf(fminf(w[0], w[1]), fminf(w[2], w[3]));
                float hi = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
                lo = lanes_min<G / 4>(lo);
                hi = lanes_max<G / 4>(hi);
                float sc = __fdiv_rn(__fsub_rn(hi, lo), L);
                sc = fmaxf(sc, 1e-8f);
                float zp = fminf(fmaxf(rintf(__fdiv_rn(-lo, sc)), 0.0f), L);
                const float rcp = __frcp_rn(sc);
#pragma unroll
                for (int i = 0; i < 4; ++i) word |= quant_code(w[i], sc, rcp, zp, L) << (8 * i + BITS * p);
                if ((lane & (G / 4 - 1)) == p) {
                    const float sb = __fmul_rn(B, sc);
                    const long long gi = (static_cast<long long>(p) * NS + s) * (128 / G) +
                                         lane / (G / 4);
                    S[static_cast<long long>(n) * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(sb));
                    ZS[static_cast<long long>(n) * NGt + gi] =
                        __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(sb, __fmul_rn(zp, sc))));
                }
            }
        }
        reinterpret_cast<uint32_t *>(packed + static_cast<long long>(n) * PS + 128 * s)[lane] = word;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            raw[p] = next[p];
            next[p] = next2[p];
        }
        n = nn;
        s = ns;
        nn = n2;
        ns = s2;
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
        float sc = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
        sc = fmaxf(sc, 1e-8f);
        const float zp = fminf(fmaxf(rintf(__fdiv_rn(-lo, sc)), 0.0f), 3.0f);
        const float rcp = __frcp_rn(sc);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) word |= quant_code(w[i], sc, rcp, zp, 3.0f) << (2 * i);
        if ((lane & 7) == 0) {
            const float s4 = __fmul_rn(4.0f, sc);
            const long long gi = 4LL * s + (lane >> 3);
            S[n * NGt + gi] = __bfloat16_as_ushort(__float2bfloat16_rn(s4));
            ZS[n * NGt + gi] =
                __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(s4, __fmul_rn(zp, sc))));
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
    const long long total = static_cast<long long>(V) * (H / (128 * (8 / BITS)));
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
