// dh_prep.cu -- step a2: group sums of x and the operand layouts of the coarse pass.
//
// xs[m, g] = sum_{k in group g} x[m, k] in fp32 (radiance_drafthead.py, _apply_head_int2:
// "xs = x.reshape(M, ng, GROUP).float().sum(-1)"), the zero-point term's multiplier.
//
// The 2-bit dequant turns bytes (0, 2) and (1, 3) of a packed 32-bit word into bf16 pairs, so
// the weight operand carries k in the order 4w+0, 4w+2, 4w+1, 4w+3 inside every aligned quad.
// The contraction order of an MMA is free as long as both operands agree, so x is staged with
// the same permutation (x'[4w + e] = x[4w + perm(e)], perm = 0, 2, 1, 3) in two layouts:
//   xt  [Npad, H]: plain K-major rows, the tcgen05 path's B operand (loaded by TMA);
//   xw  per 16-row batch chunk c, span s, plane p, n8-tile t: a 2 KB block holding the
//       mma.sync B fragments in register order, [j = 0..3][lane = 0..31][8 values] with
//       lane = 4 g + tig carrying x'[16c + 8t + g][p Q + 128 s + 32 tig + 8 j + 0..7].
// One thread handles one row and one octet of k (one 16-byte load, one or two 16-byte stores).
#include "dh_common.cuh"
#include "dh_internal.h"


namespace dh {

__device__ __forceinline__ uint4 permute_quads(uint4 v)
{
    // within each 32-bit pair of bf16 the order is (k, k+1); swap k+1 and k+2 of each quad
    uint4 o;
    o.x = __byte_perm(v.x, v.y, 0x5410); // (k0, k2)
    o.y = __byte_perm(v.x, v.y, 0x7632); // (k1, k3)
    o.z = __byte_perm(v.z, v.w, 0x5410); // (k4, k6)
    o.w = __byte_perm(v.z, v.w, 0x7632); // (k5, k7)
    return o;
}

__global__ void __launch_bounds__(256) prep_kernel(const uint16_t *__restrict__ x, int M, int H,
                                                   int rows, float *__restrict__ xs,
                                                   uint16_t *__restrict__ xw, int xw_rows,
                                                   int nt_per_chunk,
                                                   uint16_t *__restrict__ xt,
                                                   int *__restrict__ counters, int ncounters)
{
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid < ncounters) counters[tid] = 0;
    const int octs = H / 8;
    const long long total = static_cast<long long>(rows) * octs;
    // every thread of a 16-lane half-warp belongs to the same group: no early exit before the
    // shuffles, only predicated stores
    const bool live = tid < total;
    const int b = live ? static_cast<int>(tid / octs) : 0;
    const int o = live ? static_cast<int>(tid - static_cast<long long>(b) * octs) : 0;
    const int k0 = 8 * o;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (live && b < M) v = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<long long>(b) * H + k0));
    // group sum over 16 octets = 128 values
    float s = 0.f;
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            s += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xFFFF0000u);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (!live) return;
    const int NGt = H / kGroup;
    if ((o & 15) == 0) xs[static_cast<long long>(b) * NGt + (k0 >> 7)] = s;

    const uint4 pv = permute_quads(v);
    if (xt) *reinterpret_cast<uint4 *>(xt + static_cast<long long>(b) * H + k0) = pv;
    if (xw && b < xw_rows) {
        const int Q = H / 4, NG = H / 512;
        const int p = k0 / Q, rem = k0 - p * Q;
        const int sp = rem >> 7, r2 = rem & 127;
        const int tig = r2 >> 5, j = (r2 & 31) >> 3;
        const int c = b / kWarpBatch, t = (b % kWarpBatch) >> 3, g = b & 7;
        if (t < nt_per_chunk) {
            const int lane = 4 * g + tig;
            const long long blk =
                ((static_cast<long long>(c) * NG + sp) * 4 + p) * nt_per_chunk + t;
            const long long off = (blk * 4 + j) * 32 + lane;
            reinterpret_cast<uint4 *>(xw)[off] = pv;
        }
    }
}

cudaError_t launch_prep(const uint16_t *x, int M, int H, int Mpad, float *xs, uint16_t *xw,
                        uint16_t *xt, int Npad, int *counters, int ncounters,
                        cudaStream_t stream)
{
    int rows = Mpad > Npad ? Mpad : Npad;
    const int nt = (M <= 8) ? 1 : 2;
    const long long total = static_cast<long long>(rows) * (H / 8);
    long long threads = total > ncounters ? total : ncounters;
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    const int xw_rows = ((M + kWarpBatch - 1) / kWarpBatch) * kWarpBatch;
    prep_kernel<<<blocks, 256, 0, stream>>>(x, M, H, rows, xs, xw, xw_rows, nt, xt, counters,
                                            ncounters);
    return cudaGetLastError();
}

size_t warp_xw_elems(int M, int H)
{
    const int nt = (M <= 8) ? 1 : 2;
    const int chunks = (M + kWarpBatch - 1) / kWarpBatch;
    // per chunk: NG spans x 4 planes x nt tiles x 2 KB (1024 bf16)
    return static_cast<size_t>(chunks) * (H / 512) * 4 * nt * 1024;
}

// ------------------------------------------------------------------------------------------
// x staging for the 8-bit tcgen05 path.  Row m is scaled by 2^e (max |x 2^e| in [128, 256),
// exact) and written as three e4m3 terms, each the rounded residual of the ones before, scaled
// by its own power of two so that its largest magnitude lies in [128, 256):
//     r0 = x 2^e,  t1 = e4m3(r0),  r1 = r0 - t1,
//     t2 = e4m3(2^s2 r1),  r2 = r1 - 2^-s2 t2,  t3 = e4m3(2^s3 r2),
// so x 2^e ~ t1 + 2^-s2 t2 + 2^-s3 t3 (every difference is exact in fp32, no term saturates).
// Each term carries four significant bits of what the terms before left over, at the scale of
// the row's largest leftover: two terms represent every bf16 element of an ordinary row
// exactly (the ones that are not lie more than ~14 binades below the row maximum), and the
// third term covers rows whose elements span many more binades -- a few channels far above
// the rest lose nothing, since the large channels are exact in t1 and the rest get t2 and t3 at
// their own scale.  Term t of row m is row t MP + m of the staged operand.  The kernel also
// writes the group sums of the two- and three-term representations (scaled units), 2^-e, the
// term weights 2^-s2 and 2^-s3, and the number of terms the row needs: 3 when the two-term
// residual sum_k |r2_k| exceeds 2^-20 sum_k |x_k 2^e|, else 2 (each coarse launch takes the
// most any of its rows needs).  One CTA per staged row.
// ------------------------------------------------------------------------------------------
// Round to nearest even onto the e4m3 grid (three mantissa bits; normal exponents from -6, the
// subnormal spacing 2^-9 below 2^-6), for |r| < 448, in fp32 arithmetic: with 2^k <= |r| <
// 2^(k+1) (k at least -6), c = 1.5 2^(k+20) puts r + c in [2^(k+20), 2^(k+21)), whose spacing is
// e4m3's 2^(k-3) at r; the add rounds to nearest even on that grid (c is an even multiple of
// the spacing, 3 2^22 of them), and subtracting c again is exact.  The conversion units of an
// SM are few; these four operations run on the integer and fp32 pipes.
__device__ __forceinline__ float round_e4m3(float r)
{
    int ex = static_cast<int>((__float_as_uint(r) >> 23) & 0xFFu);
    ex = ex < 121 ? 121 : ex; // 121 = 127 - 6
    const float c = __uint_as_float((static_cast<uint32_t>(ex + 20) << 23) | 0x400000u);
    return __fsub_rn(__fadd_rn(r, c), c);
}

// The e4m3 bytes of two values already on the e4m3 grid (exact, no rounding): lo in bits 0-7,
// hi in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2_bits(float lo, float hi)
{
    uint16_t v;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(hi), "f"(lo));
    return v;
}

// The power of two 2^s that puts a largest magnitude mx > 0 in [128, 256) (s clamped to the
// normal fp32 exponents); s = 0 for mx = 0.
__device__ __forceinline__ int range_shift(float mx)
{
    if (!(mx > 0.f)) return 0;
    int ex;
    frexpf(mx, &ex); // mx = f 2^ex, f in [0.5, 1)
    const int s = 8 - ex;
    return s > 126 ? 126 : (s < -126 ? -126 : s);
}

__device__ __forceinline__ float pow2f(int s)
{
    return __int_as_float((s + 127) << 23);
}

constexpr int kPrepMaxThreads = 1024;
constexpr int kPrepOcts = 2; // 16-byte slices of x per thread: one per thread up to H = 8192,
                             // two up to H = 16384 (the CTA has min(H/8, 1024) threads)
constexpr float kTermsThreshold = 9.5367431640625e-7f; // 2^-20

// Largest value of v over the CTA (v >= 0); every thread gets it.  red: kPrepMaxThreads / 32.
// Every warp combines the warps' maxima with shuffles (one shared-memory read per lane).
__device__ __forceinline__ float cta_max(float v, float *red)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    __syncthreads(); // the previous use of red is over
    if (lane == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// The split of one scaled element r0 = x 2^e with term shifts s2, s3 (scales k2 = 2^s2 ...).
struct Split3 {
    float u[3];               // the terms as stored (e4m3 values, each at its own scale)
    float t1, t2, t3, r1, r2; // term values in the scaled units and the residuals
};

// The first two terms only (NT = 2) or all three; k2, k3 and their inverses are powers of two.
template <int NT>
__device__ __forceinline__ Split3 split3(float r0, float k2, float ik2, float k3, float ik3)
{
    Split3 o;
    o.u[0] = round_e4m3(r0);
    o.t1 = o.u[0];
    o.r1 = r0 - o.t1;
    o.u[1] = round_e4m3(o.r1 * k2);
    o.t2 = o.u[1] * ik2;
    o.r2 = o.r1 - o.t2;
    if constexpr (NT == 3) {
        o.u[2] = round_e4m3(o.r2 * k3);
        o.t3 = o.u[2] * ik3;
    } else {
        o.u[2] = 0.f;
        o.t3 = 0.f;
    }
    return o;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The coarse launches of one forward (batch chunks of up to 32 rows, padded to MP): one
// staging launch covers them all, block b staging row b - first[c] of chunk c.
constexpr int kMaxPrepChunks = 8; // 128 rows in chunks of 16
struct PrepChunks {
    int n;
    int first[kMaxPrepChunks + 1]; // first block of each chunk; first[n] = the grid
    int m0[kMaxPrepChunks], rows[kMaxPrepChunks], MP[kMaxPrepChunks];
    uint8_t *xt8[kMaxPrepChunks];  // the chunk's staged x
    float *small[kMaxPrepChunks];  // the chunk's group sums, row factors and term counts
};

// G: the group size of the sums (128, or 64 for the group-size ablation).
template <int G>
__global__ void __launch_bounds__(kPrepMaxThreads) prep_fp8_kernel(const uint16_t *__restrict__ x,
                                                                   int H, const PrepChunks ch,
                                                                   int *__restrict__ counters,
                                                                   int ncounters,
                                                                   uint16_t *__restrict__ xcopy)
{
    __shared__ float wred[kPrepMaxThreads / 32];
    __shared__ float wred2[kPrepMaxThreads / 32];
    __shared__ float wred3[kPrepMaxThreads / 32];
    // the coarse pass may be scheduled now: it waits for this grid before it reads x
    pdl_trigger();
    int c = 0;
    while (c + 1 < ch.n && static_cast<int>(blockIdx.x) >= ch.first[c + 1]) ++c;
    const int m = static_cast<int>(blockIdx.x) - ch.first[c];
    const int m0 = ch.m0[c], rows = ch.rows[c], MP = ch.MP[c];
    uint8_t *const xt8 = ch.xt8[c];
    float *const xs2 = ch.small[c];
    float *const xs3 = xs2 + static_cast<size_t>(kTc8MaxMP) * (H / 64);
    float *const row_f = xs2 + 2 * static_cast<size_t>(kTc8MaxMP) * (H / 64);
    int *const row_terms = reinterpret_cast<int *>(row_f + 3 * kTc8MaxMP);
    const bool valid = m < rows;
    const int octs = H / 8, NGt = H / G;
    if (counters && blockIdx.x == 0)
        for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0;
    const uint16_t *xr = x + static_cast<long long>(m0 + (valid ? m : 0)) * H;

    // the row stays in registers between the passes (H <= 1024 * 8 * kPrepOcts), and so do the
    // split's intermediate values: each pass takes one rounding further (the second slice of
    // every thread exists only when the row has more slices than the CTA has threads:
    // CTA-uniform)
    const int nj = octs > static_cast<int>(blockDim.x) ? 2 : 1;
    uint4 xv[kPrepOcts];
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        const int o = threadIdx.x + j * blockDim.x;
        xv[j] = make_uint4(0, 0, 0, 0);
        if (valid && o < octs) {
            xv[j] = __ldg(reinterpret_cast<const uint4 *>(xr) + o);
            if (xcopy)
                reinterpret_cast<uint4 *>(xcopy + static_cast<long long>(m0 + m) * H)[o] = xv[j];
        }
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
    const int e = range_shift(cta_max(mx, wred));
    const float scale = pow2f(e);

    // pass 2: r0 = x 2^e, its first term and residual; the largest residual -> s2
    float t1v[kPrepOcts][8], rv[kPrepOcts][8];
    float m1 = 0.f, l1 = 0.f; // and sum |x 2^e|
#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        if (j >= nj) break;
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float r0 = ((i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1])) * scale;
            t1v[j][i] = round_e4m3(r0);
            rv[j][i] = r0 - t1v[j][i];
            m1 = fmaxf(m1, fabsf(rv[j][i]));
            l1 += fabsf(r0);
        }
    }
    const int s2 = range_shift(cta_max(m1, wred));
    const float k2 = pow2f(s2), ik2 = pow2f(-s2);

    // pass 3: the second term of every residual, the residual after it (rv), the largest of
    // those -> s3, and the two sums that decide the row's term count, in one reduction
    float u2v[kPrepOcts][8];
    float m2 = 0.f, b2 = 0.f; // and the two-term residual sum |r2|
#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        if (j >= nj) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            u2v[j][i] = round_e4m3(rv[j][i] * k2);
            rv[j][i] = rv[j][i] - u2v[j][i] * ik2;
            m2 = fmaxf(m2, fabsf(rv[j][i]));
            b2 += fabsf(rv[j][i]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, off));
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        b2 += __shfl_xor_sync(0xffffffffu, b2, off);
    }
    __syncthreads(); // the previous use of wred is over
    if ((threadIdx.x & 31) == 0) {
        wred[threadIdx.x >> 5] = m2;
        wred2[threadIdx.x >> 5] = l1;
        wred3[threadIdx.x >> 5] = b2;
    }
    __syncthreads();
    {
        const int lane = threadIdx.x & 31;
        float v = lane < static_cast<int>(blockDim.x >> 5) ? wred[lane] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        m2 = v;
    }
    const int s3 = range_shift(m2);
    const float k3 = pow2f(s3), ik3 = pow2f(-s3);
    if (threadIdx.x == 0) {
        // per-row factors: 2^-e, then the weights of terms 2 and 3 (see the coarse kernel)
        row_f[m] = valid ? pow2f(-e) : 1.0f;
        row_f[kTc8MaxMP + m] = ik2;
        row_f[2 * kTc8MaxMP + m] = ik3;
        float L = 0.f, B = 0.f;
        for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) {
            L += wred2[i];
            B += wred3[i];
        }
        row_terms[m] = (valid && B > kTermsThreshold * L) ? 3 : 2;
    }

    // pass 4: the third terms, the terms' bytes and the group sums
#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        if (j >= nj) break; // CTA-uniform
        const int o = threadIdx.x + j * blockDim.x;
        // every lane of a warp takes part in the group shuffles: lanes past the row add 0
        const bool live = o < octs;
        float u[kTc8Terms][8];
        float sum2 = 0.f, sum3 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float t2 = u2v[j][i] * ik2;
            const float u3 = round_e4m3(rv[j][i] * k3);
            const float rep2 = t1v[j][i] + t2;
            sum2 += rep2;
            sum3 += rep2 + u3 * ik3;
            u[0][i] = t1v[j][i];
            u[1][i] = u2v[j][i];
            u[2][i] = u3;
        }
        // the terms' bytes, element i in byte i of the 8-byte slice
        uint32_t lo[kTc8Terms], hi[kTc8Terms];
#pragma unroll
        for (int t = 0; t < kTc8Terms; ++t) {
            lo[t] = e4m3x2_bits(u[t][0], u[t][1]) | (e4m3x2_bits(u[t][2], u[t][3]) << 16);
            hi[t] = e4m3x2_bits(u[t][4], u[t][5]) | (e4m3x2_bits(u[t][6], u[t][7]) << 16);
        }
        if (live)
#pragma unroll
            for (int t = 0; t < kTc8Terms; ++t)
                *reinterpret_cast<uint2 *>(xt8 + (static_cast<long long>(t) * MP + m) * H + 8 * o) =
                    make_uint2(lo[t], hi[t]);
        // the G / 8 octets of a group are consecutive lanes
#pragma unroll
        for (int off = G / 16; off > 0; off >>= 1) {
            sum2 += __shfl_xor_sync(0xffffffffu, sum2, off);
            sum3 += __shfl_xor_sync(0xffffffffu, sum3, off);
        }
        if (live && (o & (G / 8 - 1)) == 0) {
            xs2[static_cast<long long>(m) * NGt + o / (G / 8)] = sum2;
            xs3[static_cast<long long>(m) * NGt + o / (G / 8)] = sum3;
        }
    }
}

cudaError_t launch_prep_fp8(const uint16_t *x, int M, int H, int pack, const Tc8Workspace &w,
                            int *counters, int ncounters, cudaStream_t stream, uint16_t *xcopy)
{
    PrepChunks ch;
    ch.n = tc8_chunks(M, pack, H);
    if (ch.n > kMaxPrepChunks) return cudaErrorInvalidValue;
    int blocks = 0;
    for (int c = 0; c < ch.n; ++c) {
        const Tc8Chunk k = tc8_chunk(M, c, pack, H);
        ch.first[c] = blocks;
        ch.m0[c] = k.m0;
        ch.rows[c] = k.rows;
        ch.MP[c] = k.MP;
        ch.xt8[c] = w.xt8 + k.x_off;
        ch.small[c] = w.small + static_cast<size_t>(c) * tc8_small_floats(H);
        blocks += k.MP;
    }
    ch.first[ch.n] = blocks;
    auto kern = w.group == 64 ? prep_fp8_kernel<64> : prep_fp8_kernel<128>;
    // one thread per 16-byte slice of the row (a multiple of 32 threads)
    int threads = ((H / 8 + 31) / 32) * 32;
    if (threads > kPrepMaxThreads) threads = kPrepMaxThreads;
    kern<<<blocks, threads, 0, stream>>>(x, H, ch, counters, ncounters, xcopy);
    return cudaGetLastError();
}

} // namespace dh
