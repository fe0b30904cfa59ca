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

#include <cuda_fp16.h>
#include <cuda_fp8.h>

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
// exact) and split into T e4m3 terms by successive round-to-nearest: x1 = e4m3(x 2^e),
// x2 = e4m3(x 2^e - x1), x3 = e4m3(x 2^e - x1 - x2); every difference is exact in fp32.  A bf16
// value (8 significant bits) is represented exactly by two terms unless it lies more than 10
// binades below the row maximum; the third term shrinks that residual to below 2^-18 of the
// maximum.  Term t of row m is row t*MP + m of the staged operand.  xs receives the group
// sums of the represented values x1 + x2 + x3 (scaled units) and inv_scale the factor 2^-e.
// One CTA per staged row.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float e4m3_to_f32(__nv_fp8_storage_t v)
{
    const __half_raw h = __nv_cvt_fp8_to_halfraw(v, __NV_E4M3);
    return __half2float(__half(h));
}

constexpr int kPrepMaxThreads = 1024;
constexpr int kPrepOcts = 2; // 16-byte slices of x per thread: one per thread up to H = 8192,
                             // two up to H = 16384 (the CTA has min(H/8, 1024) threads)

// G: the group size of the sums xs (128, or 64 for the group-size ablation).
template <int G>
__global__ void __launch_bounds__(kPrepMaxThreads) prep_fp8_kernel(const uint16_t *__restrict__ x,
                                                                   int H,
                                                       int m0, int rows, int MP, int T,
                                                       uint8_t *__restrict__ xt8,
                                                       float *__restrict__ xs,
                                                       float *__restrict__ inv_scale,
                                                       int *__restrict__ counters, int ncounters)
{
    __shared__ float wmax[kPrepMaxThreads / 32];
    const int m = blockIdx.x;
    const bool valid = m < rows;
    const int octs = H / 8, NGt = H / G;
    if (counters && m == 0)
        for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0;
    const uint16_t *xr = x + static_cast<long long>(m0 + (valid ? m : 0)) * H;

    // the row stays in registers between the max and the split (H <= 1024 * 8 * kPrepOcts)
    uint4 xv[kPrepOcts];
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        const int o = threadIdx.x + j * blockDim.x;
        xv[j] = make_uint4(0, 0, 0, 0);
        if (valid && o < octs) xv[j] = __ldg(reinterpret_cast<const uint4 *>(xr) + o);
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                 fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, wmax[i]);
    int e = 0;
    if (mx > 0.f) {
        int ex;
        frexpf(mx, &ex); // mx = f 2^ex, f in [0.5, 1)
        e = 8 - ex;      // mx 2^e in [128, 256)
        e = e > 126 ? 126 : (e < -126 ? -126 : e);
    }
    const float scale = __int_as_float((e + 127) << 23);
    if (threadIdx.x == 0) inv_scale[m] = valid ? __int_as_float((127 - e) << 23) : 1.0f;

#pragma unroll
    for (int j = 0; j < kPrepOcts; ++j) {
        const int o = threadIdx.x + j * blockDim.x;
        if (o >= octs) break;
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        uint32_t lo[3] = {0, 0, 0}, hi[3] = {0, 0, 0};
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float xe = (i & 1) ? __uint_as_float(w[i >> 1] & 0xFFFF0000u)
                                     : __uint_as_float(w[i >> 1] << 16);
            float r = xe * scale; // exact: a power of two
            float rep = 0.f;
#pragma unroll
            for (int t = 0; t < 3; ++t) {
                if (t < T) {
                    const __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3);
                    const float bf = e4m3_to_f32(b);
                    r -= bf;
                    rep += bf;
                    if (i < 4) lo[t] |= static_cast<uint32_t>(b) << (8 * i);
                    else hi[t] |= static_cast<uint32_t>(b) << (8 * (i - 4));
                }
            }
            sum += rep;
        }
        for (int t = 0; t < T; ++t)
            *reinterpret_cast<uint2 *>(xt8 + (static_cast<long long>(t) * MP + m) * H + 8 * o) =
                make_uint2(lo[t], hi[t]);
        // the G / 8 octets of a group are consecutive lanes
#pragma unroll
        for (int off = G / 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if ((o & (G / 8 - 1)) == 0) xs[static_cast<long long>(m) * NGt + o / (G / 8)] = sum;
    }
}

cudaError_t launch_prep_fp8(const uint16_t *x, int M, int H, const Tc8Workspace &w,
                            int *counters, int ncounters, cudaStream_t stream)
{
    for (int c = 0; c < tc8_chunks(M); ++c) {
        const Tc8Chunk k = tc8_chunk(M, c);
        auto kern = w.group == 64 ? prep_fp8_kernel<64> : prep_fp8_kernel<128>;
        // one thread per 16-byte slice of the row (a multiple of 32 threads)
        int threads = ((H / 8 + 31) / 32) * 32;
        if (threads > kPrepMaxThreads) threads = kPrepMaxThreads;
        kern<<<k.MP, threads, 0, stream>>>(
            x, H, k.m0, k.rows, k.MP, k.T, w.xt8 + static_cast<size_t>(c) * w.chunk_bytes,
            w.xs + static_cast<size_t>(c) * w.xs_chunk,
            w.inv_scale + static_cast<size_t>(c) * kTc8MaxRows, c == 0 ? counters : nullptr,
            ncounters);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace dh
