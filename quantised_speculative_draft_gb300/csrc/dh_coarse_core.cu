// dh_coarse_core.cu -- kernels (2)+(3) for small batches on the CUDA cores: the coarse pass
// as fp32 FMAs on weights built from the packed bits, with the fused block top-KCAND
// epilogue.
//
// radiance_drafthead.py, _draft_head_int2 (the coarse value), the docstring's bit-pattern
// dequant bullet (weights made from the packed bits by integer ops, no lookup) and _emit (a
// block's KCAND best).  For batch row m and vocabulary row n
//     c[m, n] = sum_g ( S[n, g] p[m, n, g] - ZS[n, g] xs[m, g] ),
//     p[m, n, g] = sum_{k in g} x[m, k] (1 + v[n, k] / 4).
//
// Layout of the work (M <= 4)
//   * one work item = one selection block of 64 vocabulary rows, owned by one warp; lane l
//     owns rows l and l + 32, so each row's whole dot product stays in one thread and the
//     block's KCAND best come out of warp shuffles; items are handed out by an atomic counter;
//   * the packed rows stream through the warp's ring of 8 KB TMA stages ([64 rows x 128 B],
//     128-byte swizzle), one 128-byte chunk c of every row per stage.  Byte j of chunk c holds
//     the codes of k = p Q + 128 c + j for the four planes p (Q = H / 4), so a stage carries
//     exactly one group of each plane: groups p H/512 + c;
//   * x is held in shared memory as fp32 [MP, H]; every lane reads the same x words, so each
//     16-byte x load is a broadcast that serves two rows of all 32 lanes;
//   * dequant: a shift of the 32-bit word by 15 - 8 t puts byte t's four codes at bits
//     15 + 2 p; and-ing with code p's two bits and or-ing in the bits of 1.0f gives the
//     exact fp32 value 1 + v 2^(2 p - 8) (one shift per byte, one LOP3 per weight), and one
//     FADD2 per pair takes the 1 off again, exactly: w = v 2^(2 p - 8);
//   * FFMA2 accumulates x w in fp32 pairs, so a plane's group partial is P = 2^(2 p - 8) d
//     with d = sum x v -- the same magnitudes, hence the same rounding, as the dot product
//     with the codes themselves (an accumulator that also carried sum x, as 1 + v/4 weights
//     would, rounds at the scale of the row's largest element and fails on outlier rows);
//   * the group term folds on the accumulator:
//     S p - ZS xs = 2^(6 - 2 p) S P + (S - ZS) xs   (p = xs + d / 4).
#include "dh_common.cuh"
#include "dh_internal.h"

#include <climits>

namespace dh {

namespace {

constexpr int kCoreStage = kBlockN * kSpanBytes; // 8 KB: 64 rows x 128 packed bytes
constexpr int kCoreSmemLimit = 232448;           // 227 KB opt-in per block
constexpr int kCoreMaxWarps = 16;
// MP = 4 keeps 64 accumulators per thread: 8 warps leave it the registers it needs (its x
// rows take 80 KB of shared memory at H = 5120, so more than 9 warps would not fit anyway)
constexpr int core_max_warps(int MP) { return MP >= 4 ? 8 : kCoreMaxWarps; }
constexpr uint32_t kOneBits = 0x3F800000u;       // fp32 1.0

struct CoreParams {
    const uint16_t *x;   // [M, H] bf16
    const float *xs;     // [>= MP, NGt] group sums
    const uint16_t *S;
    const uint16_t *ZS;
    int M, V, H, kcand, nitems, nstage;
    long long ncand;     // nblk * kcand (row stride of the candidate arrays)
    float *cand_val;
    int32_t *cand_idx;
    float *coarse;
    int *counter;
    int *timeout_flag;
};

__device__ __forceinline__ uint4 lds_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t word_at(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// The fp32 value 1 + v 2^(2p - 8) of plane p's code from a word already shifted for its byte.
template <int P>
__device__ __forceinline__ float weight_of(uint32_t shifted)
{
    return __uint_as_float((shifted & (3u << (15 + 2 * P))) | kOneBits);
}

// One 32-bit word (bytes t = 0..3, four codes each) of rows a and b, plane P: the weights
// v 2^(2P - 8) against x[m, P Q + k0 + t], accumulated in pairs (t = 0, 1) and (2, 3).
template <int MP, int P>
__device__ __forceinline__ void word_plane(const uint32_t (&sa)[4], const uint32_t (&sb)[4],
                                           uint32_t xaddr, uint32_t xrow_bytes,
                                           float2 (&acc)[2][4][MP])
{
    // (1 + v 2^(2p-8)) - 1 is exact (both operands within a factor of two of each other, or v = 0)
    const float2 neg1 = make_float2(-1.f, -1.f);
    const float2 a01 = __fadd2_rn(make_float2(weight_of<P>(sa[0]), weight_of<P>(sa[1])), neg1);
    const float2 a23 = __fadd2_rn(make_float2(weight_of<P>(sa[2]), weight_of<P>(sa[3])), neg1);
    const float2 b01 = __fadd2_rn(make_float2(weight_of<P>(sb[0]), weight_of<P>(sb[1])), neg1);
    const float2 b23 = __fadd2_rn(make_float2(weight_of<P>(sb[2]), weight_of<P>(sb[3])), neg1);
#pragma unroll
    for (int m = 0; m < MP; ++m) {
        const float4 xv = lds_f4(xaddr + m * xrow_bytes);
        const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
        acc[0][P][m] = __ffma2_rn(x01, a01, acc[0][P][m]);
        acc[0][P][m] = __ffma2_rn(x23, a23, acc[0][P][m]);
        acc[1][P][m] = __ffma2_rn(x01, b01, acc[1][P][m]);
        acc[1][P][m] = __ffma2_rn(x23, b23, acc[1][P][m]);
    }
}

template <int MP>
__global__ void __launch_bounds__(32 * core_max_warps(MP), 1)
    coarse_core_kernel(const __grid_constant__ CUtensorMap tm_packed, const CoreParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int H = prm.H, Q = H / 4, NG = H / 512, NGt = H / kGroup;
    const int nstage = prm.nstage;

    // ---- shared memory: rings | x fp32 [MP][H] | xs [MP][NGt] | barriers -----------------
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const smem = smem_raw + (base - raw);
    uint8_t *const rings = smem;
    float *const x_s = reinterpret_cast<float *>(rings + static_cast<size_t>(nwarps) * nstage * kCoreStage);
    float *const xs_s = x_s + MP * H;
    uint64_t *const bars = reinterpret_cast<uint64_t *>(xs_s + ((MP * NGt + 1) & ~1));

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_packed);
        for (int i = 0; i < nwarps * nstage; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    // x as fp32 (rows >= M zero); x is the caller's input, so this needs no wait on the
    // staging kernel that precedes this one in the stream
    const int octs = H / 8;
    for (int i = threadIdx.x; i < MP * octs; i += blockDim.x) {
        const int m = i / octs, o = i - m * octs;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m < prm.M) v = __ldg(reinterpret_cast<const uint4 *>(prm.x + static_cast<long long>(m) * H) + o);
        float4 lo, hi;
        lo.x = __uint_as_float(v.x << 16);
        lo.y = __uint_as_float(v.x & 0xFFFF0000u);
        lo.z = __uint_as_float(v.y << 16);
        lo.w = __uint_as_float(v.y & 0xFFFF0000u);
        hi.x = __uint_as_float(v.z << 16);
        hi.y = __uint_as_float(v.z & 0xFFFF0000u);
        hi.z = __uint_as_float(v.w << 16);
        hi.w = __uint_as_float(v.w & 0xFFFF0000u);
        reinterpret_cast<float4 *>(x_s + m * H)[2 * o] = lo;
        reinterpret_cast<float4 *>(x_s + m * H)[2 * o + 1] = hi;
    }
    // the group sums and the zeroed work counter are written by the staging kernel
    pdl_wait();
    for (int i = threadIdx.x; i < MP * NGt; i += blockDim.x) xs_s[i] = prm.xs[i];
    __syncthreads();

    uint64_t *const my_bars = bars + warp * nstage;
    uint8_t *const my_ring = rings + static_cast<size_t>(warp) * nstage * kCoreStage;
    const uint64_t policy = l2_policy_evict_first();

    auto fetch = [&]() -> int {
        int it = 0;
        if (lane == 0) it = atomicAdd(prm.counter, 1);
        return __shfl_sync(0xffffffffu, it, 0);
    };

    // Items in flight: q0 is being consumed, q1 is the next one (or -1 before it is fetched).
    // Loads run at most one item ahead of consumption and at most nstage chunks ahead.
    int q0 = fetch(), q1 = -1;
    int is_item = q0, is_chunk = 0;
    uint32_t issued = 0, consumed = 0;
    auto try_issue = [&]() -> bool {
        if (is_chunk == NG) {
            if (is_item != q0) return false;
            if (q1 < 0) q1 = fetch();
            is_item = q1;
            is_chunk = 0;
        }
        if (is_item >= prm.nitems) return false;
        const uint32_t slot = issued % nstage;
        if (lane == 0) {
            mbar_arrive_expect_tx(&my_bars[slot], kCoreStage);
            tma_load_2d_hint(my_ring + slot * kCoreStage, &tm_packed, is_chunk * kSpanBytes,
                             is_item * kBlockN, &my_bars[slot], policy);
        }
        ++issued;
        ++is_chunk;
        return true;
    };
    while (issued < consumed + nstage && try_issue()) {
    }

    const uint32_t x_base = smem_u32(x_s);
    const uint32_t xrow_bytes = static_cast<uint32_t>(H) * 4u;
    const int sw = lane & 7; // (lane + 32) & 7 too: both rows share the swizzle phase
    bool failed = false;

    while (q0 < prm.nitems) {
        const int item = q0;
        const int row0 = item * kBlockN;
        float tot[2][MP];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int m = 0; m < MP; ++m) tot[r][m] = 0.f;

        for (int c = 0; c < NG; ++c) {
            const uint32_t slot = consumed % nstage;
            const uint32_t parity = (consumed / nstage) & 1u;
            // every lane polls the same barrier; the vote keeps the warp together if one lane's
            // bound ran out while another saw the phase complete
            const bool ok_wait = mbar_wait_bounded(&my_bars[slot], parity, prm.timeout_flag);
            if (__any_sync(0xffffffffu, !ok_wait)) {
                failed = true;
                break;
            }
            const uint32_t st = smem_u32(my_ring + slot * kCoreStage);
            const uint32_t ra = st + lane * kSpanBytes, rb = ra + 32 * kSpanBytes;
            float2 acc[2][4][MP];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int p = 0; p < 4; ++p)
#pragma unroll
                    for (int m = 0; m < MP; ++m) acc[r][p][m] = make_float2(0.f, 0.f);

            // x[m, p Q + 128 c + 16 q + 4 w + t] for word w of 16-byte piece q
            const uint32_t xc = x_base + static_cast<uint32_t>(128 * c) * 4u;
#pragma unroll 2
            for (int q = 0; q < 8; ++q) {
                const uint4 pa = lds_u4(ra + ((q ^ sw) << 4));
                const uint4 pb = lds_u4(rb + ((q ^ sw) << 4));
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t wa = word_at(pa, w), wb = word_at(pb, w);
                    const uint32_t sa[4] = {wa << 15, wa << 7, wa >> 1, wa >> 9};
                    const uint32_t sb[4] = {wb << 15, wb << 7, wb >> 1, wb >> 9};
                    const uint32_t xk = xc + static_cast<uint32_t>(16 * q + 4 * w) * 4u;
                    const uint32_t xq = static_cast<uint32_t>(Q) * 4u;
                    word_plane<MP, 0>(sa, sb, xk, xrow_bytes, acc);
                    word_plane<MP, 1>(sa, sb, xk + xq, xrow_bytes, acc);
                    word_plane<MP, 2>(sa, sb, xk + 2 * xq, xrow_bytes, acc);
                    word_plane<MP, 3>(sa, sb, xk + 3 * xq, xrow_bytes, acc);
                }
            }
            // all lanes' reads of this stage are done before lane 0 refills it
            fence_proxy_async_smem();
            __syncwarp();
            ++consumed;
            while (issued < consumed + nstage && try_issue()) {
            }

            // fold the four groups of this chunk: 2^(6-2p) S P + (S - ZS) xs
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int n = row0 + lane + 32 * r;
                const bool ok = n < prm.V;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int gi = p * NG + c;
                    float s = 0.f, z = 0.f;
                    if (ok) {
                        s = bf16_bits_to_f32(__ldg(prm.S + static_cast<long long>(n) * NGt + gi));
                        z = bf16_bits_to_f32(__ldg(prm.ZS + static_cast<long long>(n) * NGt + gi));
                    }
                    const float al = s * static_cast<float>(1 << (6 - 2 * p));
                    const float sz = s - z;
#pragma unroll
                    for (int m = 0; m < MP; ++m) {
                        const float xsv = xs_s[m * NGt + gi];
                        const float P = acc[r][p][m].x + acc[r][p][m].y;
                        tot[r][m] = fmaf(al, P, fmaf(sz, xsv, tot[r][m]));
                    }
                }
            }
        }
        if (failed) break;

        if (prm.coarse) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int n = row0 + lane + 32 * r;
#pragma unroll
                for (int m = 0; m < MP; ++m)
                    if (n < prm.V && m < prm.M)
                        prm.coarse[static_cast<long long>(m) * prm.V + n] = tot[r][m];
            }
        }
        // the block's KCAND best per batch row, best first, equal values -> lower row
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            if (m >= prm.M) break;
            const int n0 = row0 + lane, n1 = n0 + 32;
            float v0 = n0 < prm.V ? tot[0][m] : -INFINITY;
            float v1 = n1 < prm.V ? tot[1][m] : -INFINITY;
            int i0 = n0 < prm.V ? n0 : INT_MAX;
            int i1 = n1 < prm.V ? n1 : INT_MAX;
            const long long off = static_cast<long long>(m) * prm.ncand +
                                  static_cast<long long>(item) * prm.kcand;
            for (int k = 0; k < prm.kcand; ++k) {
                float bv = v0;
                int bi = i0;
                if (better(v1, i1, bv, bi)) {
                    bv = v1;
                    bi = i1;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if (bi != INT_MAX) {
                    if (i0 == bi) {
                        v0 = -INFINITY;
                        i0 = INT_MAX;
                    } else if (i1 == bi) {
                        v1 = -INFINITY;
                        i1 = INT_MAX;
                    }
                }
                if (lane == 0) {
                    const bool valid = bi != INT_MAX;
                    prm.cand_val[off + k] = valid ? bv : -INFINITY;
                    prm.cand_idx[off + k] = valid ? bi : -1;
                }
            }
        }
        if (q1 < 0) q1 = fetch();
        q0 = q1;
        q1 = -1;
    }
    // the selection kernel that follows in the stream may start its prologue
    pdl_trigger();
}

struct CoreGeometry {
    int MP = 0, nwarps = 0, nstage = 0;
    size_t smem = 0;
};

CoreGeometry core_geometry(int M, int H)
{
    CoreGeometry g;
    if (M < 1 || M > 4 || H < 512 || H % 512 != 0) return g;
    g.MP = M <= 1 ? 1 : (M <= 2 ? 2 : 4);
    const int NGt = H / kGroup;
    const size_t fixed = 1024 /*alignment slack*/ + static_cast<size_t>(g.MP) * H * 4 +
                         static_cast<size_t>((g.MP * NGt + 1) & ~1) * 4 +
                         8 * 2 * kCoreMaxWarps /*barriers*/;
    g.nstage = 2; // one stage in flight per warp: 8 KB x 8+ warps covers the HBM latency
    const long long room = kCoreSmemLimit - static_cast<long long>(fixed);
    int nw = room > 0 ? static_cast<int>(room / (static_cast<long long>(g.nstage) * kCoreStage)) : 0;
    if (nw > core_max_warps(g.MP)) nw = core_max_warps(g.MP);
    if (nw < 4) return CoreGeometry{};
    g.nwarps = nw;
    g.smem = fixed + static_cast<size_t>(nw) * g.nstage * kCoreStage;
    return g;
}

template <int MP>
cudaError_t launch_mp(const CoarseArgs &a, const CUtensorMap &tm, const CoreGeometry &g,
                      cudaStream_t stream)
{
    static PerDeviceOnce attr;
    cudaError_t err = attr.run([] {
        return cudaFuncSetAttribute(coarse_core_kernel<MP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kCoreSmemLimit);
    });
    if (err != cudaSuccess) return err;
    const int nblk = (a.V + kBlockN - 1) / kBlockN;
    CoreParams prm;
    prm.x = a.x;
    prm.xs = a.xs;
    prm.S = a.S;
    prm.ZS = a.ZS;
    prm.M = a.M;
    prm.V = a.V;
    prm.H = a.H;
    prm.kcand = a.kcand;
    prm.nitems = nblk;
    prm.nstage = g.nstage;
    prm.ncand = static_cast<long long>(nblk) * a.kcand;
    prm.cand_val = a.cand_val;
    prm.cand_idx = a.cand_idx;
    prm.coarse = a.coarse;
    prm.counter = a.counters;
    prm.timeout_flag = a.timeout_flag;
    const int sms = device_sm_count();
    const int grid = nblk < sms ? nblk : sms;
    return launch_pdl(coarse_core_kernel<MP>, dim3(grid), dim3(32 * g.nwarps), g.smem, stream,
                      tm, prm);
}

} // namespace

bool core_supported(int M, int H) { return core_geometry(M, H).nwarps > 0; }

cudaError_t launch_coarse_core(const CoarseArgs &a, cudaStream_t stream)
{
    const CoreGeometry g = core_geometry(a.M, a.H);
    if (g.nwarps == 0) return cudaErrorInvalidConfiguration;
    CUtensorMap tm;
    CUresult r = encode_tensor_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                      const_cast<uint8_t *>(a.packed), a.H / 4, a.V, a.H / 4,
                                      kSpanBytes, kBlockN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (g.MP == 1) return launch_mp<1>(a, tm, g, stream);
    if (g.MP == 2) return launch_mp<2>(a, tm, g, stream);
    return launch_mp<4>(a, tm, g, stream);
}

int core_mpad(int M) { return M <= 1 ? 1 : (M <= 2 ? 2 : 4); }

} // namespace dh
