// dh_coarse_warp.cu -- kernels (2)+(3), warp-level path: coarse pass on mma.sync tensor cores
// with the fused block top-KCAND epilogue.
//
// radiance_drafthead.py, _draft_head_int2 and _emit.  For a vocabulary row n and batch row m:
//     c[m, n] = sum_g ( S[n, g] * p[m, n, g] - ZS[n, g] * xs[m, g] ),
//     p[m, n, g] = sum_{k in g} x[m, k] * (1 + v[n, k] / 4)
// where (1 + v/4) is produced straight from the packed bits (bit-pattern dequant) and the
// scale and zero are applied to the fp32 accumulator once per group, never to the weight.
// Every block of 64 vocabulary rows then emits its KCAND best (value, row) pairs per batch
// row, best first, equal values -> lower row (the first maximum, as _emit's argmax).
//
// GB300 layout of the work
//   * one work item = one selection block = 64 vocabulary rows x all of H, owned by one warp;
//     items are handed out by an atomic counter, so warps stay busy until the head is done;
//   * each warp streams its packed rows through its own ring of 8 KB TMA stages
//     ([64 rows x 128 bytes], 128-byte swizzle; 128 bytes of a row = one pass over the four
//     planes of one span), issued by lane 0 and tracked by one mbarrier per stage;
//   * the batch operand x (16 rows at a time, quad-permuted, in mma.sync fragment order) stays
//     resident in shared memory for the whole kernel, so HBM sees only the weight stream;
//   * swap-AB mma.sync m16n8k16: A = 16 dequantised vocabulary rows, B = 8 batch rows; per
//     plane a warp runs 8 k-steps x 4 m-tiles x NT n-tiles, then folds the group's partial p
//     into the running accumulator with its scale and zero.
#include "dh_common.cuh"
#include "dh_internal.h"

#include <climits>

namespace dh {

namespace {

constexpr int kStageBytes = kWarpRowsPerWarp * kSpanBytes; // 8 KB
constexpr int kSmemLimit = 232448;                          // 227 KB opt-in per block
constexpr int kMaxWarpsPerCta = 8;

struct WarpParams {
    const uint4 *xw;     // this chunk's B-fragment operand
    const float *xs;     // [rows, NGt], rows of this chunk start at m0
    const uint16_t *S;
    const uint16_t *ZS;
    int V, H, m0, mrows, kcand, nitems, nstage;
    long long ncand;     // nblk * kcand (row stride of the candidate arrays)
    float *cand_val;
    int32_t *cand_idx;
    float *coarse;
    int *counter;
    int *timeout_flag;
    uint32_t xw_bytes;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int NT, int P>
__device__ __forceinline__ void plane_pass(const uint4 (&pk)[4][2][2], uint32_t xw_plane,
                                           int lane, float (&p)[4][NT][4])
{
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) p[mt][nt][i] = 0.f;
    uint4 xb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) xb[nt][j] = lds128(xw_plane + ((nt * 4 + j) * 32 + lane) * 16);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const uint32_t w0 = word_of(pk[mt][0][s >> 2], s & 3); // row g
            const uint32_t w1 = word_of(pk[mt][1][s >> 2], s & 3); // row g + 8
            const uint32_t a0 = deq_pair_even<P>(w0);
            const uint32_t a1 = deq_pair_even<P>(w1);
            const uint32_t a2 = deq_pair_odd<P>(w0);
            const uint32_t a3 = deq_pair_odd<P>(w1);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 &b = xb[nt][s >> 1];
                const uint32_t b0 = (s & 1) ? b.z : b.x;
                const uint32_t b1 = (s & 1) ? b.w : b.y;
                mma_bf16_16816(p[mt][nt], a0, a1, a2, a3, b0, b1);
            }
        }
    }
}

template <int NT>
__device__ __forceinline__ void plane_epilogue(const float (&p)[4][NT][4], float (&acc)[4][NT][4],
                                               const WarpParams &prm, int row0, int g, int tig,
                                               int gi, int NGt, const float *xs_s)
{
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
        const int r0 = row0 + 16 * mt + g, r1 = r0 + 8;
        float s0 = 0.f, z0 = 0.f, s1 = 0.f, z1 = 0.f;
        if (r0 < prm.V) {
            s0 = bf16_bits_to_f32(__ldg(prm.S + static_cast<long long>(r0) * NGt + gi));
            z0 = bf16_bits_to_f32(__ldg(prm.ZS + static_cast<long long>(r0) * NGt + gi));
        }
        if (r1 < prm.V) {
            s1 = bf16_bits_to_f32(__ldg(prm.S + static_cast<long long>(r1) * NGt + gi));
            z1 = bf16_bits_to_f32(__ldg(prm.ZS + static_cast<long long>(r1) * NGt + gi));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c0 = 8 * nt + 2 * tig;
            const float x0 = xs_s[c0 * (NGt + 1) + gi];
            const float x1 = xs_s[(c0 + 1) * (NGt + 1) + gi];
            acc[mt][nt][0] = fmaf(s0, p[mt][nt][0], fmaf(-z0, x0, acc[mt][nt][0]));
            acc[mt][nt][1] = fmaf(s0, p[mt][nt][1], fmaf(-z0, x1, acc[mt][nt][1]));
            acc[mt][nt][2] = fmaf(s1, p[mt][nt][2], fmaf(-z1, x0, acc[mt][nt][2]));
            acc[mt][nt][3] = fmaf(s1, p[mt][nt][3], fmaf(-z1, x1, acc[mt][nt][3]));
        }
    }
}

// Block top-KCAND over the warp's 64 rows for each of its batch columns.  Thread (g, tig)
// holds rows 16 mt + g + 8 h of columns 8 nt + 2 tig + e; the 8 lanes sharing tig hold one
// column's 64 values.
template <int NT>
__device__ __forceinline__ void emit_block(float (&acc)[4][NT][4], const WarpParams &prm,
                                           int item, int g, int tig)
{
    const int row0 = item * kWarpRowsPerWarp;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 8 * nt + 2 * tig + e;
            float v[8];
            int r[8];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = row0 + 16 * mt + g + 8 * h;
                    const bool ok = row < prm.V;
                    v[mt * 2 + h] = ok ? acc[mt][nt][2 * h + e] : -INFINITY;
                    r[mt * 2 + h] = ok ? row : INT_MAX;
                }
            const bool col_ok = col < prm.mrows;
            const long long base =
                static_cast<long long>(prm.m0 + col) * prm.ncand + static_cast<long long>(item) * prm.kcand;
            for (int k = 0; k < prm.kcand; ++k) {
                float bv = v[0];
                int bi = r[0];
#pragma unroll
                for (int i = 1; i < 8; ++i)
                    if (better(v[i], r[i], bv, bi)) {
                        bv = v[i];
                        bi = r[i];
                    }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (r[i] == bi) {
                        v[i] = -INFINITY;
                        r[i] = INT_MAX;
                    }
                if (g == 0 && col_ok) {
                    const bool valid = bi != INT_MAX;
                    prm.cand_val[base + k] = valid ? bv : -INFINITY;
                    prm.cand_idx[base + k] = valid ? bi : -1;
                }
            }
        }
}

template <int NT>
__global__ void __launch_bounds__(32 * kMaxWarpsPerCta, 1)
    coarse_warp_kernel(const __grid_constant__ CUtensorMap tm_packed, const WarpParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const int NGt = prm.H / kGroup, NG = prm.H / 512;
    const int nstage = prm.nstage;

    // ---- shared memory carve-up -------------------------------------------------------
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const smem = smem_raw + (base - raw);
    uint8_t *const rings = smem;                                   // nwarps*nstage*8 KB
    uint8_t *const xw_s = rings + static_cast<size_t>(nwarps) * nstage * kStageBytes;
    float *const xs_s = reinterpret_cast<float *>(xw_s + prm.xw_bytes); // [8NT][NGt+1]
    const int xs_floats = (8 * NT * (NGt + 1) + 1) & ~1;                 // keep 8-byte alignment
    uint64_t *const bars = reinterpret_cast<uint64_t *>(xs_s + xs_floats);
    uint64_t *const xw_bar = bars + nwarps * nstage;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_packed);
        for (int i = 0; i < nwarps * nstage; ++i) mbar_init(&bars[i], 1);
        mbar_init(xw_bar, 1);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < 8 * NT * NGt; i += blockDim.x) {
        const int row = i / NGt, gg = i - row * NGt;
        xs_s[row * (NGt + 1) + gg] = prm.xs[static_cast<long long>(prm.m0 + row) * NGt + gg];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(xw_bar, prm.xw_bytes);
        bulk_load(xw_s, prm.xw, prm.xw_bytes, xw_bar);
    }

    uint64_t *const my_bars = bars + warp * nstage;
    uint8_t *const my_ring = rings + static_cast<size_t>(warp) * nstage * kStageBytes;
    const uint64_t policy = l2_policy_evict_first();

    auto fetch = [&]() -> int {
        int it = 0;
        if (lane == 0) it = atomicAdd(prm.counter, 1);
        return __shfl_sync(0xffffffffu, it, 0);
    };

    // Items in flight: q0 is being consumed, q1 is the next one (or -1 before it is fetched).
    // Loads are issued at most one item ahead of consumption and at most nstage spans ahead.
    int q0 = fetch(), q1 = -1;
    int is_item = q0, is_span = 0;
    uint32_t issued = 0, consumed = 0;
    auto try_issue = [&]() -> bool {
        if (is_span == NG) {
            if (is_item != q0) return false;
            if (q1 < 0) q1 = fetch();
            is_item = q1;
            is_span = 0;
        }
        if (is_item >= prm.nitems) return false;
        const uint32_t slot = issued % nstage;
        if (lane == 0) {
            mbar_arrive_expect_tx(&my_bars[slot], kStageBytes);
            tma_load_2d_hint(my_ring + slot * kStageBytes, &tm_packed, is_span * kSpanBytes,
                             is_item * kWarpRowsPerWarp, &my_bars[slot], policy);
        }
        ++issued;
        ++is_span;
        return true;
    };
    while (issued < consumed + nstage && try_issue()) {
    }

    if (!mbar_wait_bounded(xw_bar, 0, prm.timeout_flag)) return;
    const uint32_t xw_base = smem_u32(xw_s);

    while (q0 < prm.nitems) {
        const int item = q0;
        const int row0 = item * kWarpRowsPerWarp;
        float acc[4][NT][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;

        for (int span = 0; span < NG; ++span) {
            const uint32_t slot = consumed % nstage;
            const uint32_t parity = (consumed / nstage) & 1u;
            if (!mbar_wait_bounded(&my_bars[slot], parity, prm.timeout_flag)) return;
            const uint32_t st = smem_u32(my_ring + slot * kStageBytes);
            uint4 pk[4][2][2];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = 16 * mt + 8 * h + g; // r & 7 == g
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        pk[mt][h][c] = lds128(st + r * kSpanBytes + (((2 * tig + c) ^ g) << 4));
                }
            // all lanes' reads of this stage are done before lane 0 refills it
            fence_proxy_async_smem();
            __syncwarp();
            ++consumed;
            while (issued < consumed + nstage && try_issue()) {
            }

            const uint32_t xw_span = xw_base + span * (4 * NT * 2048);
            float p[4][NT][4];
            plane_pass<NT, 0>(pk, xw_span + 0 * NT * 2048, lane, p);
            plane_epilogue<NT>(p, acc, prm, row0, g, tig, 0 * NG + span, NGt, xs_s);
            plane_pass<NT, 1>(pk, xw_span + 1 * NT * 2048, lane, p);
            plane_epilogue<NT>(p, acc, prm, row0, g, tig, 1 * NG + span, NGt, xs_s);
            plane_pass<NT, 2>(pk, xw_span + 2 * NT * 2048, lane, p);
            plane_epilogue<NT>(p, acc, prm, row0, g, tig, 2 * NG + span, NGt, xs_s);
            plane_pass<NT, 3>(pk, xw_span + 3 * NT * 2048, lane, p);
            plane_epilogue<NT>(p, acc, prm, row0, g, tig, 3 * NG + span, NGt, xs_s);
        }

        if (prm.coarse) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = row0 + 16 * mt + g + 8 * (i >> 1);
                        const int col = 8 * nt + 2 * tig + (i & 1);
                        if (row < prm.V && col < prm.mrows)
                            prm.coarse[static_cast<long long>(prm.m0 + col) * prm.V + row] =
                                acc[mt][nt][i];
                    }
        }
        emit_block<NT>(acc, prm, item, g, tig);
        if (q1 < 0) q1 = fetch();
        q0 = q1;
        q1 = -1;
    }
}

// Shared memory a launch needs besides its stage rings: the staged x of NT n8 tiles, the group
// sums and small scratch.
size_t warp_fixed_smem(int NT, int H)
{
    const size_t xw_bytes = static_cast<size_t>(H / 512) * 4 * NT * 2048;
    return 1024 /*alignment slack*/ + xw_bytes + static_cast<size_t>(8 * NT) * (H / kGroup + 1) * 4 +
           16 + 8 * 64;
}

template <int NT>
cudaError_t launch_nt(const CoarseArgs &a, const CUtensorMap &tm, cudaStream_t stream)
{
    const int H = a.H, NG = H / 512;
    const int nblk = (a.V + kBlockN - 1) / kBlockN;
    const uint32_t xw_bytes = static_cast<uint32_t>(NG) * 4 * NT * 2048;
    const size_t fixed = warp_fixed_smem(NT, H);
    const int nstage = NG >= 3 ? 3 : NG; // never more stages than spans per item
    int nwarps = static_cast<int>((kSmemLimit - static_cast<long long>(fixed)) /
                                  (static_cast<long long>(nstage) * kStageBytes));
    if (nwarps > kMaxWarpsPerCta) nwarps = kMaxWarpsPerCta;
    int use_stage = nstage;
    if (nwarps < 2 && use_stage > 2) { // fewer stages, more warps
        use_stage = 2;
        nwarps = static_cast<int>((kSmemLimit - static_cast<long long>(fixed)) /
                                  (2LL * kStageBytes));
        if (nwarps > kMaxWarpsPerCta) nwarps = kMaxWarpsPerCta;
    }
    if (nwarps < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = fixed + static_cast<size_t>(nwarps) * use_stage * kStageBytes;
    // raise the kernel's shared-memory cap (a per-device attribute) once on every device to
    // the most any call needs
    static PerDeviceOnce attr;
    cudaError_t err = attr.run([] {
        return cudaFuncSetAttribute(coarse_warp_kernel<NT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    });
    if (err != cudaSuccess) return err;
    const int chunks = (a.M + kWarpBatch - 1) / kWarpBatch;
    const int sms = device_sm_count();
    const int grid = nblk < sms ? nblk : sms;
    for (int c = 0; c < chunks; ++c) {
        WarpParams prm;
        prm.xw = reinterpret_cast<const uint4 *>(a.xw) + static_cast<size_t>(c) * (xw_bytes / 16);
        prm.xs = a.xs;
        prm.S = a.S;
        prm.ZS = a.ZS;
        prm.V = a.V;
        prm.H = a.H;
        prm.m0 = c * kWarpBatch;
        prm.mrows = (a.M - prm.m0) < kWarpBatch ? (a.M - prm.m0) : kWarpBatch;
        prm.kcand = a.kcand;
        prm.nitems = nblk;
        prm.nstage = use_stage;
        prm.ncand = static_cast<long long>(nblk) * a.kcand;
        prm.cand_val = a.cand_val;
        prm.cand_idx = a.cand_idx;
        prm.coarse = a.coarse;
        prm.counter = a.counters + c;
        prm.timeout_flag = a.timeout_flag;
        prm.xw_bytes = xw_bytes;
        coarse_warp_kernel<NT><<<grid, 32 * nwarps, smem, stream>>>(tm, prm);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

} // namespace

bool warp_supported(int M, int H)
{
    if (M < 1 || M > kMaxM || H <= 0 || H % 512 != 0) return false;
    const int NT = M <= 8 ? 1 : 2;
    return warp_fixed_smem(NT, H) + 2 * static_cast<size_t>(kStageBytes) <=
           static_cast<size_t>(kSmemLimit);
}

cudaError_t launch_coarse_warp(const CoarseArgs &a, cudaStream_t stream)
{
    CUtensorMap tm;
    CUresult r = encode_tensor_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                      const_cast<uint8_t *>(a.packed), a.H / 4, a.V, a.H / 4,
                                      kSpanBytes, kWarpRowsPerWarp, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (a.M <= 8) return launch_nt<1>(a, tm, stream);
    return launch_nt<2>(a, tm, stream);
}

} // namespace dh
