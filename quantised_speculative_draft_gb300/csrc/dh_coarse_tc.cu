// dh_coarse_tc.cu -- kernels (2)+(3), tcgen05 path: coarse pass on 5th-generation tensor cores
// with tensor-memory accumulators, and the fused block top-KCAND epilogue.
//
// radiance_drafthead.py, _draft_head_int2 and _emit: for vocabulary row n and batch row m
//     c[m, n] = sum_g ( S[n, g] * p[m, n, g] - ZS[n, g] * xs[m, g] ),
//     p[m, n, g] = sum_{k in g} x[m, k] * (1 + v[n, k] / 4),
// the scale and zero applied to the fp32 partial of each group (never to the weight), then
// the KCAND best (value, row) pairs of every 64-row block per batch row.
//
// GB300 design (swap-AB: vocabulary rows are the MMA's M = 128, the padded batch is N):
//   * persistent CTAs, one per SM, walk 128-row vocabulary tiles;
//   * warp 0 issues TMA: per span (128 packed bytes of every row = the four planes of one
//     span) one [128 rows x 128 B] box of the packed weight and eight [64 k x N] boxes of the
//     staged, quad-permuted x (128-byte swizzle), into a ring of shared-memory stages;
//   * warps 4-11 dequantise: each thread owns one vocabulary row (one TMEM lane), reads its
//     128 bytes, and writes plane q as bf16 pairs 1 + v/4 (bit-pattern dequant) straight into
//     a tensor-memory A buffer with tcgen05.st -- the weight never touches shared memory as
//     bf16 and never gets a scale;
//   * warp 1 issues tcgen05.mma kind::f16, A from tensor memory, B (x) from shared memory,
//     D = the group's fp32 partial p in tensor memory (8 MMAs of K = 16 per group);
//   * warps 12-15 read each group's partial with tcgen05.ld, fold it into per-row running
//     accumulators in registers with the group's scale and zero, and at the end of the tile
//     run the block top-KCAND selection;
//   * every handoff is an mbarrier; every wait is bounded and gives up with a flag.
//
// kWS (the page's scale-placement ablation, module docstring: 'The scale is applied to the
// accumulator, never to the weight tile'): the dequant warps instead write every weight as
// bf16(S (1 + v/4) - ZS) -- the group's scale and zero applied to each element -- and all
// MMAs of a tile accumulate into one buffer, so the epilogue has no per-group fold.
#include "dh_common.cuh"
#include "dh_internal.h"
#include "dh_tcgen05.cuh"

#include <climits>

namespace dh {

namespace {

constexpr int kTileRows = 128;
constexpr int kThreads = 512; // 16 warps
constexpr int kTmemCols = 512;
constexpr int kPkBytes = kTileRows * kSpanBytes; // 16 KB packed box per span
constexpr int kMaxN = 64;                       // batch rows per launch
constexpr int kSmemLimitTc = 232448;

// Tensor memory (512 columns x 128 lanes): a ring of A buffers (64 columns = 128 bf16 of K,
// one group's dequantised weights) followed by a ring of D buffers (N fp32 columns, one
// group's partial p).  Deep rings let dequant, MMA and epilogue run several groups apart.
template <int N> struct Rings {
    static constexpr int kA = (N <= 32) ? 6 : 4;
    static constexpr int kD0 = (kTmemCols - kA * 64) / N;
    static constexpr int kD = kD0 > 8 ? 8 : kD0;
    static constexpr uint32_t kAcol = 0;
    static constexpr uint32_t kDcol = kA * 64;
    static_assert(kD >= 2, "tensor memory too small for two accumulators");
};

struct TcParams {
    const uint16_t *S;
    const uint16_t *ZS;
    const float *xs; // [rows, NGt], this launch's rows start at m0
    int V, H, m0, mrows, kcand, ntiles, nstage;
    long long ncand;
    float *cand_val;
    int32_t *cand_idx;
    float *coarse;
    int *timeout_flag;
};

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M = 128, N.
__host__ __device__ constexpr uint32_t make_idesc(int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

// ---- the kernel -------------------------------------------------------------------------

template <int N, bool kWS>
__global__ void __launch_bounds__(kThreads, 1)
    coarse_tc_kernel(const __grid_constant__ CUtensorMap tm_packed,
                     const __grid_constant__ CUtensorMap tm_x, const TcParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = prm.H / 512, NGt = prm.H / kGroup;
    const int nstage = prm.nstage;
    constexpr uint32_t kXBytes = N * 1024;          // 4 planes x 128 k x N rows x 2 B
    constexpr uint32_t kStage = kPkBytes + kXBytes; // multiple of 1024

    // ---- shared memory ------------------------------------------------------------------
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t *const stages = smem_raw + pad;                          // nstage * kStage
    float *const red = reinterpret_cast<float *>(stages + static_cast<size_t>(nstage) * kStage);
    float *const xs_s = red + N * kTileRows;                         // [NGt][N]
    uint64_t *const bars = reinterpret_cast<uint64_t *>(xs_s + NGt * N);
    uint64_t *const full = bars;                  // [nstage]  TMA -> consumers
    uint64_t *const empty = full + nstage;        // [nstage]  consumers -> TMA
    constexpr int kA = Rings<N>::kA, kD = Rings<N>::kD;
    uint64_t *const a_full = empty + nstage;      // [kA]      dequant -> MMA
    uint64_t *const a_empty = a_full + kA;        // [kA]      MMA -> dequant
    uint64_t *const d_full = a_empty + kA;        // [kD]      MMA -> epilogue
    uint64_t *const d_empty = d_full + kD;        // [kD]      epilogue -> MMA
    uint64_t *const fin = d_empty + kD;           // [1]       MMA drain before teardown
    uint64_t *const red_full = fin + 1;           // [1]       epilogue warps: tile written
    uint64_t *const red_free = red_full + 1;      // [1]       epilogue warps: tile selected
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(red_free + 1);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_packed);
        prefetch_tensormap(&tm_x);
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 8 + 1); // 8 dequant warps + 1 MMA commit
        }
        for (int i = 0; i < kA; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < kD; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], 4);
        }
        mbar_init(fin, 1);
        mbar_init(red_full, 4);
        mbar_init(red_free, 4);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < NGt * N; i += blockDim.x) {
        const int g = i / N, m = i - g * N;
        xs_s[i] = prm.xs[static_cast<long long>(prm.m0 + m) * NGt + g];
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int first_tile = blockIdx.x, tile_step = gridDim.x;
    bool failed = false;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            uint32_t s = 0;
            for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step) {
                for (int span = 0; span < NG; ++span, ++s) {
                    const uint32_t st = s % nstage;
                    if (!mbar_wait_bounded(&empty[st], ((s / nstage) & 1u) ^ 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    uint8_t *const stage = stages + static_cast<size_t>(st) * kStage;
                    mbar_arrive_expect_tx(&full[st], kStage);
                    tma_load_2d_hint(stage, &tm_packed, span * kSpanBytes, tile * kTileRows,
                                     &full[st], policy);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d(stage + kPkBytes + (q * 2 + h) * (N * 128), &tm_x,
                                        q * (prm.H / 4) + span * 128 + h * 64, 0, &full[st]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(N);
            uint32_t s = 0, t = 0, it = 0;
            for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step, ++it) {
                // kWS: the tile's one accumulator, free once the epilogue read tile it - kD
                const uint32_t dt = it % kD;
                if (kWS && !mbar_wait_bounded(&d_empty[dt], ((it / kD) & 1u) ^ 1u,
                                              prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                for (int span = 0; span < NG && !failed; ++span, ++s) {
                    const uint32_t st = s % nstage;
                    if (!mbar_wait_bounded(&full[st], (s / nstage) & 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    const uint32_t xbase = smem_u32(stages + static_cast<size_t>(st) * kStage + kPkBytes);
                    for (int q = 0; q < 4; ++q, ++t) {
                        const uint32_t a = t % kA, d = kWS ? dt : t % kD;
                        if (!mbar_wait_bounded(&a_full[a], (t / kA) & 1u, prm.timeout_flag) ||
                            (!kWS && !mbar_wait_bounded(&d_empty[d], ((t / kD) & 1u) ^ 1u,
                                                        prm.timeout_flag))) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + Rings<N>::kDcol + d * N;
                        const uint32_t a_tmem = tmem + Rings<N>::kAcol + a * 64;
                        // kWS: one accumulation over the whole tile
                        const bool fresh = !kWS || (span == 0 && q == 0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t b_addr = xbase + (q * 2 + (i >> 2)) * (N * 128) + (i & 3) * 32;
                            mma_ts(d_tmem, a_tmem + i * 8, sw128_desc(b_addr), idesc,
                                   (i > 0 || !fresh) ? 1u : 0u);
                        }
                        mma_commit(&a_empty[a]);
                        if (!kWS || (span == NG - 1 && q == 3)) mma_commit(&d_full[d]);
                    }
                    if (!failed) mma_commit(&empty[st]);
                }
            }
            // drain: everything issued has completed before TMEM is released
            mma_commit(fin);
            mbar_wait_bounded(fin, 0, prm.timeout_flag);
        }
    } else if (warp >= 4 && warp < 12) {
        // ---------------- dequant: warps 4-7 planes 0 and 2, warps 8-11 planes 1 and 3 -------
        const int row = ((warp & 3) << 5) | lane; // TMEM lane == tile row
        const int qoff = (warp < 8) ? 0 : 1;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        uint32_t s = 0;
        for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step) {
            const int grow = tile * kTileRows + row;
            const bool row_ok = grow < prm.V;
            const uint16_t *Srow = prm.S + static_cast<long long>(row_ok ? grow : 0) * NGt;
            const uint16_t *Zrow = prm.ZS + static_cast<long long>(row_ok ? grow : 0) * NGt;
            for (int span = 0; span < NG; ++span, ++s) {
                const uint32_t st = s % nstage;
                if (!warp_wait(&full[st], (s / nstage) & 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                const uint32_t pk = smem_u32(stages + static_cast<size_t>(st) * kStage) + row * kSpanBytes;
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = pk + ((c ^ (row & 7)) << 4);
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]),
                                   "=r"(w[4 * c + 3])
                                 : "r"(addr));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int q = qoff + 2 * qq;
                    const uint32_t t = s * 4 + q;      // global group counter
                    const uint32_t a = t % kA;
                    if (!warp_wait(&a_empty[a], ((t / kA) & 1u) ^ 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    uint32_t r[64];
                    if (q == 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r[2 * i] = deq_pair_even<0>(w[i]);
                            r[2 * i + 1] = deq_pair_odd<0>(w[i]);
                        }
                    } else if (q == 1) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r[2 * i] = deq_pair_even<1>(w[i]);
                            r[2 * i + 1] = deq_pair_odd<1>(w[i]);
                        }
                    } else if (q == 2) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r[2 * i] = deq_pair_even<2>(w[i]);
                            r[2 * i + 1] = deq_pair_odd<2>(w[i]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r[2 * i] = deq_pair_even<3>(w[i]);
                            r[2 * i + 1] = deq_pair_odd<3>(w[i]);
                        }
                    }
                    if constexpr (kWS) {
                        // the group's scale and zero on every weight: bf16(S (1 + v/4) - ZS),
                        // the inner value exact, one rounding to bf16
                        const int gi = q * NG + span;
                        const float sv = row_ok ? bf16_bits_to_f32(__ldg(Srow + gi)) : 0.f;
                        const float zv = row_ok ? bf16_bits_to_f32(__ldg(Zrow + gi)) : 0.f;
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            const float lo = fmaf(sv, __uint_as_float(r[i] << 16), -zv);
                            const float hi = fmaf(sv, __uint_as_float(r[i] & 0xFFFF0000u), -zv);
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                            r[i] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                    }
                    tmem_st_x64(tmem + lane_base + Rings<N>::kAcol + a * 64, r);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[a]);
                }
                if (failed) break;
            }
        }
    } else if (warp >= 12) {
        // ---------------- epilogue: scale/zero fold + block top-KCAND ----------------
        const int row = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
        uint32_t t = 0, it = 0;
        for (int tile = first_tile; tile < prm.ntiles && !failed; tile += tile_step, ++it) {
            const int grow = tile * kTileRows + row;
            const bool row_ok = grow < prm.V;
            const uint16_t *Srow = prm.S + static_cast<long long>(row_ok ? grow : 0) * NGt;
            const uint16_t *Zrow = prm.ZS + static_cast<long long>(row_ok ? grow : 0) * NGt;
            float acc[N];
#pragma unroll
            for (int m = 0; m < N; ++m) acc[m] = 0.f;
            if constexpr (kWS) {
                // the tile's single accumulator holds the coarse values
                const uint32_t dt = it % kD;
                if (!warp_wait(&d_full[dt], (it / kD) & 1u, prm.timeout_flag)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < N / 16; ++c) {
                    float v[16];
                    tmem_ld_x16(tmem + lane_base + Rings<N>::kDcol + dt * N + c * 16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[c * 16 + j] = v[j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[dt]);
            }
            for (int span = 0; span < NG && !failed && !kWS; ++span) {
                for (int q = 0; q < 4; ++q, ++t) {
                    const uint32_t d = t % kD;
                    if (!warp_wait(&d_full[d], (t / kD) & 1u, prm.timeout_flag)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const int gi = q * NG + span;
                    const float sv = row_ok ? bf16_bits_to_f32(__ldg(Srow + gi)) : 0.f;
                    const float zv = row_ok ? bf16_bits_to_f32(__ldg(Zrow + gi)) : 0.f;
                    const float4 *xg = reinterpret_cast<const float4 *>(xs_s + gi * N);
#pragma unroll
                    for (int c = 0; c < N / 16; ++c) {
                        float v[16];
                        tmem_ld_x16(tmem + lane_base + Rings<N>::kDcol + d * N + c * 16, v);
                        tmem_wait_ld();
                        if (c == N / 16 - 1) {
                            // the partial has been read out: hand the D buffer back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&d_empty[d]);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 x4 = xg[c * 4 + j];
                            const int m = c * 16 + 4 * j;
                            acc[m + 0] = fmaf(sv, v[4 * j + 0], fmaf(-zv, x4.x, acc[m + 0]));
                            acc[m + 1] = fmaf(sv, v[4 * j + 1], fmaf(-zv, x4.y, acc[m + 1]));
                            acc[m + 2] = fmaf(sv, v[4 * j + 2], fmaf(-zv, x4.z, acc[m + 2]));
                            acc[m + 3] = fmaf(sv, v[4 * j + 3], fmaf(-zv, x4.w, acc[m + 3]));
                        }
                    }
                }
            }
            if (failed) break;
            // the previous tile's selection has finished reading the exchange buffer
            if (!warp_wait(red_free, (it & 1u) ^ 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            // coarse values of the tile -> shared [N][128], optional debug copy to global
#pragma unroll
            for (int m = 0; m < N; ++m) red[m * kTileRows + row] = row_ok ? acc[m] : -INFINITY;
            if (prm.coarse && row_ok) {
#pragma unroll
                for (int m = 0; m < N; ++m)
                    if (m < prm.mrows)
                        prm.coarse[static_cast<long long>(prm.m0 + m) * prm.V + grow] = acc[m];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_full);
            if (!warp_wait(red_full, it & 1u, prm.timeout_flag)) {
                failed = true;
                break;
            }
            // block top-KCAND: pair p = (batch column m, block b of the tile)
            const int ew = warp & 3;
            for (int pidx = ew; pidx < 2 * prm.mrows; pidx += 4) {
                const int m = pidx >> 1, b = pidx & 1;
                const int blk = tile * 2 + b;
                if (static_cast<long long>(blk) * kBlockN >= prm.V) continue;
                const int r0 = b * 64 + lane, r1 = r0 + 32;
                float v0 = red[m * kTileRows + r0], v1 = red[m * kTileRows + r1];
                int i0 = tile * kTileRows + r0, i1 = tile * kTileRows + r1;
                if (i0 >= prm.V) i0 = INT_MAX;
                if (i1 >= prm.V) i1 = INT_MAX;
                const long long base = static_cast<long long>(prm.m0 + m) * prm.ncand +
                                       static_cast<long long>(blk) * prm.kcand;
                for (int k = 0; k < prm.kcand; ++k) {
                    float bv = v0;
                    int bi = i0;
                    if (better(v1, i1, bv, bi)) {
                        bv = v1;
                        bi = i1;
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                        if (better(ov, oi, bv, bi)) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    if (i0 == bi) {
                        v0 = -INFINITY;
                        i0 = INT_MAX;
                    }
                    if (i1 == bi) {
                        v1 = -INFINITY;
                        i1 = INT_MAX;
                    }
                    if (lane == 0) {
                        const bool valid = bi != INT_MAX;
                        prm.cand_val[base + k] = valid ? bv : -INFINITY;
                        prm.cand_idx[base + k] = valid ? bi : -1;
                    }
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
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int N, bool kWS>
cudaError_t launch_n(const CUtensorMap &tm_packed, const uint16_t *xt_chunk, const TcParams &base,
                     cudaStream_t stream)
{
    CUtensorMap tm_x;
    CUresult r = encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                      const_cast<uint16_t *>(xt_chunk), base.H, N,
                                      static_cast<uint64_t>(base.H) * 2, 64, N,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const int NGt = base.H / kGroup;
    constexpr int kStage = kPkBytes + N * 1024;
    const size_t fixed = 1024 + static_cast<size_t>(N) * kTileRows * 4 +
                         static_cast<size_t>(NGt) * N * 4 + 96 * 8 + 32;
    int nstage = static_cast<int>((kSmemLimitTc - static_cast<long long>(fixed)) / kStage);
    if (nstage > 4) nstage = 4;
    if (nstage < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = fixed + static_cast<size_t>(nstage) * kStage;
    // the shared-memory limit is a per-device attribute: raised once on every device
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        return cudaFuncSetAttribute(coarse_tc_kernel<N, kWS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimitTc);
    });
    if (e != cudaSuccess) return e;
    TcParams prm = base;
    prm.nstage = nstage;
    const int sms = device_sm_count();
    const int grid = prm.ntiles < sms ? prm.ntiles : sms;
    coarse_tc_kernel<N, kWS><<<grid, kThreads, smem, stream>>>(tm_packed, tm_x, prm);
    return cudaGetLastError();
}

} // namespace

int tc_npad(int M)
{
    return ((M + 15) / 16) * 16;
}

int tc_launches(int M)
{
    return (M + kMaxN - 1) / kMaxN;
}

bool tc_supported(int M, int H)
{
    // the staged x of a span and the reduction buffer must fit next to two stages
    return M >= 1 && M <= kMaxM && H % 512 == 0 && H <= 16384;
}

cudaError_t launch_coarse_tc(const CoarseArgs &a, cudaStream_t stream)
{
    CUtensorMap tm_packed;
    CUresult r = encode_tensor_map_2d(&tm_packed, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                      const_cast<uint8_t *>(a.packed), a.H / 4, a.V, a.H / 4,
                                      kSpanBytes, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    TcParams base;
    base.S = a.S;
    base.ZS = a.ZS;
    base.xs = a.xs;
    base.V = a.V;
    base.H = a.H;
    base.kcand = a.kcand;
    base.ntiles = (a.V + kTileRows - 1) / kTileRows;
    base.ncand = static_cast<long long>((a.V + kBlockN - 1) / kBlockN) * a.kcand;
    base.cand_val = a.cand_val;
    base.cand_idx = a.cand_idx;
    base.coarse = a.coarse;
    base.timeout_flag = a.timeout_flag;
    base.nstage = 2;
    for (int m0 = 0; m0 < a.M; m0 += kMaxN) {
        const int rows = (a.M - m0) < kMaxN ? (a.M - m0) : kMaxN;
        const int n = tc_npad(rows);
        base.m0 = m0;
        base.mrows = rows;
        const uint16_t *xt_chunk = a.xt + static_cast<size_t>(m0) * a.H;
        cudaError_t e;
        if (a.pack == kPackWside) {
            switch (n) {
            case 16: e = launch_n<16, true>(tm_packed, xt_chunk, base, stream); break;
            case 32: e = launch_n<32, true>(tm_packed, xt_chunk, base, stream); break;
            case 48: e = launch_n<48, true>(tm_packed, xt_chunk, base, stream); break;
            default: e = launch_n<64, true>(tm_packed, xt_chunk, base, stream); break;
            }
        } else {
            switch (n) {
            case 16: e = launch_n<16, false>(tm_packed, xt_chunk, base, stream); break;
            case 32: e = launch_n<32, false>(tm_packed, xt_chunk, base, stream); break;
            case 48: e = launch_n<48, false>(tm_packed, xt_chunk, base, stream); break;
            default: e = launch_n<64, false>(tm_packed, xt_chunk, base, stream); break;
            }
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace dh
