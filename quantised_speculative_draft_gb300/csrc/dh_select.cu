// dh_select.cu -- steps a5-a7: global top-RERANK selection, exact rerank, top-k merge.
//
// radiance_drafthead.py, _apply_head_int2: idx = BI.gather(BM.topk(RERANK)) (a5), then
// _rerank_exact, bf16 branch: e[m, j] = sum_k x[m, k] * W[idx[m, j], k] in fp32 (a6), then the
// best TOPK of the reranked entries (a7; only reranked entries are eligible, TOPK = 1 is the
// argmax caller).  Ordering everywhere: value descending, equal values -> lower index.
#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

namespace {

constexpr int kSelThreads = 512;

// 64-bit ranking key: order-preserving value bits above the complemented index, so a larger
// key is a better (value, index) pair.  0 marks an empty slot (no valid entry maps to 0).
__device__ __forceinline__ unsigned long long rank_key(float v, int idx)
{
    return (static_cast<unsigned long long>(f32_order_key(v)) << 32) |
           static_cast<unsigned long long>(~static_cast<uint32_t>(idx));
}

// ----------------------------------------------------------------------------------------
// a5: top-R of one chunk of a row's candidates by MSB-first radix selection on rank_key.
// grid (P, M); chunk p of row m covers entries [p CH, min(n_in, (p+1) CH)).  Writes the
// chunk's R best (unordered) to out[(m P + p) R + j]; a chunk with fewer valid entries pads
// with (-inf, -1).  With final_idx != null (P == 1) it writes the indices to final_idx[m R + j].
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) topr_kernel(const float *__restrict__ in_val,
                                                           const int32_t *__restrict__ in_idx,
                                                           long long stride_in, long long n_in,
                                                           int R, float *__restrict__ out_val,
                                                           int32_t *__restrict__ out_idx,
                                                           int32_t *__restrict__ final_idx)
{
    __shared__ unsigned long long keys[kSelectChunk];
    __shared__ uint32_t hist[256];
    __shared__ unsigned long long s_prefix, s_mask;
    __shared__ int s_needed, s_eq, s_nvalid, s_count;

    const int P = gridDim.x, p = blockIdx.x, m = blockIdx.y;
    const long long c0 = static_cast<long long>(p) * kSelectChunk;
    const float *vrow = in_val + static_cast<long long>(m) * stride_in;
    const int32_t *irow = in_idx + static_cast<long long>(m) * stride_in;

    if (threadIdx.x == 0) {
        s_nvalid = 0;
        s_count = 0;
    }
    __syncthreads();
    int my_valid = 0;
    for (int i = threadIdx.x; i < kSelectChunk; i += blockDim.x) {
        const long long e = c0 + i;
        unsigned long long k = 0;
        if (e < n_in) {
            const int id = irow[e];
            if (id >= 0) {
                k = rank_key(vrow[e], id);
                ++my_valid;
            }
        }
        keys[i] = k;
    }
    // count valid entries
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_valid += __shfl_xor_sync(0xffffffffu, my_valid, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_nvalid, my_valid);
    __syncthreads();
    const int nvalid = s_nvalid;
    const int want = nvalid < R ? nvalid : R;

    unsigned long long prefix = 0, mask = 0;
    if (want > 0 && want < nvalid) {
        int needed = want;
        for (int pass = 0; pass < 8; ++pass) {
            const int shift = 56 - 8 * pass;
            for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < kSelectChunk; i += blockDim.x) {
                const unsigned long long k = keys[i];
                if (k != 0 && (k & mask) == prefix)
                    atomicAdd(&hist[static_cast<int>((k >> shift) & 0xFFu)], 1u);
            }
            __syncthreads();
            if (threadIdx.x < 32) {
                // lane l owns digits 255-8l .. 248-8l (descending)
                const int lane = threadIdx.x;
                uint32_t loc[8];
                uint32_t tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    loc[j] = hist[255 - 8 * lane - j];
                    tot += loc[j];
                }
                uint32_t incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const uint32_t excl = incl - tot;
                const bool hit = excl < static_cast<uint32_t>(needed) &&
                                 incl >= static_cast<uint32_t>(needed);
                const unsigned ball = __ballot_sync(0xffffffffu, hit);
                const int src = __ffs(ball) - 1;
                if (lane == src) {
                    uint32_t cum = excl;
                    int d = 0;
                    uint32_t eq = 0;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (cum + loc[j] >= static_cast<uint32_t>(needed)) {
                            d = 255 - 8 * lane - j;
                            eq = loc[j];
                            break;
                        }
                        cum += loc[j];
                    }
                    s_prefix = prefix | (static_cast<unsigned long long>(d) << shift);
                    s_mask = mask | (0xFFull << shift);
                    s_needed = needed - static_cast<int>(cum);
                    s_eq = static_cast<int>(eq);
                }
            }
            __syncthreads();
            prefix = s_prefix;
            mask = s_mask;
            needed = s_needed;
            const int eq = s_eq;
            __syncthreads();
            if (eq == needed) break;
        }
    }
    // collect: every valid key whose masked bits reach the prefix (all of them when want ==
    // nvalid, since prefix = mask = 0)
    float *const ov = out_val + (static_cast<long long>(m) * P + p) * R;
    int32_t *const oi = out_idx + (static_cast<long long>(m) * P + p) * R;
    int32_t *const fi = final_idx ? final_idx + static_cast<long long>(m) * R : nullptr;
    for (int i = threadIdx.x; i < kSelectChunk; i += blockDim.x) {
        const unsigned long long k = keys[i];
        if (k != 0 && (k & mask) >= prefix) {
            const int slot = atomicAdd(&s_count, 1);
            if (slot < R) {
                const int id = static_cast<int>(~static_cast<uint32_t>(k));
                if (fi) {
                    fi[slot] = id;
                } else {
                    ov[slot] = f32_from_order_key(static_cast<uint32_t>(k >> 32));
                    oi[slot] = id;
                }
            }
        }
    }
    __syncthreads();
    for (int j = s_count + threadIdx.x; j < R; j += blockDim.x) {
        if (fi) {
            fi[j] = -1;
        } else {
            ov[j] = -INFINITY;
            oi[j] = -1;
        }
    }
}

// ----------------------------------------------------------------------------------------
// a6 + a7: exact rerank, then the top-k of the row.  One CTA of 128 threads per (row m,
// candidate j): every thread takes H/1024 16-byte slices of x and of the candidate's bf16 row
// (products of bf16 values are exact in fp32), sums them in two fp32 partials, and the CTA
// combines the 256 partials in fp64.  The last CTA to finish a row (an atomic count per row,
// zeroed by the staging kernel) sorts that row's R exact values and writes its top-k.
// ----------------------------------------------------------------------------------------
constexpr int kRerankThreads = 128;

__global__ void __launch_bounds__(kRerankThreads) rerank_topk_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ W, int H, int V,
    const int32_t *__restrict__ sel_idx, int R, float *__restrict__ ex,
    int *__restrict__ row_done, int topk, int32_t *__restrict__ out_idx,
    float *__restrict__ out_logit)
{
    __shared__ double part[kRerankThreads / 32];
    __shared__ unsigned long long k[kMaxRerank];
    __shared__ int s_last;
    const long long pair = blockIdx.x;
    const int m = static_cast<int>(pair / R);
    const int n = sel_idx[pair];
    const int tid = threadIdx.x, lane = tid & 31;

    float a0 = 0.f, a1 = 0.f;
    if (n >= 0 && n < V) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<long long>(m) * H);
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + static_cast<long long>(n) * H);
        const int nv = H / 8;
#pragma unroll 4
        for (int i = tid; i < nv; i += kRerankThreads) {
            const uint4 xv = __ldg(xr + i);
            const uint4 wv = __ldg(wr + i);
            const uint32_t xs4[4] = {xv.x, xv.y, xv.z, xv.w};
            const uint32_t ws4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a0 = fmaf(__uint_as_float(xs4[q] << 16), __uint_as_float(ws4[q] << 16), a0);
                a1 = fmaf(__uint_as_float(xs4[q] & 0xFFFF0000u),
                          __uint_as_float(ws4[q] & 0xFFFF0000u), a1);
            }
        }
    }
    double d = static_cast<double>(a0) + static_cast<double>(a1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) part[tid >> 5] = d;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int i = 0; i < kRerankThreads / 32; ++i) t += part[i];
        ex[pair] = (n >= 0 && n < V) ? static_cast<float>(t) : -INFINITY;
        __threadfence();
        s_last = atomicAdd(&row_done[m], 1) == R - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // this CTA finished row m last: top-k of its R reranked entries (bitonic, descending)
    int n2 = 1;
    while (n2 < R) n2 <<= 1;
    for (int i = tid; i < n2; i += kRerankThreads) {
        unsigned long long key = 0;
        if (i < R) {
            const int id = __ldcg(sel_idx + static_cast<long long>(m) * R + i);
            if (id >= 0 && id < V) key = rank_key(__ldcg(ex + static_cast<long long>(m) * R + i), id);
        }
        k[i] = key;
    }
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += kRerankThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = k[i], b = k[j];
                    if (desc ? (a < b) : (a > b)) {
                        k[i] = b;
                        k[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int t = tid; t < topk; t += kRerankThreads) {
        const unsigned long long key = k[t];
        const bool ok = key != 0;
        out_idx[static_cast<long long>(m) * topk + t] =
            ok ? static_cast<int>(~static_cast<uint32_t>(key)) : -1;
        out_logit[static_cast<long long>(m) * topk + t] =
            ok ? f32_from_order_key(static_cast<uint32_t>(key >> 32)) : -INFINITY;
    }
}

} // namespace

void select_plan(int M, long long ncand, int R, int *passes, long long *scratch_entries)
{
    long long n = ncand;
    int np = 0;
    long long most = 0;
    for (;;) {
        const long long P = (n + kSelectChunk - 1) / kSelectChunk;
        ++np;
        if (P <= 1) break;
        const long long e = static_cast<long long>(M) * P * R;
        if (e > most) most = e;
        n = P * R;
    }
    *passes = np;
    *scratch_entries = most;
}

cudaError_t launch_select(const float *cand_val, const int32_t *cand_idx, int M, long long ncand,
                          int R, float *scratch_val[2], int32_t *scratch_idx[2],
                          long long scratch_entries, int32_t *sel_idx, cudaStream_t stream)
{
    (void)scratch_entries;
    const float *in_v = cand_val;
    const int32_t *in_i = cand_idx;
    long long stride = ncand, n = ncand;
    int buf = 0;
    for (;;) {
        const long long P = (n + kSelectChunk - 1) / kSelectChunk;
        dim3 grid(static_cast<unsigned>(P), static_cast<unsigned>(M));
        if (P <= 1) {
            topr_kernel<<<grid, kSelThreads, 0, stream>>>(in_v, in_i, stride, n, R, nullptr,
                                                          nullptr, sel_idx);
            return cudaGetLastError();
        }
        topr_kernel<<<grid, kSelThreads, 0, stream>>>(in_v, in_i, stride, n, R, scratch_val[buf],
                                                      scratch_idx[buf], nullptr);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        in_v = scratch_val[buf];
        in_i = scratch_idx[buf];
        n = P * R;
        stride = n;
        buf ^= 1;
    }
}

cudaError_t launch_rerank_topk(const uint16_t *x, const uint16_t *W, int M, int H, int V,
                               const int32_t *sel_idx, int R, float *ex, int *row_done, int topk,
                               int32_t *out_idx, float *out_logit, cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>(static_cast<long long>(M) * R);
    rerank_topk_kernel<<<blocks, kRerankThreads, 0, stream>>>(x, W, H, V, sel_idx, R, ex,
                                                              row_done, topk, out_idx, out_logit);
    return cudaGetLastError();
}

} // namespace dh
