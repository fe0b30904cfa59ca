// dh_select.cu -- steps a5-a7: global top-RERANK selection, exact rerank, top-k merge.
//
// radiance_drafthead.py, _apply_head_int2: idx = BI.gather(BM.topk(RERANK)) (a5), then
// _rerank_exact, bf16 branch: e[m, j] = sum_k x[m, k] * W[idx[m, j], k] in fp32 (a6), then the
// best TOPK of the reranked entries (a7; only reranked entries are eligible, TOPK = 1 is the
// argmax caller).  Ordering everywhere: value descending, equal values -> lower index.
#include "dh_common.cuh"
#include "dh_internal.h"

#include <cooperative_groups.h>
#include <type_traits>

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
// with (-inf, -1).  With final_idx != null (P == 1) it writes the R best in rank order (value
// descending, lower index first; a shared-memory sort makes the order deterministic): the
// indices plus id_offset to final_idx[m R + j] (-1 for empty slots) and, with
// final_val != null, the values to final_val[m R + j].
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) topr_kernel(const float *__restrict__ in_val,
                                                           const int32_t *__restrict__ in_idx,
                                                           long long stride_in, long long n_in,
                                                           int R, float *__restrict__ out_val,
                                                           int32_t *__restrict__ out_idx,
                                                           int32_t *__restrict__ final_idx,
                                                           float *__restrict__ final_val,
                                                           int id_offset)
{
    __shared__ unsigned long long keys[kSelectChunk];
    __shared__ unsigned long long outk[kMaxRerank]; // the final pass's R best, sorted
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
    for (int i = threadIdx.x; i < kSelectChunk; i += blockDim.x) {
        const unsigned long long k = keys[i];
        if (k != 0 && (k & mask) >= prefix) {
            const int slot = atomicAdd(&s_count, 1);
            if (slot < R) {
                if (final_idx) {
                    outk[slot] = k;
                } else {
                    ov[slot] = f32_from_order_key(static_cast<uint32_t>(k >> 32));
                    oi[slot] = static_cast<int>(~static_cast<uint32_t>(k));
                }
            }
        }
    }
    __syncthreads();
    const int got = s_count < R ? s_count : R;
    if (!final_idx) {
        for (int j = got + threadIdx.x; j < R; j += blockDim.x) {
            ov[j] = -INFINITY;
            oi[j] = -1;
        }
        return;
    }
    // final pass: sort the R best (bitonic, descending) so that the output is in rank order
    int n2 = 1;
    while (n2 < R) n2 <<= 1;
    for (int j = got + threadIdx.x; j < n2; j += blockDim.x) outk[j] = 0ull;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = outk[i], b = outk[j];
                    if (desc ? (a < b) : (a > b)) {
                        outk[i] = b;
                        outk[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    int32_t *const fi = final_idx + static_cast<long long>(m) * R;
    float *const fv = final_val ? final_val + static_cast<long long>(m) * R : nullptr;
    for (int j = threadIdx.x; j < R; j += blockDim.x) {
        const unsigned long long k = outk[j];
        fi[j] = k ? static_cast<int>(~static_cast<uint32_t>(k)) + id_offset : -1;
        if (fv) fv[j] = k ? f32_from_order_key(static_cast<uint32_t>(k >> 32)) : -INFINITY;
    }
}

// ----------------------------------------------------------------------------------------
// a5, one launch per batch row when the sizes allow it.  Every block's candidate list is in
// rank order (value descending, lower row first), so a candidate can be among the row's R
// best only if its block's best is among the R best block maxima: if R blocks have a better
// maximum, R candidates beat everything in the block.  For R <= 32 the 32 best block maxima
// are found by CTAs of 512 maxima and merged by the row's last CTA, which then keeps the 32
// best of those blocks' candidates and writes the R best indices in rank order.  Sorting is
// warp-level (bitonic sorts of 32 keys, merges of sorted 32-lists), so nothing needs a
// block-wide sort.  Keys are unique (the index is part of the key), so the cut is exact.
// ----------------------------------------------------------------------------------------
constexpr int kRowSelThreads = 128; // 4 warps
constexpr int kRowSelChunk = 128;   // keys per warp sort unit (4 lists of 32)
constexpr int kRowSelCtaKeys = 512; // block maxima per CTA in phase 1
constexpr int kRowSelMaxCtas = 16;  // CTAs per row (block count <= 8192)
constexpr int kRowSelR = 32;        // lists keep the 32 best

__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b)
{
    return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long kmin(unsigned long long a, unsigned long long b)
{
    return a < b ? a : b;
}

// Sorts N warp lists (one key per lane each) descending, in lockstep (bitonic, 15 stages).
template <int N>
__device__ __forceinline__ void warp_sort32xN_desc(unsigned long long (&v)[N])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
#pragma unroll
            for (int r = 0; r < N; ++r) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[r], stride);
                v[r] = keep_max ? kmax(v[r], o) : kmin(v[r], o);
            }
        }
    }
}

// The 32 best of two descending warp lists, descending: the half-cleaner of a against b
// reversed leaves the 32 largest as a bitonic sequence, five more stages sort it.
__device__ __forceinline__ unsigned long long warp_merge32_desc(unsigned long long a,
                                                                unsigned long long b)
{
    const int lane = threadIdx.x & 31;
    unsigned long long v = kmax(a, __shfl_sync(0xffffffffu, b, 31 - lane));
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
        v = (lane & stride) == 0 ? kmax(v, o) : kmin(v, o);
    }
    return v;
}

// The 32 best (descending, one per lane) of the 128 keys k[0..127] (0 = empty).
__device__ __forceinline__ unsigned long long warp_top32_of128(const unsigned long long *k)
{
    const int lane = threadIdx.x & 31;
    unsigned long long v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = k[r * 32 + lane];
    warp_sort32xN_desc<4>(v);
    return warp_merge32_desc(warp_merge32_desc(v[0], v[1]), warp_merge32_desc(v[2], v[3]));
}

// The 32 best (descending, one per lane) of the 64 keys k[0..63] (0 = empty).
__device__ __forceinline__ unsigned long long warp_top32_of64(const unsigned long long *k)
{
    const int lane = threadIdx.x & 31;
    unsigned long long v[2] = {k[lane], k[32 + lane]};
    warp_sort32xN_desc<2>(v);
    return warp_merge32_desc(v[0], v[1]);
}

// The 32 best of n keys in shared memory (n a multiple of 128, keys beyond the data 0), by the
// CTA's four warps; returns the list in lists[0] (descending).  All threads must call it.
__device__ void cta_top32(const unsigned long long *keys, int n, unsigned long long (*lists)[32])
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long acc = 0;
    for (int c = warp; c * kRowSelChunk < n; c += 4)
        acc = warp_merge32_desc(acc, warp_top32_of128(keys + c * kRowSelChunk));
    lists[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long a = warp_merge32_desc(lists[0][lane], lists[1][lane]);
        const unsigned long long b = warp_merge32_desc(lists[2][lane], lists[3][lane]);
        lists[0][lane] = warp_merge32_desc(a, b);
    }
    __syncthreads();
}

// Phase 1, grid (P, M): CTA p keeps the 32 best of block maxima [512 p, 512 p + 512) of row m
// and writes them to partial[(m P + p) 32 ..]; the last CTA of the row (per-row counter,
// zeroed by the staging kernel) merges the P lists, takes the 32 best blocks' candidates and
// writes the row's R best indices in rank order.  No CTA waits for another.
__global__ void __launch_bounds__(kRowSelThreads) select_rows_kernel(
    const float *__restrict__ cand_val, const int32_t *__restrict__ cand_idx, long long ncand,
    int nblk, int kcand, int R, unsigned long long *__restrict__ partial, int *__restrict__ row_cnt,
    int32_t *__restrict__ sel_idx, float *__restrict__ sel_val, int id_offset)
{
    __shared__ unsigned long long keys[kRowSelR * kBlockN]; // 2048: the largest candidate set
    __shared__ unsigned long long lists[4][32];
    __shared__ int sblk[kRowSelR];
    __shared__ int s_last;
    const int P = gridDim.x, p = blockIdx.x, m = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const float *vrow = cand_val + static_cast<long long>(m) * ncand;
    const int32_t *irow = cand_idx + static_cast<long long>(m) * ncand;

    {
        // every load issued before any is used (value and index independently)
        constexpr int kPer = kRowSelCtaKeys / kRowSelThreads;
        int ids[kPer];
        float vals[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int bk = p * kRowSelCtaKeys + threadIdx.x + u * kRowSelThreads;
            const long long e = static_cast<long long>(bk < nblk ? bk : 0) * kcand;
            ids[u] = __ldcg(irow + e);
            vals[u] = __ldcg(vrow + e);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int bk = p * kRowSelCtaKeys + threadIdx.x + u * kRowSelThreads;
            keys[threadIdx.x + u * kRowSelThreads] =
                (bk < nblk && ids[u] >= 0) ? rank_key(vals[u], ids[u]) : 0ull;
        }
    }
    __syncthreads();
    cta_top32(keys, kRowSelCtaKeys, lists);
    if (threadIdx.x < 32) partial[(static_cast<long long>(m) * P + p) * 32 + lane] = lists[0][lane];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&row_cnt[m], 1) == P - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // the row's last CTA: the 32 best blocks from the P lists
    const int np = ((P * 32 + kRowSelChunk - 1) / kRowSelChunk) * kRowSelChunk;
    for (int i = threadIdx.x; i < np; i += kRowSelThreads)
        keys[i] = i < P * 32 ? __ldcg(partial + static_cast<long long>(m) * P * 32 + i) : 0ull;
    __syncthreads();
    cta_top32(keys, np, lists);
    if (threadIdx.x < kRowSelR) {
        const unsigned long long key = lists[0][threadIdx.x];
        sblk[threadIdx.x] = key ? static_cast<int>(~static_cast<uint32_t>(key)) / kBlockN : -1;
    }
    __syncthreads();
    // their candidates; the R best in rank order
    const int nc = kRowSelR * kcand;
    const int ncp = ((nc + kRowSelChunk - 1) / kRowSelChunk) * kRowSelChunk;
    for (int e = threadIdx.x; e < ncp; e += kRowSelThreads) {
        unsigned long long key = 0;
        if (e < nc) {
            const int bk = sblk[e / kcand];
            if (bk >= 0) {
                const long long c = static_cast<long long>(bk) * kcand + e % kcand;
                const int id = irow[c];
                if (id >= 0) key = rank_key(vrow[c], id);
            }
        }
        keys[e] = key;
    }
    __syncthreads();
    cta_top32(keys, ncp, lists);
    if (threadIdx.x < R) {
        const unsigned long long key = lists[0][threadIdx.x];
        sel_idx[static_cast<long long>(m) * R + threadIdx.x] =
            key ? static_cast<int>(~static_cast<uint32_t>(key)) + id_offset : -1;
        if (sel_val)
            sel_val[static_cast<long long>(m) * R + threadIdx.x] =
                key ? f32_from_order_key(static_cast<uint32_t>(key >> 32)) : -INFINITY;
    }
}

int row_select_ctas(long long ncand, int kcand)
{
    const long long nblk = ncand / kcand;
    return static_cast<int>((nblk + kRowSelCtaKeys - 1) / kRowSelCtaKeys);
}

bool row_select_fits(long long ncand, int kcand, int R)
{
    return R <= kRowSelR && row_select_ctas(ncand, kcand) <= kRowSelMaxCtas;
}

// ----------------------------------------------------------------------------------------
// a6 + a7: exact rerank, then the top-k of the row.  One CTA of 256 threads per (row m,
// candidate j): every thread takes H/2048 16-byte slices of x and of the candidate's bf16 row
// (products of bf16 values are exact in fp32), sums them in two fp32 partials, and the CTA
// combines the 512 partials in float-float arithmetic (an unevaluated sum hi + lo of two
// fp32 values, about 44 significant bits: the CUDA cores' fp32 pipes instead of GB300's few
// fp64 units), rounded once to fp32 at the end.  The last CTA to finish a row (an atomic count per row,
// zeroed by the staging kernel) sorts that row's R exact values and writes its top-k.
// ----------------------------------------------------------------------------------------
constexpr int kRerankThreads = 256;

// Float-float value hi + lo (|lo| <= ulp(hi) / 2 after normalisation).  Explicitly rounded
// operations keep the compiler from contracting or reassociating them.
struct FF {
    float hi, lo;
};

// hi + lo = a + b exactly (Knuth's TwoSum, any magnitudes).
__device__ __forceinline__ FF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return FF{s, e};
}

// a + b for float-float values: the exact sum of the high parts plus both low parts, then
// renormalised (Dekker's FastTwoSum, |s.hi| >= |t| up to the low parts' rounding).
__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    const FF s = two_sum(a.hi, b.hi);
    const float t = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s.hi, t);
    return FF{hi, __fsub_rn(t, __fsub_rn(hi, s.hi))};
}

__device__ __forceinline__ FF ff_shfl_xor(FF v, int o)
{
    return FF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

// The CTA-wide sum of the 256 threads' values, the same order in every caller: an xor-shuffle
// tree per warp, then the eight warps in order (part: eight slots of shared memory).  The
// result reaches thread 0 only, rounded to fp32.
__device__ __forceinline__ FF ff_warp_sum(FF v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
    return v;
}

__device__ __forceinline__ float ff_sum8(const FF *part)
{
    FF t = part[0];
#pragma unroll
    for (int i = 1; i < kRerankThreads / 32; ++i) t = ff_add(t, part[i]);
    return __fadd_rn(t.hi, t.lo);
}

__device__ void sort_write_topk(unsigned long long *k, int n2, int topk, int32_t *oidx,
                                float *ologit);

// One thread's share of the exact logit x . W[n] (n < 0: none), the same arithmetic in every
// caller so that every path reranks to the same bits: the thread takes the 8-weight slices
// i = tid, tid + 256, ... of the row, sums their products in two fp32 partials (products of
// bf16 values are exact in fp32; an fp8 weight is first rounded to fp32(e4m3 * scale)), and
// returns their exact sum as a float-float value.  The caller reduces the 256 values with
// ff_warp_sum and ff_sum8.
template <bool kFp8>
__device__ __forceinline__ FF rerank_partial(const uint16_t *__restrict__ xrow,
                                                 const void *__restrict__ Wv,
                                                 const float *__restrict__ w_scale, int n, int H,
                                                 int tid)
{
    float a0 = 0.f, a1 = 0.f;
    if (n >= 0) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(xrow);
        const int nv = H / 8; // 8 weights per step
        if constexpr (kFp8) {
            const uint2 *wr = reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(Wv) +
                                                              static_cast<long long>(n) * H);
            const float rs = __ldg(w_scale + n);
#pragma unroll 4
            for (int i = tid; i < nv; i += kRerankThreads) {
                const uint4 xv = __ldg(xr + i);
                const uint2 wv = __ldg(wr + i);
                const uint32_t xs4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t wb = (q < 2 ? wv.x : wv.y) >> (16 * (q & 1));
                    a0 = fmaf(__uint_as_float(xs4[q] << 16), __fmul_rn(e4m3_to_f32(wb), rs), a0);
                    a1 = fmaf(__uint_as_float(xs4[q] & 0xFFFF0000u),
                              __fmul_rn(e4m3_to_f32(wb >> 8), rs), a1);
                }
            }
        } else {
            const uint4 *wr = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(Wv) +
                                                              static_cast<long long>(n) * H);
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
    }
    return two_sum(a0, a1);
}

// rerank_partial for NR rows at once (rows n[r] < 0: none), with every row's FMA sequence
// exactly rerank_partial's (slices in increasing i, the same two chains), so each d[r] has
// the same bits.  The slices are taken kBatch at a time with all their loads issued before
// the arithmetic, so the rows' HBM latencies overlap instead of following one another.
template <bool kFp8, int NR>
__device__ __forceinline__ void rerank_partial_rows(const uint16_t *__restrict__ xrow,
                                                    const void *__restrict__ Wv,
                                                    const float *__restrict__ w_scale,
                                                    const int (&n)[NR], int H, int tid,
                                                    FF (&d)[NR])
{
    constexpr int kBatch = 3; // slices per thread in flight (H = 5120: all of them)
    using WVec = typename std::conditional<kFp8, uint2, uint4>::type;
    float a0[NR], a1[NR], rs[NR];
    const WVec *wr[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        a0[r] = 0.f;
        a1[r] = 0.f;
        const long long row = n[r] >= 0 ? n[r] : 0;
        if constexpr (kFp8) {
            wr[r] = reinterpret_cast<const WVec *>(static_cast<const uint8_t *>(Wv) + row * H);
            rs[r] = n[r] >= 0 ? __ldg(w_scale + row) : 0.f;
        } else {
            wr[r] = reinterpret_cast<const WVec *>(static_cast<const uint16_t *>(Wv) + row * H);
            rs[r] = 0.f;
        }
    }
    const uint4 *xr = reinterpret_cast<const uint4 *>(xrow);
    const int nv = H / 8;
    for (int i0 = tid; i0 < nv; i0 += kBatch * kRerankThreads) {
        uint4 xv[kBatch];
        WVec wv[kBatch][NR];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * kRerankThreads;
            if (i < nv) {
                xv[b] = __ldg(xr + i);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    if (n[r] >= 0) wv[b][r] = __ldg(wr[r] + i);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * kRerankThreads;
            if (i >= nv) break;
            const uint32_t xs4[4] = {xv[b].x, xv[b].y, xv[b].z, xv[b].w};
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (n[r] < 0) continue;
                if constexpr (kFp8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t wb = (q < 2 ? wv[b][r].x : wv[b][r].y) >> (16 * (q & 1));
                        a0[r] = fmaf(__uint_as_float(xs4[q] << 16),
                                     __fmul_rn(e4m3_to_f32(wb), rs[r]), a0[r]);
                        a1[r] = fmaf(__uint_as_float(xs4[q] & 0xFFFF0000u),
                                     __fmul_rn(e4m3_to_f32(wb >> 8), rs[r]), a1[r]);
                    }
                } else {
                    const uint32_t ws4[4] = {wv[b][r].x, wv[b][r].y, wv[b][r].z, wv[b][r].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        a0[r] = fmaf(__uint_as_float(xs4[q] << 16), __uint_as_float(ws4[q] << 16),
                                     a0[r]);
                        a1[r] = fmaf(__uint_as_float(xs4[q] & 0xFFFF0000u),
                                     __uint_as_float(ws4[q] & 0xFFFF0000u), a1[r]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) d[r] = two_sum(a0[r], a1[r]);
}

// kFp8: W holds e4m3 rows and w_scale the per-row fp32 scales; each weight is the fp32
// product e4m3(b) * w_scale[n], rounded once (radiance_drafthead.py, _rerank_exact, FP8 branch:
// the selected fp8 rows are dequantised to fp32 before the dot product).  Otherwise W is bf16.
template <bool kFp8>
__global__ void __launch_bounds__(kRerankThreads) rerank_topk_kernel(
    const uint16_t *__restrict__ x, const void *__restrict__ Wv,
    const float *__restrict__ w_scale, int H, int V, const int32_t *__restrict__ sel_idx, int R,
    float *__restrict__ ex, int *__restrict__ row_done, int topk, int32_t *__restrict__ out_idx,
    float *__restrict__ out_logit, int id_offset)
{
    __shared__ FF part[kRerankThreads / 32];
    __shared__ unsigned long long k[kMaxRerank];
    __shared__ int s_last;
    const long long pair = blockIdx.x;
    const int m = static_cast<int>(pair / R);
    const int gid = sel_idx[pair];
    const int n = gid >= 0 ? gid - id_offset : -1; // row of W (a shard starts at id_offset)
    const int tid = threadIdx.x, lane = tid & 31;

    const FF d = ff_warp_sum(rerank_partial<kFp8>(x + static_cast<long long>(m) * H, Wv, w_scale,
                                                  (n >= 0 && n < V) ? n : -1, H, tid));
    if (lane == 0) part[tid >> 5] = d;
    __syncthreads();
    if (tid == 0) {
        const float t = ff_sum8(part);
        ex[pair] = (n >= 0 && n < V) ? t : -INFINITY;
        s_last = 0;
        if (topk > 0) { // only a top-k that follows needs to know which CTA finished last
            __threadfence();
            s_last = atomicAdd(&row_done[m], 1) == R - 1;
        }
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
            const int local = id >= 0 ? id - id_offset : -1;
            if (local >= 0 && local < V)
                key = rank_key(__ldcg(ex + static_cast<long long>(m) * R + i), id);
        }
        k[i] = key;
    }
    __syncthreads();
    sort_write_topk(k, n2, topk, out_idx + static_cast<long long>(m) * topk,
                    out_logit + static_cast<long long>(m) * topk);
}

// ----------------------------------------------------------------------------------------
// a5 + a6 + a7 fused for R <= 32: one cluster of kSrCtas CTAs per batch row, no hand-off
// through global memory between the steps.
//   1. CTA p keeps the 32 best block maxima of its slice of the row's blocks (warp sorts and a
//      tree of warp merges), gathers those blocks' candidates and keeps their 32 best: list
//      L_p in its shared memory.
//   2. After a cluster barrier every CTA merges the kSrCtas lists, read from the other CTAs'
//      shared memory, into the row's 32 best candidates G (rank order).  Exact: a candidate
//      of the row's top 32 has a block among the 32 best maxima of the row, hence of its
//      CTA's slice, and fewer than 32 candidates of that CTA's gathered set beat it.
//   3. CTA p reranks G[p], G[p + kSrCtas], ... with the 256-thread dot product of the rerank
//      kernel (same bits) and writes each exact value's rank key into CTA 0's shared memory.
//   4. After a second cluster barrier CTA 0 sorts the R keys (one warp) and writes the top-k.
// Every CTA finishes its reads of remote shared memory before the second barrier, so no CTA
// exits while another still reads its memory.
// ----------------------------------------------------------------------------------------
constexpr int kSrCtas = 8;      // CTAs per row (a portable cluster)
constexpr int kSrThreads = 256; // = kRerankThreads: the rerank's reduction shape
constexpr int kSrRows = 4;      // reranked rows per CTA: R <= kSrCtas * kSrRows = 32
constexpr int kSrPrefetch = 8;  // weight rows of L_p's best candidates prefetched into L2

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Descending bitonic sort of 32 keys, one per lane.
__device__ __forceinline__ unsigned long long warp_sort32_desc(unsigned long long v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
            v = keep_max ? kmax(v, o) : kmin(v, o);
        }
    }
    return v;
}

// Tree merge of the eight warps' descending lists lists[0..7]; the result in lists[0].  Each
// level's warps read their own slot and one above the level, which nobody writes in it.
__device__ __forceinline__ void tree_merge8(unsigned long long (*lists)[32])
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int n = 4; n >= 1; n >>= 1) {
        if (warp < n) lists[warp][lane] = warp_merge32_desc(lists[warp][lane], lists[warp + n][lane]);
        __syncthreads();
    }
}

template <bool kFp8>
__global__ void __cluster_dims__(kSrCtas, 1, 1) __launch_bounds__(kSrThreads, 1)
    select_rerank_kernel(const float *__restrict__ cand_val, const int32_t *__restrict__ cand_idx,
                         long long ncand, int nblk, int kcand, int R,
                         const uint16_t *__restrict__ x, const void *__restrict__ Wv,
                         const float *__restrict__ w_scale, int H, int V,
                         int32_t *__restrict__ sel_idx, float *__restrict__ ex, int topk,
                         int32_t *__restrict__ out_idx, float *__restrict__ out_logit)
{
    namespace cg = cooperative_groups;
    __shared__ unsigned long long keys[kRowSelR * kBlockN]; // 2048: the largest gather
    __shared__ unsigned long long lists[kSrThreads / 32][32];
    __shared__ unsigned long long mylist[32];               // L_p, read by the cluster
    __shared__ unsigned long long exk[32];                  // CTA 0: the R exact rank keys
    __shared__ FF part[kSrRows][kSrThreads / 32];
    __shared__ int sblk[kRowSelR];
    cg::cluster_group cluster = cg::this_cluster();
    const int p = static_cast<int>(cluster.block_rank());
    const int m = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t wrow_bytes = static_cast<uint32_t>(H) * (kFp8 ? 1u : 2u);
    // x is the caller's input (complete before the staging kernel ran): its row goes to L2 for
    // the rerank while the selection runs
    if (tid == 0) prefetch_l2_bulk(x + static_cast<long long>(m) * H, static_cast<uint32_t>(H) * 2u);
    // launched while the coarse pass may still run: the candidates are its output
    pdl_wait();
    const float *vrow = cand_val + static_cast<long long>(m) * ncand;
    const int32_t *irow = cand_idx + static_cast<long long>(m) * ncand;

    // 1a. the 32 best block maxima of this CTA's slice (a block's first entry is its best);
    // 64 keys per warp and round, so that all eight warps sort
    const int per = (nblk + kSrCtas - 1) / kSrCtas;
    const int b0 = p * per, b1 = min(nblk, b0 + per);
    constexpr int kWarpKeys = 64;
    constexpr int kRound = (kSrThreads / 32) * kWarpKeys; // 512 keys
    unsigned long long acc = 0;
    bool have = false; // warp-uniform: acc holds a list
    for (int base = b0; base < b1; base += kRound) {
        // every load of the round issued before any is used (value and index independently)
        constexpr int kPer = kRound / kSrThreads;
        int ids[kPer];
        float vals[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int bk = base + tid + u * kSrThreads;
            const long long e = static_cast<long long>(bk < b1 ? bk : b0) * kcand;
            ids[u] = __ldcg(irow + e);
            vals[u] = __ldcg(vrow + e);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int bk = base + tid + u * kSrThreads;
            keys[tid + u * kSrThreads] =
                (bk < b1 && ids[u] >= 0) ? rank_key(vals[u], ids[u]) : 0ull;
        }
        __syncthreads();
        if (base + warp * kWarpKeys < b1) { // warp-uniform
            const unsigned long long top = warp_top32_of64(keys + warp * kWarpKeys);
            acc = have ? warp_merge32_desc(acc, top) : top;
            have = true;
        }
        __syncthreads();
    }
    lists[warp][lane] = acc;
    __syncthreads();
    tree_merge8(lists);
    if (tid < kRowSelR) {
        const unsigned long long key = lists[0][tid];
        sblk[tid] = key ? static_cast<int>(~static_cast<uint32_t>(key)) / kBlockN : -1;
    }
    __syncthreads();

    // 1b. those blocks' candidates; their 32 best -> L_p
    const int nc = kRowSelR * kcand;
    const int nchunks = (nc + kRowSelChunk - 1) / kRowSelChunk;
    for (int e0 = 0; e0 < nchunks * kRowSelChunk; e0 += 2 * kSrThreads) {
        int ids[2];
        float vals[2];
        bool live[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = e0 + tid + u * kSrThreads;
            const int bk = e < nc ? sblk[e / kcand] : -1;
            live[u] = bk >= 0;
            const long long c = live[u] ? static_cast<long long>(bk) * kcand + e % kcand : 0;
            ids[u] = __ldcg(irow + c);
            vals[u] = __ldcg(vrow + c);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = e0 + tid + u * kSrThreads;
            if (e < nchunks * kRowSelChunk)
                keys[e] = (live[u] && ids[u] >= 0) ? rank_key(vals[u], ids[u]) : 0ull;
        }
    }
    __syncthreads();
    acc = 0;
    if (nc <= (kSrThreads / 32) * 32) {
        // one 32-key list per warp (entries past nc empty: the gather wrote whole 128-key
        // chunks only, and the rest of keys[] still holds phase 1a's keys): a single sort,
        // then the tree merge
        const int e = warp * 32 + lane;
        acc = warp_sort32_desc(e < nc ? keys[e] : 0ull);
    } else {
        for (int c = warp; c < nchunks; c += kSrThreads / 32)
            acc = warp_merge32_desc(acc, warp_top32_of128(keys + c * kRowSelChunk));
    }
    lists[warp][lane] = acc;
    __syncthreads();
    tree_merge8(lists);
    if (warp == 0) mylist[lane] = lists[0][lane];
    // the weight rows of this CTA's best candidates start on their way to L2: the rows the
    // cluster reranks are the 32 best of the eight lists, mostly near the top of each
    if (tid < kSrPrefetch) {
        const unsigned long long key = lists[0][tid];
        const int id = key ? static_cast<int>(~static_cast<uint32_t>(key)) : -1;
        if (id >= 0 && id < V)
            prefetch_l2_bulk(static_cast<const uint8_t *>(Wv) + static_cast<long long>(id) * wrow_bytes,
                             wrow_bytes);
    }
    cluster.sync();

    // 2. every CTA merges the cluster's lists into G (lists[0], rank order)
    {
        const unsigned long long *rl = cluster.map_shared_rank(mylist, warp % kSrCtas);
        lists[warp][lane] = warp < kSrCtas ? rl[lane] : 0ull;
    }
    __syncthreads();
    tree_merge8(lists);

    // 3. rerank G[p + kSrCtas r] (the four rows' loads in flight together)
    int gid[kSrRows], nrow[kSrRows];
    FF d[kSrRows];
#pragma unroll
    for (int r = 0; r < kSrRows; ++r) {
        const int j = p + kSrCtas * r;
        const unsigned long long key = j < R ? lists[0][j] : 0ull;
        gid[r] = key ? static_cast<int>(~static_cast<uint32_t>(key)) : -1;
        nrow[r] = (gid[r] >= 0 && gid[r] < V) ? gid[r] : -1;
    }
    rerank_partial_rows<kFp8, kSrRows>(x + static_cast<long long>(m) * H, Wv, w_scale, nrow, H,
                                       tid, d);
#pragma unroll
    for (int r = 0; r < kSrRows; ++r) {
        d[r] = ff_warp_sum(d[r]);
        if (lane == 0) part[r][warp] = d[r];
    }
    __syncthreads();
    if (tid < kSrRows) {
        const int r = tid, j = p + kSrCtas * r;
        if (j < R) {
            const float t = ff_sum8(part[r]);
            const bool ok = gid[r] >= 0 && gid[r] < V;
            const float e = ok ? t : -INFINITY;
            sel_idx[static_cast<long long>(m) * R + j] = gid[r];
            ex[static_cast<long long>(m) * R + j] = e;
            unsigned long long *exk0 = cluster.map_shared_rank(exk, 0);
            exk0[j] = ok ? rank_key(e, gid[r]) : 0ull;
        }
    }
    cluster.sync();

    // 4. CTA 0: the row's top-k of the R exact values
    if (p == 0 && warp == 0) {
        const unsigned long long key = warp_sort32_desc(lane < R ? exk[lane] : 0ull);
        if (lane < topk) {
            out_idx[static_cast<long long>(m) * topk + lane] =
                key ? static_cast<int>(~static_cast<uint32_t>(key)) : -1;
            out_logit[static_cast<long long>(m) * topk + lane] =
                key ? f32_from_order_key(static_cast<uint32_t>(key >> 32)) : -INFINITY;
        }
    }
}

// ----------------------------------------------------------------------------------------
// Sharded head, last step: per-rank partial exact values of the R selected ids (each id is
// owned by one rank, the others hold -inf) merged by max, then the row's top-k.  One CTA per
// row.
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRerankThreads) merge_topk_kernel(
    const float *__restrict__ parts, const int32_t *__restrict__ sel_idx, int P, int M, int R,
    int topk, int32_t *__restrict__ out_idx, float *__restrict__ out_logit)
{
    __shared__ unsigned long long k[kMaxRerank];
    const int m = blockIdx.x;
    int n2 = 1;
    while (n2 < R) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += kRerankThreads) {
        unsigned long long key = 0;
        if (i < R) {
            const int id = sel_idx[static_cast<long long>(m) * R + i];
            float e = -INFINITY;
            for (int p = 0; p < P; ++p)
                e = fmaxf(e, parts[(static_cast<long long>(p) * M + m) * R + i]);
            if (id >= 0 && e > -INFINITY) key = rank_key(e, id);
        }
        k[i] = key;
    }
    __syncthreads();
    sort_write_topk(k, n2, topk, out_idx + static_cast<long long>(m) * topk,
                    out_logit + static_cast<long long>(m) * topk);
}

// Sorts n2 (a power of two) keys in shared memory descending with the whole CTA and writes the
// first topk as (index, value); empty keys give (-1, -inf).
__device__ void sort_write_topk(unsigned long long *k, int n2, int topk, int32_t *oidx,
                                float *ologit)
{
    const int tid = threadIdx.x;
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += blockDim.x) {
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
    for (int t = tid; t < topk; t += blockDim.x) {
        const unsigned long long key = k[t];
        const bool ok = key != 0;
        oidx[t] = ok ? static_cast<int>(~static_cast<uint32_t>(key)) : -1;
        ologit[t] = ok ? f32_from_order_key(static_cast<uint32_t>(key >> 32)) : -INFINITY;
    }
}

} // namespace

void select_plan(int M, long long ncand, int kcand, int R, bool blocks, int *passes,
                 long long *scratch_entries)
{
    if (blocks && row_select_fits(ncand, kcand, R)) {
        // the partial lists: M x P x 32 keys of 8 bytes in the first value buffer
        *passes = 1;
        *scratch_entries = static_cast<long long>(M) * row_select_ctas(ncand, kcand) * 32 * 2;
        return;
    }
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
                          int kcand, int R, float *scratch_val[2], int32_t *scratch_idx[2],
                          long long scratch_entries, int *row_cnt, bool blocks,
                          int32_t *sel_idx, float *sel_val, int id_offset, cudaStream_t stream)
{
    (void)scratch_entries;
    if (blocks && row_select_fits(ncand, kcand, R)) {
        const int nblk = static_cast<int>(ncand / kcand);
        dim3 grid(static_cast<unsigned>(row_select_ctas(ncand, kcand)), static_cast<unsigned>(M));
        select_rows_kernel<<<grid, kRowSelThreads, 0, stream>>>(
            cand_val, cand_idx, ncand, nblk, kcand, R,
            reinterpret_cast<unsigned long long *>(scratch_val[0]), row_cnt, sel_idx, sel_val,
            id_offset);
        return cudaGetLastError();
    }
    const float *in_v = cand_val;
    const int32_t *in_i = cand_idx;
    long long stride = ncand, n = ncand;
    int buf = 0;
    for (;;) {
        const long long P = (n + kSelectChunk - 1) / kSelectChunk;
        dim3 grid(static_cast<unsigned>(P), static_cast<unsigned>(M));
        if (P <= 1) {
            topr_kernel<<<grid, kSelThreads, 0, stream>>>(in_v, in_i, stride, n, R, nullptr,
                                                          nullptr, sel_idx, sel_val, id_offset);
            return cudaGetLastError();
        }
        topr_kernel<<<grid, kSelThreads, 0, stream>>>(in_v, in_i, stride, n, R, scratch_val[buf],
                                                      scratch_idx[buf], nullptr, nullptr, 0);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        in_v = scratch_val[buf];
        in_i = scratch_idx[buf];
        n = P * R;
        stride = n;
        buf ^= 1;
    }
}

cudaError_t launch_merge_topk(const float *parts, const int32_t *sel_idx, int P, int M, int R,
                              int topk, int32_t *out_idx, float *out_logit, cudaStream_t stream)
{
    merge_topk_kernel<<<M, kRerankThreads, 0, stream>>>(parts, sel_idx, P, M, R, topk, out_idx,
                                                        out_logit);
    return cudaGetLastError();
}

cudaError_t launch_rerank_topk(const uint16_t *x, const void *W, const float *w_scale, int M,
                               int H, int V,
                               const int32_t *sel_idx, int R, float *ex, int *row_done, int topk,
                               int32_t *out_idx, float *out_logit, int id_offset,
                               cudaStream_t stream)
{
    const unsigned blocks = static_cast<unsigned>(static_cast<long long>(M) * R);
    if (w_scale)
        rerank_topk_kernel<true><<<blocks, kRerankThreads, 0, stream>>>(
            x, W, w_scale, H, V, sel_idx, R, ex, row_done, topk, out_idx, out_logit, id_offset);
    else
        rerank_topk_kernel<false><<<blocks, kRerankThreads, 0, stream>>>(
            x, W, nullptr, H, V, sel_idx, R, ex, row_done, topk, out_idx, out_logit, id_offset);
    return cudaGetLastError();
}

bool select_rerank_fits(int R, int kcand)
{
    return R >= 1 && R <= kSrCtas * kSrRows && R <= kRowSelR && kcand >= 1 && kcand <= kBlockN;
}

cudaError_t launch_select_rerank(const float *cand_val, const int32_t *cand_idx, int M,
                                 long long ncand, int kcand, int R, const uint16_t *x,
                                 const void *W, const float *w_scale, int H, int V,
                                 int32_t *sel_idx, float *ex, int topk, int32_t *out_idx,
                                 float *out_logit, cudaStream_t stream)
{
    const int nblk = static_cast<int>(ncand / kcand);
    const dim3 grid(kSrCtas, static_cast<unsigned>(M));
    if (w_scale)
        return launch_pdl(select_rerank_kernel<true>, grid, dim3(kSrThreads), 0, stream, cand_val,
                          cand_idx, ncand, nblk, kcand, R, x, W, w_scale, H, V, sel_idx, ex, topk,
                          out_idx, out_logit);
    return launch_pdl(select_rerank_kernel<false>, grid, dim3(kSrThreads), 0, stream, cand_val,
                      cand_idx, ncand, nblk, kcand, R, x, W, static_cast<const float *>(nullptr),
                      H, V, sel_idx, ex, topk, out_idx, out_logit);
}

} // namespace dh
