// dh_internal.h -- host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>
#include <utility>

namespace dh {

// ---- geometry shared by the host layer and the kernels ----------------------------------
constexpr int kGroup = 128;             // quantisation group along H
constexpr int kBlockN = 64;             // vocabulary columns per selection block
constexpr int kSpanBytes = 128;         // packed bytes of a row covered by one pass over the planes
constexpr int kNumSMsFallback = 152; // GB300; used only if the device query fails
constexpr int kWarpBatch = 16;          // batch rows per warp-path pass (two n8 tiles)
constexpr int kWarpRowsPerWarp = 64;    // vocabulary rows per warp work item (one block)
constexpr int kSelectChunk = 4096;      // candidates per CTA in one top-R selection pass
constexpr int kMaxRerank = 1024;
constexpr int kMaxM = 128;
constexpr int kNumCounters = 384;   // [0, 64): work queues, [128, 256): per-row rerank
                                    // completion, [256, 384): per-row selection completion
constexpr int kRowDoneOffset = 128;
constexpr int kSelDoneOffset = 256;

// Packed layouts of the head: the 2-bit quarter split (the default), the 4-bit half split, the
// 2-bit contiguous-4 layout (the page's packing ablation) and the quarter split with groups of
// 64 (the page's group-size ablation; S, ZS [V, H/64]).
constexpr int kPackQuarter2 = 0;
constexpr int kPackHalf4 = 1;
constexpr int kPackContig2 = 2;
constexpr int kPackG64 = 3;     // the quarter split with groups of 64 (group-size ablation)
constexpr int kPackWside = 4;   // the quarter split, dequantised on the weight side (bf16
                                // tcgen05 path; the scale-placement ablation)

// ---- per-device host state ---------------------------------------------------------------
// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount), queried
// once per device; the persistent grids are sized from it.
int device_sm_count();

// Launch with programmatic stream serialization: the kernel may be scheduled before its
// predecessor in the stream has finished; it must call pdl_wait() before it reads anything
// the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Host-side set-up that applies to the current device only (a kernel's shared-memory limit):
// run(fn) calls fn once per device, with that device current, and remembers success.
class PerDeviceOnce {
  public:
    template <class F> cudaError_t run(F fn)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return fn(); // untracked: set it every time
        std::lock_guard<std::mutex> lk(mu_);
        if (done_[dev]) return cudaSuccess;
        e = fn();
        if (e == cudaSuccess) done_[dev] = true;
        return e;
    }

  private:
    static constexpr int kMaxDevices = 64;
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
};

// ---- launchers (each returns the launch status) ------------------------------------------
// W: bf16 rows (wsc null) or e4m3 rows with per-row fp32 scales wsc.  bits: 2 (quarter
// split, packed [V, H/4]) or 4 (half split, packed [V, H/2]).  group: 128, or 64 for the
// 2-bit bf16 head of the group-size ablation (S, ZS [V, H/64]).
cudaError_t launch_quantize(const void *W, const float *wsc, int V, int H, int bits, int group,
                            uint8_t *packed, uint16_t *S, uint16_t *ZS, cudaStream_t stream);
// The bf16 head in the contiguous-4 layout, packed [V, H/4].
cudaError_t launch_quantize_c4(const uint16_t *W, int V, int H, uint8_t *packed, uint16_t *S,
                               uint16_t *ZS, cudaStream_t stream);

// x [M,H] bf16 -> group sums xs [Mpad, NGt] fp32 and the operand layouts of the coarse paths:
//   xw (warp path): per 16-row batch chunk, B fragments in mma.sync register order
//   xt (tcgen05 path): [Npad, H] K-major rows with every aligned quad of k permuted [0,2,1,3]
// Rows >= M are zero.  Either of xw / xt may be null.  Also zeroes `counters` (ncounters).
cudaError_t launch_prep(const uint16_t *x, int M, int H, int Mpad, float *xs, uint16_t *xw,
                        uint16_t *xt, int Npad, int *counters, int ncounters,
                        cudaStream_t stream);

struct CoarseArgs {
    const uint16_t *x;  // [M, H] bf16 (the CUDA-core path reads it directly)
    const uint8_t *packed;
    const uint16_t *S;
    const uint16_t *ZS;
    const float *xs;    // [Mpad, NGt]
    const uint16_t *xw; // warp path operand (per chunk)
    const uint16_t *xt; // tcgen05 path operand
    int M, H, V, kcand;
    int pack = 0;       // kPack*: the packed layout (all but the quarter split run on the
                        // 8-bit tcgen05 path only)
    float *cand_val;    // [M, nblk*kcand]
    int32_t *cand_idx;
    float *coarse;      // optional [M, V]
    int *counters;      // work-queue counters, zeroed by prep
    int *timeout_flag;
};

cudaError_t launch_coarse_warp(const CoarseArgs &a, cudaStream_t stream);

// CUDA-core path for M <= 4 (H a multiple of 512): fp32 FMAs on weights made from the packed
// bits, x read from CoarseArgs::x, group sums from xs (core_mpad(M) rows).
bool core_supported(int M, int H);
int core_mpad(int M);
cudaError_t launch_coarse_core(const CoarseArgs &a, cudaStream_t stream);
size_t warp_xw_elems(int M, int H); // bf16 elements of the warp-path operand
// the warp path's shared memory holds its staged x and at least two stages of one warp
bool warp_supported(int M, int H);

// tcgen05 path with 8-bit operands.  The batch runs in launches of at most
// tc8_max_rows(pack, H) rows; launch c pads its rows to MP in {16, 32, 64} and stages them as kTc8Terms e4m3 terms
// ([kTc8Terms * MP, H], term t in rows t * MP ..), of which it uses 2 or 3 (chosen on the
// device from the staged rows' representation error).
constexpr int kTc8Terms = 3;
constexpr int kTc8MaxMP = 64;
int tc8_max_rows(int pack, int H);
struct Tc8Chunk {
    int m0, rows, MP;
    size_t x_off; // byte offset of the launch's staged x in Tc8Workspace::xt8
};
int tc8_chunks(int M, int pack, int H);
Tc8Chunk tc8_chunk(int M, int c, int pack, int H);
size_t tc8_x_bytes(int M, int H); // staged-x bytes, enough for every pack
// Per launch, tc8_small_floats(H) floats: xs of the 2-term and of the 3-term representation
// ([kTc8MaxMP][H / 64] each, scaled units), per-row factors [3][kTc8MaxMP] (2^-e and the
// weights of terms 2 and 3), terms per row [kTc8MaxMP] (int).
inline size_t tc8_small_floats(int H)
{
    return 2 * static_cast<size_t>(kTc8MaxMP) * (H / 64) + 4 * kTc8MaxMP;
}
struct Tc8Workspace {
    uint8_t *xt8;  // staged x of every launch
    float *small;  // per launch tc8_small_floats(H) floats
    int group = 128; // group size of xs (64: the group-size ablation)
};
// xcopy (nullable): a device copy [M, H] of x, written as the rows are read (x may then be
// pinned host memory read across the host link: the rerank reads the copy)
cudaError_t launch_prep_fp8(const uint16_t *x, int M, int H, int pack, const Tc8Workspace &w,
                            int *counters, int ncounters, cudaStream_t stream,
                            uint16_t *xcopy = nullptr);
cudaError_t launch_coarse_tc8(const CoarseArgs &a, const Tc8Workspace &w, cudaStream_t stream);
// the 8-bit tcgen05 path runs these sizes (shared memory and tensor memory fit)
bool tc8_supported(int M, int H, int bits = 2, int group = 128);

bool tc_supported(int M, int H);
cudaError_t launch_coarse_tc(const CoarseArgs &a, cudaStream_t stream);
int tc_npad(int M);
int tc_launches(int M); // coarse-pass launches of the tcgen05 path

// Top-R selection over candidate lists.  `blocks`: the lists are the coarse pass's per-block
// lists (rank-ordered, KCAND per 64-row block), which allows the one-launch path; otherwise a
// generic radix selection runs.  select_plan returns the number of passes it will take and the
// scratch entries it needs (two ping-pong buffers of `scratch_entries` (val, idx) pairs).
// launch_select writes the R best indices plus id_offset to sel_idx [M, R] (-1 when empty) and,
// with sel_val != null, their values.
void select_plan(int M, long long ncand, int kcand, int R, bool blocks, int *passes,
                 long long *scratch_entries);
cudaError_t launch_select(const float *cand_val, const int32_t *cand_idx, int M, long long ncand,
                          int kcand, int R, float *scratch_val[2], int32_t *scratch_idx[2],
                          long long scratch_entries, int *row_cnt, bool blocks,
                          int32_t *sel_idx, float *sel_val, int id_offset, cudaStream_t stream);

// Exact rerank of the selected rows and, fused (last CTA per row), the per-row top-k (topk 0:
// none).  W holds rows [id_offset, id_offset + V) of the head: bf16 (w_scale null) or e4m3
// with per-row fp32 scales w_scale.  Selected ids outside that range get -inf.  row_done: M
// zeroed counters.
cudaError_t launch_rerank_topk(const uint16_t *x, const void *W, const float *w_scale, int M,
                               int H, int V,
                               const int32_t *sel_idx, int R, float *ex, int *row_done, int topk,
                               int32_t *out_idx, float *out_logit, int id_offset,
                               cudaStream_t stream);
// Selection, rerank and top-k fused (R <= 32, any kcand <= 64): one 8-CTA cluster per batch
// row on the coarse pass's block lists; writes sel_idx / ex [M, R] (the reranked ids in rank
// order and their exact values) and the top-k, with the rerank kernel's arithmetic.
bool select_rerank_fits(int R, int kcand);
cudaError_t launch_select_rerank(const float *cand_val, const int32_t *cand_idx, int M,
                                 long long ncand, int kcand, int R, const uint16_t *x,
                                 const void *W, const float *w_scale, int H, int V,
                                 int32_t *sel_idx, float *ex, int topk, int32_t *out_idx,
                                 float *out_logit, cudaStream_t stream);
// Per-rank partial exact values parts [P, M, R] merged by max, then the per-row top-k.
cudaError_t launch_merge_topk(const float *parts, const int32_t *sel_idx, int P, int M, int R,
                              int topk, int32_t *out_idx, float *out_logit, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
CUresult encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

} // namespace dh
