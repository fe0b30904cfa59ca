// dh_api.cu -- host layer of the draft-head library: the C ABI declared in include/dh.h.
//
// Every entry point validates its arguments on the host, carves the caller's workspace, and
// enqueues the kernels on the caller's stream.  Nothing here allocates device memory,
// synchronises (except dh_device_status, which exists to read a flag) or touches the host
// copy of any tensor.
#include "dh.h"
#include "dh_internal.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace dh {

namespace {

thread_local std::string g_last_error;
int g_path = DH_PATH_AUTO;
std::mutex g_path_mu;

// Set by any kernel whose bounded wait gave up.  The host learns its address per device.
__device__ int g_timeout_flag;

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int ok()
{
    g_last_error.clear();
    return DH_OK;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

size_t align256(size_t v)
{
    return (v + 255u) & ~static_cast<size_t>(255u);
}

int *timeout_flag_ptr()
{
    // one address per device; the symbol address is resolved with that device current
    static std::mutex mu;
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_timeout_flag) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int *>(p);
    }
    return addr[dev];
}

} // namespace

int device_sm_count()
{
    static std::mutex mu;
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kNumSMsFallback;
    std::lock_guard<std::mutex> lk(mu);
    if (count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return kNumSMsFallback;
        count[dev] = n;
    }
    return count[dev];
}

namespace {

long long valid_candidates(int V, int kcand)
{
    const long long nblk = (V + kBlockN - 1) / kBlockN;
    const int kc = kcand < kBlockN ? kcand : kBlockN;
    const int tail = V - static_cast<int>((nblk - 1) * kBlockN);
    return (nblk - 1) * kc + (kcand < tail ? kcand : tail);
}

struct Layout {
    int Mpad_w = 0, Npad = 0, rows = 0;
    long long nblk = 0, ncand = 0, scratch_entries = 0;
    int passes = 0;
    size_t xs = 0, xw = 0, xt = 0, cval = 0, cidx = 0, sval[2] = {0, 0}, sidx[2] = {0, 0},
           sel = 0, ex = 0, counters = 0, xt8 = 0, small8 = 0, xcopy = 0, total = 0;
};


Layout layout_for(int M, int H, int V, int kcand, int rerank)
{
    Layout L;
    L.Mpad_w = ((M + kWarpBatch - 1) / kWarpBatch) * kWarpBatch;
    L.Npad = tc_npad(M);
    L.rows = L.Mpad_w > L.Npad ? L.Mpad_w : L.Npad;
    L.nblk = (V + kBlockN - 1) / kBlockN;
    L.ncand = L.nblk * kcand;
    select_plan(M, L.ncand, kcand, rerank, true, &L.passes, &L.scratch_entries);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    L.xs = take(static_cast<size_t>(L.rows) * (H / kGroup) * 4);
    L.xw = take(warp_xw_elems(M, H) * 2);
    L.xt = take(static_cast<size_t>(L.Npad) * H * 2);
    L.cval = take(static_cast<size_t>(M) * L.ncand * 4);
    L.cidx = take(static_cast<size_t>(M) * L.ncand * 4);
    for (int b = 0; b < 2; ++b) {
        L.sval[b] = take(static_cast<size_t>(L.scratch_entries) * 4);
        L.sidx[b] = take(static_cast<size_t>(L.scratch_entries) * 4);
    }
    L.sel = take(static_cast<size_t>(M) * rerank * 4);
    L.ex = take(static_cast<size_t>(M) * rerank * 4);
    L.counters = take(kNumCounters * 4);
    // the 8-bit path's staged x (the largest any packed layout needs) and, per launch, the
    // small per-row data (group sums, 2^-e, term weights and counts); the 4-bit layout takes
    // the most launches (16 rows each)
    L.xt8 = take(tc8_x_bytes(M, H));
    L.small8 = take(static_cast<size_t>(tc8_chunks(M, kPackHalf4, H)) * tc8_small_floats(H) * 4);
    // a device copy of x for the calls that take x in host memory (dh_forward_host)
    L.xcopy = take(static_cast<size_t>(M) * H * 2);
    L.total = off;
    return L;
}

int check_shapes(int M, int H, int V, int kcand, int rerank, int topk)
{
    if (M < 1 || M > kMaxM) return fail(DH_ERR_SHAPE, "M=%d outside [1, %d]", M, kMaxM);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (static_cast<long long>(V) * H / 4 > (1LL << 40))
        return fail(DH_ERR_SHAPE, "V*H=%lld too large", static_cast<long long>(V) * H);
    if (kcand < 1 || kcand > kBlockN)
        return fail(DH_ERR_SELECT, "kcand=%d outside [1, %d]", kcand, kBlockN);
    long long nv = valid_candidates(V, kcand);
    long long rmax = nv < kMaxRerank ? nv : kMaxRerank;
    if (rerank < 1 || rerank > rmax)
        return fail(DH_ERR_SELECT, "rerank=%d outside [1, %lld] (valid candidates %lld)", rerank,
                    rmax, nv);
    if (topk < 1 || topk > rerank)
        return fail(DH_ERR_SELECT, "topk=%d outside [1, rerank=%d]", topk, rerank);
    return DH_OK;
}

int choose_path(int M, int H)
{
    int p;
    {
        std::lock_guard<std::mutex> lk(g_path_mu);
        p = g_path;
    }
    if (p == DH_PATH_TC) return tc8_supported(M, H) ? p : -1;
    if (p == DH_PATH_TC_BF16) return tc_supported(M, H) ? p : -1;
    if (p == DH_PATH_WARP) return warp_supported(M, H) ? p : -1;
    if (p == DH_PATH_CORE) return core_supported(M, H) ? p : -1;
    // automatic: the 8-bit tcgen05 path where it is available, else the warp path
    if (tc8_supported(M, H)) return DH_PATH_TC;
    return warp_supported(M, H) ? DH_PATH_WARP : -1;
}

// W: the head's rows for the rerank, bf16 (w_scale null) or e4m3 with per-row fp32 scales.
int forward_impl(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                 const uint16_t *zeros, const void *W, int M, int H, int V, int kcand,
                 int rerank, int topk, int32_t *idx, float *logit, void *workspace,
                 size_t ws_bytes, float *coarse, float *cand_val, int32_t *cand_idx,
                 int32_t *sel_idx, float *sel_exact, void *const *events, cudaStream_t stream,
                 float *sel_val = nullptr, int id_offset = 0, bool candidates_only = false,
                 const float *w_scale = nullptr, int pack = kPackQuarter2,
                 uint16_t *x_copy = nullptr)
{
    // x_copy (8-bit tcgen05 path only): the staging kernel writes a device copy of x there as
    // it reads x (which may then be pinned host memory), and the rerank reads the copy
    // candidates_only: stop after the top-R selection (a vocabulary shard's local candidates,
    // indices offset by id_offset, values into sel_val); W, idx and logit are not used
    if (candidates_only) {
        if (!x || !packed || !scales || !zeros || !sel_idx || !sel_val || !workspace)
            return fail(DH_ERR_NULL, "a required pointer is NULL");
    } else if (!x || !packed || !scales || !zeros || !W || !idx || !logit || !workspace) {
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    }
    int rc = check_shapes(M, H, V, kcand, rerank, candidates_only ? 1 : topk);
    if (rc != DH_OK) return rc;
    const void *ptrs[] = {x, packed, scales, zeros, workspace};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    if (!candidates_only && (!aligned16(W) || !aligned16(idx) || !aligned16(logit)))
        return fail(DH_ERR_ALIGN, "W, idx or logit is not 16-byte aligned");
    const Layout L = layout_for(M, H, V, kcand, rerank);
    if (ws_bytes < L.total)
        return fail(DH_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, L.total);
    int path = choose_path(M, H);
    if (pack == kPackWside) // the weight-side ablation runs on the bf16 tcgen05 path
        path = tc_supported(M, H) ? DH_PATH_TC_BF16 : -1;
    if (path < 0)
        return fail(DH_ERR_ARG, "no coarse path takes M=%d, H=%d (the one set by dh_set_coarse_path, "
                                "or with the automatic choice none fits its shared memory)", M, H);
    if (pack != kPackQuarter2 && pack != kPackWside &&
        (path != DH_PATH_TC || !tc8_supported(M, H, pack == kPackHalf4 ? 4 : 2,
                                              pack == kPackG64 ? 64 : 128)))
        return fail(DH_ERR_ARG,
                    "the %s head runs on the 8-bit tcgen05 path only (M=%d, H=%d: %s)",
                    pack == kPackHalf4 ? "4-bit"
                                       : (pack == kPackG64 ? "64-group" : "contiguous-4"),
                    M, H,
                    path != DH_PATH_TC ? "another coarse path is selected"
                                       : "the path does not take these sizes");
    int *tflag = timeout_flag_ptr();
    if (!tflag) return fail(DH_ERR_CUDA, "cannot resolve the device status flag");

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *xs = reinterpret_cast<float *>(ws + L.xs);
    uint16_t *xw = reinterpret_cast<uint16_t *>(ws + L.xw);
    uint16_t *xt = reinterpret_cast<uint16_t *>(ws + L.xt);
    float *cval = cand_val ? cand_val : reinterpret_cast<float *>(ws + L.cval);
    int32_t *cidx = cand_idx ? cand_idx : reinterpret_cast<int32_t *>(ws + L.cidx);
    float *sv[2] = {reinterpret_cast<float *>(ws + L.sval[0]), reinterpret_cast<float *>(ws + L.sval[1])};
    int32_t *si[2] = {reinterpret_cast<int32_t *>(ws + L.sidx[0]),
                      reinterpret_cast<int32_t *>(ws + L.sidx[1])};
    int32_t *sel = sel_idx ? sel_idx : reinterpret_cast<int32_t *>(ws + L.sel);
    float *ex = sel_exact ? sel_exact : reinterpret_cast<float *>(ws + L.ex);
    int *counters = reinterpret_cast<int *>(ws + L.counters);

    auto rec = [&](int i) -> bool {
        return !events || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess;
    };
    cudaError_t err;
    if (!rec(0)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
    Tc8Workspace w8;
    w8.xt8 = ws + L.xt8;
    w8.small = reinterpret_cast<float *>(ws + L.small8);
    w8.group = pack == kPackG64 ? 64 : 128;
    if (x_copy && path != DH_PATH_TC)
        return fail(DH_ERR_ARG, "x_copy needs the 8-bit tcgen05 path");
    const uint16_t *x_rr = x_copy ? x_copy : x; // the x the rerank reads
    if (path == DH_PATH_TC)
        err = launch_prep_fp8(x, M, H, pack, w8, counters, kNumCounters, stream, x_copy);
    else if (path == DH_PATH_CORE)
        err = launch_prep(x, M, H, core_mpad(M), xs, nullptr, nullptr, 0, counters,
                          kNumCounters, stream);
    else
        err = launch_prep(x, M, H, path == DH_PATH_WARP ? L.Mpad_w : 0, xs,
                          path == DH_PATH_WARP ? xw : nullptr,
                          path == DH_PATH_TC_BF16 ? xt : nullptr,
                          path == DH_PATH_TC_BF16 ? L.Npad : 0, counters, kNumCounters, stream);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "prep launch: %s", cudaGetErrorString(err));
    if (!rec(1)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");

    CoarseArgs a;
    a.x = x;
    a.packed = packed;
    a.S = scales;
    a.ZS = zeros;
    a.xs = xs;
    a.xw = xw;
    a.xt = xt;
    a.M = M;
    a.H = H;
    a.V = V;
    a.kcand = kcand;
    a.pack = pack;
    a.cand_val = cval;
    a.cand_idx = cidx;
    a.coarse = coarse;
    a.counters = counters;
    a.timeout_flag = tflag;
    if (path == DH_PATH_TC) err = launch_coarse_tc8(a, w8, stream);
    else if (path == DH_PATH_TC_BF16) err = launch_coarse_tc(a, stream);
    else if (path == DH_PATH_CORE) err = launch_coarse_core(a, stream);
    else err = launch_coarse_warp(a, stream);
    if (err != cudaSuccess)
        return fail(DH_ERR_CUDA, "coarse launch (%s path): %s",
                    path == DH_PATH_TC
                        ? "tcgen05 8-bit"
                        : (path == DH_PATH_TC_BF16 ? "tcgen05 bf16"
                                                   : (path == DH_PATH_CORE ? "CUDA-core" : "warp")),
                    cudaGetErrorString(err));
    if (!rec(2)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
    if (!candidates_only && select_rerank_fits(rerank, kcand)) {
        // one launch for the selection, the rerank and the top-k (the stage events 3 and 4
        // then enclose nothing)
        err = launch_select_rerank(cval, cidx, M, L.ncand, kcand, rerank, x_rr, W, w_scale, H,
                                   V, sel, ex, topk, idx, logit, stream);
        if (err != cudaSuccess)
            return fail(DH_ERR_CUDA, "select/rerank launch: %s", cudaGetErrorString(err));
        if (!rec(3) || !rec(4) || !rec(5)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
        return ok();
    }
    err = launch_select(cval, cidx, M, L.ncand, kcand, rerank, sv, si, L.scratch_entries,
                        counters + kSelDoneOffset, true, sel, sel_val, id_offset, stream);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "select launch: %s", cudaGetErrorString(err));
    if (candidates_only) return ok();
    if (!rec(3)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
    err = launch_rerank_topk(x_rr, W, w_scale, M, H, V, sel, rerank, ex,
                             counters + kRowDoneOffset, topk, idx, logit, 0, stream);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "rerank launch: %s", cudaGetErrorString(err));
    if (!rec(4)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
    if (!rec(5)) return fail(DH_ERR_CUDA, "cudaEventRecord failed");
    return ok();
}

// Fixed scratch of dh_forward_noalloc: the whole forward workspace for callers that cannot
// allocate.  Host code must not use this name as an address (it is a host-side stand-in);
// its device address is resolved per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DH_NOALLOC_WORKSPACE_BYTES];

// Device address of g_noalloc_scratch on the current device, resolved once per device with
// that device current; nullptr if the runtime cannot resolve it.
void *noalloc_scratch_ptr()
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

} // namespace

CUresult encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

} // namespace dh

using namespace dh;

extern "C" {

int dh_quantize(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                uint16_t *zeros, void *stream)
{
    if (!W_bf16 || !packed || !scales || !zeros)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    const void *ptrs[] = {W_bf16, packed, scales, zeros};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    cudaError_t err = launch_quantize(W_bf16, nullptr, V, H, 2, 128, packed, scales, zeros,
                                      static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(err));
    return ok();
}

size_t dh_workspace_bytes(int M, int H, int V, int kcand, int rerank)
{
    if (check_shapes(M, H, V, kcand, rerank, 1) != DH_OK) return 0;
    return layout_for(M, H, V, kcand, rerank).total;
}

int dh_forward(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
               const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V, int kcand,
               int rerank, int topk, int32_t *idx, float *logit, void *workspace,
               size_t ws_bytes, void *stream)
{
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                        nullptr, static_cast<cudaStream_t>(stream));
}

int dh_forward_host(const uint16_t *x_host, const uint8_t *packed, const uint16_t *scales,
                    const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                    int kcand, int rerank, int topk, int32_t *idx_host, float *logit_host,
                    void *workspace, size_t ws_bytes, void *stream)
{
    if (!x_host || !idx_host || !logit_host || !workspace)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    // every host buffer must be pinned and mapped into the device's address space; its device
    // address is what the kernels use (checked here, before anything runs)
    const void *host_ptrs[3] = {x_host, idx_host, logit_host};
    void *dev_ptrs[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i < 3; ++i) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, host_ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return fail(DH_ERR_ARG, "cannot query pointer %p", host_ptrs[i]);
        }
        if (a.type != cudaMemoryTypeHost || !a.devicePointer)
            return fail(DH_ERR_ARG,
                        "%s at %p is not pinned host memory mapped into the device's address space",
                        i == 0 ? "x" : (i == 1 ? "idx" : "logit"), host_ptrs[i]);
        dev_ptrs[i] = a.devicePointer;
    }
    int rc = check_shapes(M, H, V, kcand, rerank, topk);
    if (rc != DH_OK) return rc;
    if (!aligned16(workspace)) return fail(DH_ERR_ALIGN, "workspace is not 16-byte aligned");
    const Layout L = layout_for(M, H, V, kcand, rerank);
    if (ws_bytes < L.total)
        return fail(DH_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, L.total);
    uint16_t *xc = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) + L.xcopy);
    const auto *xd = static_cast<const uint16_t *>(dev_ptrs[0]);
    auto *id = static_cast<int32_t *>(dev_ptrs[1]);
    auto *ld = static_cast<float *>(dev_ptrs[2]);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (choose_path(M, H) == DH_PATH_TC) // the staging kernel reads x across the host link
        return forward_impl(xd, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, id,
                            ld, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                            nullptr, st, nullptr, 0, false, nullptr, kPackQuarter2, xc);
    // the other coarse paths: one copy of x to the device first
    if (!aligned16(xd)) return fail(DH_ERR_ALIGN, "x is not 16-byte aligned");
    const cudaError_t e = cudaMemcpyAsync(xc, x_host, static_cast<size_t>(M) * H * 2,
                                          cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail(DH_ERR_CUDA, "copy of x: %s", cudaGetErrorString(e));
    return forward_impl(xc, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, id, ld,
                        workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                        st);
}

int dh_quantize_fp8(const uint8_t *W_e4m3, const float *row_scale, int V, int H, uint8_t *packed,
                    uint16_t *scales, uint16_t *zeros, void *stream)
{
    if (!W_e4m3 || !row_scale || !packed || !scales || !zeros)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    const void *ptrs[] = {W_e4m3, packed, scales, zeros};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    if (reinterpret_cast<uintptr_t>(row_scale) & 3u)
        return fail(DH_ERR_ALIGN, "row_scale %p is not 4-byte aligned", row_scale);
    cudaError_t err = launch_quantize(W_e4m3, row_scale, V, H, 2, 128, packed, scales, zeros,
                                      static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_forward_fp8w(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                    const uint16_t *zeros, const uint8_t *W_e4m3, const float *row_scale, int M,
                    int H, int V, int kcand, int rerank, int topk, int32_t *idx, float *logit,
                    void *workspace, size_t ws_bytes, void *stream)
{
    if (!row_scale) return fail(DH_ERR_NULL, "row_scale is NULL");
    if (reinterpret_cast<uintptr_t>(row_scale) & 3u)
        return fail(DH_ERR_ALIGN, "row_scale %p is not 4-byte aligned", row_scale);
    return forward_impl(x, packed, scales, zeros, W_e4m3, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                        nullptr, static_cast<cudaStream_t>(stream), nullptr, 0, false, row_scale);
}

int dh_quantize4(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                 uint16_t *zeros, void *stream)
{
    if (!W_bf16 || !packed || !scales || !zeros)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    const void *ptrs[] = {W_bf16, packed, scales, zeros};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    cudaError_t err = launch_quantize(W_bf16, nullptr, V, H, 4, 128, packed, scales, zeros,
                                      static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_forward4(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V, int kcand,
                int rerank, int topk, int32_t *idx, float *logit, void *workspace,
                size_t ws_bytes, void *stream)
{
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                        nullptr, static_cast<cudaStream_t>(stream), nullptr, 0, false, nullptr,
                        kPackHalf4);
}

int dh_forward4_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                      const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                      int kcand, int rerank, int topk, int32_t *idx, float *logit,
                      void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                      int32_t *cand_idx, int32_t *sel_idx, float *sel_exact, void *stream)
{
    const void *opt[] = {coarse, cand_val, cand_idx, sel_idx, sel_exact};
    for (const void *p : opt)
        if (p && !aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, coarse, cand_val, cand_idx, sel_idx,
                        sel_exact, nullptr, static_cast<cudaStream_t>(stream), nullptr, 0, false,
                        nullptr, kPackHalf4);
}

int dh_forward4_timed(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                      const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                      int kcand, int rerank, int topk, int32_t *idx, float *logit,
                      void *workspace, size_t ws_bytes, void *const *events, void *stream)
{
    if (!events) return fail(DH_ERR_NULL, "events is NULL");
    for (int i = 0; i < DH_NUM_STAGE_EVENTS; ++i)
        if (!events[i]) return fail(DH_ERR_NULL, "events[%d] is NULL", i);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                        events, static_cast<cudaStream_t>(stream), nullptr, 0, false, nullptr,
                        kPackHalf4);
}

int dh_quantize_c4(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                   uint16_t *zeros, void *stream)
{
    if (!W_bf16 || !packed || !scales || !zeros)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    const void *ptrs[] = {W_bf16, packed, scales, zeros};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    cudaError_t err = launch_quantize_c4(W_bf16, V, H, packed, scales, zeros,
                                         static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_forward_c4_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                        int kcand, int rerank, int topk, int32_t *idx, float *logit,
                        void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                        int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                        void *const *events, void *stream)
{
    const void *opt[] = {coarse, cand_val, cand_idx, sel_idx, sel_exact};
    for (const void *p : opt)
        if (p && !aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    if (events)
        for (int i = 0; i < DH_NUM_STAGE_EVENTS; ++i)
            if (!events[i]) return fail(DH_ERR_NULL, "events[%d] is NULL", i);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, coarse, cand_val, cand_idx, sel_idx,
                        sel_exact, events, static_cast<cudaStream_t>(stream), nullptr, 0, false,
                        nullptr, kPackContig2);
}

int dh_quantize_g64(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                    uint16_t *zeros, void *stream)
{
    if (!W_bf16 || !packed || !scales || !zeros)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    const void *ptrs[] = {W_bf16, packed, scales, zeros};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    cudaError_t err = launch_quantize(W_bf16, nullptr, V, H, 2, 64, packed, scales, zeros,
                                      static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_forward_g64_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                         const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                         int kcand, int rerank, int topk, int32_t *idx, float *logit,
                         void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                         int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                         void *const *events, void *stream)
{
    const void *opt[] = {coarse, cand_val, cand_idx, sel_idx, sel_exact};
    for (const void *p : opt)
        if (p && !aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    if (events)
        for (int i = 0; i < DH_NUM_STAGE_EVENTS; ++i)
            if (!events[i]) return fail(DH_ERR_NULL, "events[%d] is NULL", i);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, coarse, cand_val, cand_idx, sel_idx,
                        sel_exact, events, static_cast<cudaStream_t>(stream), nullptr, 0, false,
                        nullptr, kPackG64);
}

int dh_forward_wside_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                           const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                           int kcand, int rerank, int topk, int32_t *idx, float *logit,
                           void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                           int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                           void *const *events, void *stream)
{
    const void *opt[] = {coarse, cand_val, cand_idx, sel_idx, sel_exact};
    for (const void *p : opt)
        if (p && !aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    if (events)
        for (int i = 0; i < DH_NUM_STAGE_EVENTS; ++i)
            if (!events[i]) return fail(DH_ERR_NULL, "events[%d] is NULL", i);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, coarse, cand_val, cand_idx, sel_idx,
                        sel_exact, events, static_cast<cudaStream_t>(stream), nullptr, 0, false,
                        nullptr, kPackWside);
}

int dh_forward_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                     const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                     int kcand, int rerank, int topk, int32_t *idx, float *logit,
                     void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                     int32_t *cand_idx, int32_t *sel_idx, float *sel_exact, void *stream)
{
    const void *opt[] = {coarse, cand_val, cand_idx, sel_idx, sel_exact};
    for (const void *p : opt)
        if (p && !aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, coarse, cand_val, cand_idx, sel_idx,
                        sel_exact, nullptr, static_cast<cudaStream_t>(stream));
}

int dh_forward_timed(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                     const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                     int kcand, int rerank, int topk, int32_t *idx, float *logit,
                     void *workspace, size_t ws_bytes, void *const *events, void *stream)
{
    if (!events) return fail(DH_ERR_NULL, "events is NULL");
    for (int i = 0; i < DH_NUM_STAGE_EVENTS; ++i)
        if (!events[i]) return fail(DH_ERR_NULL, "events[%d] is NULL", i);
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                        events, static_cast<cudaStream_t>(stream));
}

int dh_forward_noalloc(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                       int kcand, int rerank, int topk, int32_t *idx, float *logit,
                       void *stream)
{
    if (!x || !packed || !scales || !zeros || !W_bf16 || !idx || !logit)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    int rc = check_shapes(M, H, V, kcand, rerank, topk);
    if (rc != DH_OK) return rc;
    const size_t need = layout_for(M, H, V, kcand, rerank).total;
    if (need > DH_NOALLOC_WORKSPACE_BYTES)
        return fail(DH_ERR_WORKSPACE,
                    "M=%d H=%d V=%d kcand=%d rerank=%d need %zu bytes of scratch; the fixed "
                    "buffer of dh_forward_noalloc holds %u (use dh_forward with a workspace)",
                    M, H, V, kcand, rerank, need, DH_NOALLOC_WORKSPACE_BYTES);
    void *ws = noalloc_scratch_ptr();
    if (!ws) return fail(DH_ERR_CUDA, "cannot resolve the device address of the fixed scratch");
    return forward_impl(x, packed, scales, zeros, W_bf16, M, H, V, kcand, rerank, topk, idx,
                        logit, ws, DH_NOALLOC_WORKSPACE_BYTES, nullptr, nullptr, nullptr,
                        nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

int dh_set_coarse_path(int path)
{
    if (path != DH_PATH_AUTO && path != DH_PATH_WARP && path != DH_PATH_TC &&
        path != DH_PATH_TC_BF16 && path != DH_PATH_CORE)
        return fail(DH_ERR_ARG, "unknown coarse path %d", path);
    std::lock_guard<std::mutex> lk(g_path_mu);
    const int prev = g_path;
    g_path = path;
    return prev;
}

int dh_coarse_path_for(int M)
{
    if (M < 1 || M > kMaxM) return fail(DH_ERR_SHAPE, "M=%d outside [1, %d]", M, kMaxM);
    return choose_path(M, 5120);
}

int dh_forward_launch_count(int M, int H, int V, int kcand, int rerank)
{
    if (check_shapes(M, H, V, kcand, rerank, 1) != DH_OK) return 0;
    const Layout L = layout_for(M, H, V, kcand, rerank);
    const int path = choose_path(M, H);
    if (path < 0) return 0;
    int prep = 1, coarse = (M + kWarpBatch - 1) / kWarpBatch;
    if (path == DH_PATH_TC) coarse = tc8_chunks(M, kPackQuarter2, H); // one staging launch
    else if (path == DH_PATH_TC_BF16) coarse = tc_launches(M);
    else if (path == DH_PATH_CORE) coarse = 1;
    if (select_rerank_fits(rerank, kcand)) return prep + coarse + 1; // fused select + rerank
    return prep + coarse + L.passes /*selection*/ + 1 /*rerank + top-k*/;
}

int dh_device_status(int reset)
{
    int *p = timeout_flag_ptr();
    if (!p) return fail(DH_ERR_CUDA, "cannot resolve the device status flag");
    if (cudaDeviceSynchronize() != cudaSuccess)
        return fail(DH_ERR_CUDA, "device synchronize failed");
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail(DH_ERR_CUDA, "cannot read the device status flag");
    if (reset) {
        const int z = 0;
        if (cudaMemcpy(p, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess)
            return fail(DH_ERR_CUDA, "cannot reset the device status flag");
    }
    if (v) return fail(DH_ERR_DEVICE_TIMEOUT, "a device-side wait timed out");
    return ok();
}

const char *dh_last_error(void)
{
    return g_last_error.c_str();
}

int dh_version(void)
{
    return (1 << 16) | 4;
}


// ---- vocabulary-parallel head ------------------------------------------------------------

int dh_shard_candidates(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, int M, int H, int Vs, long long vocab_offset,
                        int kcand, int rerank, float *out_val, int32_t *out_idx,
                        void *workspace, size_t ws_bytes, void *stream)
{
    if (vocab_offset < 0 || vocab_offset % kBlockN != 0)
        return fail(DH_ERR_SHAPE, "vocab_offset=%lld is not a non-negative multiple of %d",
                    vocab_offset, kBlockN);
    if (Vs >= 1 && vocab_offset + Vs > 0x7FFFFFFFLL)
        return fail(DH_ERR_SHAPE, "vocab_offset + Vs exceeds the 32-bit index range");
    return forward_impl(x, packed, scales, zeros, nullptr, M, H, Vs, kcand, rerank, 1, nullptr,
                        nullptr, workspace, ws_bytes, nullptr, nullptr, nullptr, out_idx, nullptr,
                        nullptr, static_cast<cudaStream_t>(stream), out_val,
                        static_cast<int>(vocab_offset), true);
}

size_t dh_shard_rerank_workspace_bytes(int M, long long ncand_all, int rerank)
{
    if (M < 1 || M > kMaxM || ncand_all < 1 || rerank < 1 || rerank > kMaxRerank ||
        rerank > ncand_all)
        return 0;
    int passes = 0;
    long long entries = 0;
    select_plan(M, ncand_all, 1, rerank, false, &passes, &entries);
    // two ping-pong (value, index) buffers of `entries`, then the counters
    return 4 * align256(static_cast<size_t>(entries) * 4) + align256(kNumCounters * 4);
}

int dh_rerank(const uint16_t *x, const uint16_t *W_bf16, int M, int H, int V, const int32_t *idx,
              long long n, float *exact, void *stream)
{
    if (!x || !W_bf16 || !idx || !exact) return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (M < 1 || M > kMaxM) return fail(DH_ERR_SHAPE, "M=%d outside [1, %d]", M, kMaxM);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    if (V < 1) return fail(DH_ERR_SHAPE, "V=%d must be >= 1", V);
    if (n < 1 || n * M > 0x7FFFFFFFLL)
        return fail(DH_ERR_SHAPE, "n=%lld: need 1 <= n and M n < 2^31", n);
    const void *ptrs[] = {x, W_bf16};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    cudaError_t err = launch_rerank_topk(x, W_bf16, nullptr, M, H, V, idx, static_cast<int>(n),
                                         exact, nullptr, 0, nullptr, nullptr, 0,
                                         static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "rerank launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_shard_rerank(const uint16_t *x, const uint16_t *W_shard, int M, int H, int Vs,
                    long long vocab_offset, const float *all_val, const int32_t *all_idx,
                    long long ncand_all, int rerank, int32_t *sel_idx, float *exact,
                    void *workspace, size_t ws_bytes, void *stream)
{
    if (!x || !W_shard || !all_val || !all_idx || !sel_idx || !exact || !workspace)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (M < 1 || M > kMaxM) return fail(DH_ERR_SHAPE, "M=%d outside [1, %d]", M, kMaxM);
    if (H <= 0 || H % 512 != 0)
        return fail(DH_ERR_SHAPE, "H=%d is not a positive multiple of 512", H);
    if (Vs < 1) return fail(DH_ERR_SHAPE, "Vs=%d must be >= 1", Vs);
    if (vocab_offset < 0 || vocab_offset + Vs > 0x7FFFFFFFLL)
        return fail(DH_ERR_SHAPE, "vocab_offset=%lld out of range", vocab_offset);
    if (ncand_all < 1 || rerank < 1 || rerank > kMaxRerank || rerank > ncand_all)
        return fail(DH_ERR_SELECT, "rerank=%d outside [1, min(%lld, %d)]", rerank, ncand_all,
                    kMaxRerank);
    const void *ptrs[] = {x, W_shard, workspace};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(DH_ERR_ALIGN, "pointer %p is not 16-byte aligned", p);
    const size_t need = dh_shard_rerank_workspace_bytes(M, ncand_all, rerank);
    if (ws_bytes < need)
        return fail(DH_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
    int passes = 0;
    long long entries = 0;
    select_plan(M, ncand_all, 1, rerank, false, &passes, &entries);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t eb = align256(static_cast<size_t>(entries) * 4);
    float *sv[2] = {reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + eb)};
    int32_t *si[2] = {reinterpret_cast<int32_t *>(ws + 2 * eb),
                      reinterpret_cast<int32_t *>(ws + 3 * eb)};
    int *counters = reinterpret_cast<int *>(ws + 4 * eb);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaMemsetAsync(counters, 0, kNumCounters * 4, st);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "counter reset: %s", cudaGetErrorString(err));
    // the global top-R over every shard's local candidates: the same on every rank
    err = launch_select(all_val, all_idx, M, ncand_all, 1, rerank, sv, si, entries,
                        counters + kSelDoneOffset, false, sel_idx, nullptr, 0, st);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "select launch: %s", cudaGetErrorString(err));
    // exact values of the ids this shard owns; the others get -inf
    err = launch_rerank_topk(x, W_shard, nullptr, M, H, Vs, sel_idx, rerank, exact,
                             counters + kRowDoneOffset, 0, nullptr, nullptr,
                             static_cast<int>(vocab_offset), st);
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "rerank launch: %s", cudaGetErrorString(err));
    return ok();
}

int dh_shard_topk(const float *exact_parts, const int32_t *sel_idx, int P, int M, int rerank,
                  int topk, int32_t *idx, float *logit, void *stream)
{
    if (!exact_parts || !sel_idx || !idx || !logit)
        return fail(DH_ERR_NULL, "a required pointer is NULL");
    if (P < 1) return fail(DH_ERR_ARG, "P=%d must be >= 1", P);
    if (M < 1 || M > kMaxM) return fail(DH_ERR_SHAPE, "M=%d outside [1, %d]", M, kMaxM);
    if (rerank < 1 || rerank > kMaxRerank)
        return fail(DH_ERR_SELECT, "rerank=%d outside [1, %d]", rerank, kMaxRerank);
    if (topk < 1 || topk > rerank)
        return fail(DH_ERR_SELECT, "topk=%d outside [1, rerank=%d]", topk, rerank);
    cudaError_t err = launch_merge_topk(exact_parts, sel_idx, P, M, rerank, topk, idx, logit,
                                        static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return fail(DH_ERR_CUDA, "merge launch: %s", cudaGetErrorString(err));
    return ok();
}

} // extern "C"
