/*
 * dh.h -- C ABI of the GB300 2-bit draft head with exact rerank.
 *
 * The operation (page "radiance_drafthead.py"): a speculative-decoding draft LM head that
 * replaces the stock bf16 head x[M,H] @ W[H,V].  W is quantised once to 2 bits per weight
 * with an asymmetric scale and zero per (vocabulary row, group of 128 hidden positions)
 * (_quantize_head_now); a coarse pass streams the 2-bit weight, applies the scale and zero
 * to the fp32 accumulator in the collapsed form (4s)*p - (4s + zp*s)*sum_k x_k, with
 * p = sum_k x_k (1 + v_k/4) read through the bf16 bit pattern 0x3F80 | (v << 5)
 * (module docstring, bullets "Bit-pattern dequant, hoisted" and "The scale is applied to the
 * accumulator"; _draft_head_int2); every block of 64 vocabulary columns emits its KCAND best
 * candidates (_emit); the RERANK best candidates of each row are rescored exactly against
 * the bf16 weight (_rerank_exact) and the best TOPK of those are returned (TOPK = 1 is the
 * argmax caller, TOPK = 16 the selector_top_k caller of _apply_head_int2).
 *
 * Conventions for every entry point
 *   - bf16 tensors are passed as uint16_t* holding the raw bit patterns.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, contiguous row-major,
 *     16-byte aligned.  The library never allocates, frees or synchronises: all work is
 *     enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and the call
 *     returns as soon as it is enqueued.  Outputs are valid once the stream reaches them.
 *   - Every entry point checks its arguments on the host before launching anything and
 *     returns a status (DH_OK or a negative DH_ERR_*); dh_last_error() then describes it.
 *     No entry point aborts, traps or prints.
 *   - Entry points are thread-safe as long as concurrent calls use distinct workspaces.
 *   - Device-side waits are bounded: a wait that times out records DH_ERR_DEVICE_TIMEOUT in
 *     a device flag (read with dh_device_status) and the kernel returns early.
 *
 * Shapes
 *   M  rows of hidden states per call (draft positions), 1 <= M <= 128
 *   H  hidden size, a positive multiple of 512 (every quarter of a row holds whole groups)
 *   V  vocabulary rows of the head, V >= 1
 *   G  = 128 (quantisation group), BLOCK_N = 64 (selection block), nblk = ceil(V / 64)
 */
#ifndef DH_H
#define DH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DH_OK 0
#define DH_ERR_NULL (-1)           /* a required pointer is NULL */
#define DH_ERR_SHAPE (-2)          /* M, H or V out of range (see Shapes) */
#define DH_ERR_SELECT (-3)         /* kcand, rerank or topk out of range */
#define DH_ERR_WORKSPACE (-4)      /* workspace smaller than dh_workspace_bytes() */
#define DH_ERR_ALIGN (-5)          /* a pointer is not 16-byte aligned */
#define DH_ERR_CUDA (-6)           /* a CUDA runtime call or launch failed */
#define DH_ERR_DEVICE_TIMEOUT (-7) /* a bounded device-side wait gave up (dh_device_status) */
#define DH_ERR_ARG (-8)            /* any other invalid argument */

/*
 * dh_quantize -- one-time quantise and pack of the bf16 head.
 * Page: radiance_drafthead.py, _quantize_head_now (BITS = 2, GROUP = 128).
 *
 *   W_bf16  [V, H]       bf16 head weight, row n = vocabulary entry n          (input)
 *   packed  [V, H/4]     u8: byte j of row n holds the 2-bit codes of k = j, H/4+j, H/2+j,
 *                        3H/4+j in bits 0-1, 2-3, 4-5, 6-7 (quarter split)        (output)
 *   scales  [V, H/128]   bf16 S  = bf16(4 * sc) per (row, group)                 (output)
 *   zeros   [V, H/128]   bf16 ZS = bf16(4 * sc + zp * sc) per (row, group)       (output)
 * with, per group of 128 consecutive k and in IEEE fp32: lo/hi = min/max,
 * sc = max((hi - lo) / 3, 1e-8), zp = clamp(round(-lo / sc), 0, 3),
 * q = clamp(round(w / sc + zp), 0, 3), round = half to even.  Bit-exact with that definition.
 * Returns DH_OK, DH_ERR_NULL, DH_ERR_SHAPE, DH_ERR_ALIGN or DH_ERR_CUDA.
 */
int dh_quantize(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                uint16_t *zeros, void *stream);

/*
 * dh_workspace_bytes -- device scratch that dh_forward needs for these sizes (bytes), or 0
 * when the sizes are invalid.  The pages need no such call because their host framework
 * allocates per call; here the caller allocates once and reuses it.
 */
size_t dh_workspace_bytes(int M, int H, int V, int kcand, int rerank);

/*
 * dh_forward -- the draft-head forward.
 * Page: radiance_drafthead.py, _apply_head_int2 with _draft_head_int2, _emit and
 * _rerank_exact (bf16 branch).
 *
 *   x        [M, H]          bf16 hidden states                                  (input)
 *   packed, scales, zeros    the output of dh_quantize for W_bf16                (input)
 *   W_bf16   [V, H]          bf16 head weight the rerank scores against          (input)
 *   kcand    1..64           candidates each 64-column block emits
 *   rerank   1..min(valid candidates, 1024), and <= V
 *                            candidates per row rescored exactly; valid candidates =
 *                            sum over blocks of min(kcand, columns in the block)
 *   topk     1..rerank       results per row; 1 is the argmax caller
 *   idx      [M, topk] int32 vocabulary indices, best first                     (output)
 *   logit    [M, topk] fp32  their exact logits sum_k x[m,k] W[idx,k]            (output)
 *   workspace, ws_bytes      device scratch of at least dh_workspace_bytes(...)
 * Ranking: coarse values and exact values are compared in fp32; equal values go to the
 * lower vocabulary index.  Only reranked entries are eligible for the result.
 * Sizes: every M with H <= 15360 has a coarse path (the 8-bit tcgen05 path in launches of 32
 * rows up to H = 7168 and of 16 rows above; the warp path where its shared memory holds the
 * staged x); wider rows, or a forced path (dh_set_coarse_path) that does not take the sizes,
 * give DH_ERR_ARG.
 * Returns DH_OK or a negative DH_ERR_* (checked before any launch).
 */
int dh_forward(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
               const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V, int kcand,
               int rerank, int topk, int32_t *idx, float *logit, void *workspace,
               size_t ws_bytes, void *stream);

/*
 * dh_forward_host -- dh_forward with x, idx and logit in host memory: the call a host-side
 * caller makes once per step, with the step's transfers inside it.  The pages' counterpart is
 * the same forward fed from and read back to the host by the serving loop.
 *
 *   x_host     [M, H] bf16      pinned host memory, mapped into the device's address space
 *                               (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with
 *                               cudaHostRegisterMapped), 16-byte aligned               (input)
 *   idx_host   [M, topk] int32  pinned, mapped host memory, 16-byte aligned            (output)
 *   logit_host [M, topk] fp32   pinned, mapped host memory, 16-byte aligned            (output)
 *   everything else as dh_forward: the head and the workspace in device memory.
 * On the 8-bit tcgen05 path the staging kernel reads x across the host link and keeps a
 * device copy for the rerank (in the workspace); on the other coarse paths x is first copied
 * to the workspace on the stream.  The last kernel writes idx and logit into the host
 * buffers: they hold the result once the stream has been synchronised, and must not be read
 * or written before.  Results are bit-identical to dh_forward's for the same inputs.
 * Returns DH_ERR_ARG (before anything runs) if a host buffer is not pinned and mapped, and
 * otherwise what dh_forward returns.
 */
int dh_forward_host(const uint16_t *x_host, const uint8_t *packed, const uint16_t *scales,
                    const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                    int kcand, int rerank, int topk, int32_t *idx_host, float *logit_host,
                    void *workspace, size_t ws_bytes, void *stream);

/*
 * dh_forward_debug -- dh_forward that also writes the intermediates, for parity checks.
 * Any of the extra outputs may be NULL.
 *   coarse    [M, V] fp32                 coarse values c[m, n]
 *   cand_val  [M, nblk*kcand] fp32        block candidates, block-major, best first inside
 *   cand_idx  [M, nblk*kcand] int32       a block; missing slots (block shorter than kcand)
 *                                         hold -inf / -1
 *   sel_idx   [M, rerank] int32           the reranked vocabulary indices (any order)
 *   sel_exact [M, rerank] fp32            their exact logits, same order as sel_idx
 */
int dh_forward_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                     const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                     int kcand, int rerank, int topk, int32_t *idx, float *logit,
                     void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                     int32_t *cand_idx, int32_t *sel_idx, float *sel_exact, void *stream);

/*
 * dh_forward_timed -- dh_forward that records caller-created CUDA events (cudaEvent_t, cast
 * to void*) at the stage boundaries, for per-kernel timing inside a benchmark:
 *   events[0] before staging x, [1] before the coarse pass, [2] before candidate
 *   selection, [3] before the rerank (which also runs the top-k merge), [4] and [5] after it.
 * `events` must hold DH_NUM_STAGE_EVENTS valid events.
 */
#define DH_NUM_STAGE_EVENTS 6
int dh_forward_timed(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                     const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                     int kcand, int rerank, int topk, int32_t *idx, float *logit,
                     void *workspace, size_t ws_bytes, void *const *events, void *stream);

/*
 * dh_forward_noalloc -- dh_forward for callers that cannot allocate device memory.
 * The pages have no counterpart: their host framework allocates per call.
 *
 * Some callers have no way to hand this library a workspace: a serving engine that has
 * already reserved nearly all free device memory for its KV cache (an extra cudaMalloc would
 * fail or eat into that cache), runtimes with a fixed memory pool, and latency-critical
 * paths where cudaMalloc's implicit device synchronisation is not acceptable.  For them this
 * entry point takes no workspace at all: its scratch is one file-scope device array of
 * DH_NOALLOC_WORKSPACE_BYTES inside the library, which every GPU that loads the library holds
 * until the process exits.  The caller still passes (and owns) every input and output.
 *
 *   Arguments, layouts, results and status codes are those of dh_forward without
 *   workspace/ws_bytes.  Sizes whose workspace (dh_workspace_bytes) exceeds
 *   DH_NOALLOC_WORKSPACE_BYTES are rejected with DH_ERR_WORKSPACE before anything runs.
 *   No cudaMalloc, cudaFree or other allocating routine is ever called.
 *   The first call on a device resolves the array's device address for that device (with
 *   that device current); make that first call before any stream capture.
 *   Every call uses the same array, which keeps the previous call's contents (the forward
 *   clears what must start at zero itself): calls that can overlap on the GPU -- on different
 *   streams, or concurrently from several host threads -- race on it and must be serialised
 *   by the caller.
 */
#define DH_NOALLOC_WORKSPACE_BYTES (16u << 20)
int dh_forward_noalloc(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                       int kcand, int rerank, int topk, int32_t *idx, float *logit,
                       void *stream);

/*
 * Coarse-pass implementation choice (process-wide).
 *   DH_PATH_AUTO     DH_PATH_TC where its shared-memory layout fits (H up to 8192), else
 *                    DH_PATH_WARP (default)
 *   DH_PATH_WARP     warp-level mma.sync on bf16 operands (the page's 1 + v/4 bit pattern),
 *                    batch handled 16 rows at a time
 *   DH_PATH_TC       tcgen05 with 8-bit operands: each 2-bit code masked in place is an exact
 *                    e4m3 weight; each bf16 x row is scaled by a power of two and written as
 *                    two e4m3 terms (three when the row's two-term residual is not negligible),
 *                    each at its own power-of-two scale, stacked along N; batch in launches of
 *                    16 or 32 rows
 *   DH_PATH_TC_BF16  tcgen05 on bf16 operands (the page's 1 + v/4 bit pattern)
 *   DH_PATH_CORE     CUDA cores, M <= 4 and H a multiple of 512: fp32 FMAs on weights made from
 *                    the packed bits (1 + v 2^(2p-8) by a shift and an and-or, minus 1.0
 *                    exactly), x as fp32 in shared memory; the small-batch alternative to the
 *                    tensor paths, never chosen by DH_PATH_AUTO (slower at every M it takes)
 * The bf16 paths and DH_PATH_CORE compute the coarse values from the exact bf16 x, up to fp32
 * rounding order.
 * DH_PATH_TC computes them from its e4m3 representation of x: exact for every element within
 * ~13 binades of its row's maximum with two terms, and with a third term for rows whose
 * elements span more; the remaining difference is below the coarse tolerance the tests apply
 * (1e-3 (1 + |value|)) for rows with outliers up to 2^12 times the rest.  Every path evaluates
 * the group term S p - ZS xs in fp32, so rows with far larger outliers lose precision to
 * cancellation on every path.  dh_set_coarse_path returns the previous setting, or DH_ERR_ARG
 * for an unknown value.  dh_coarse_path_for(M) reports which path a forward with M rows would
 * take.
 */
#define DH_PATH_AUTO 0
#define DH_PATH_WARP 1
#define DH_PATH_TC 2
#define DH_PATH_TC_BF16 3
#define DH_PATH_CORE 4
int dh_set_coarse_path(int path);
int dh_coarse_path_for(int M);

/*
 * dh_forward_launch_count -- number of kernels one dh_forward with these sizes launches on the
 * current coarse-path setting (0 when the sizes are invalid).  For benchmarks that count
 * device launches.
 */
int dh_forward_launch_count(int M, int H, int V, int kcand, int rerank);

/*
 * dh_device_status -- DH_OK, or DH_ERR_DEVICE_TIMEOUT when a kernel since the last reset
 * gave up on a bounded wait.  Synchronises the current device to read the flag; reset != 0
 * clears it.  Returns DH_ERR_CUDA if the device cannot be read.
 */
int dh_device_status(int reset);

/* Human-readable description of the last error on this thread ("" if none). */
const char *dh_last_error(void);

/* ABI version: (major << 16) | minor.  1.0: the head and its sharded calls; 1.2: the fp8
 * head; 1.3: the 4-bit head and the design-choice ablations; 1.4: dh_forward_host.  Minor
 * versions only add calls. */
int dh_version(void);

/*
 * dh_rerank -- the exact step alone: exact[m, j] = sum_k x[m, k] W[idx[m, j], k] for arbitrary
 * index lists, the same dot product (and bits) as the rerank inside dh_forward.
 * Page: radiance_drafthead.py, _rerank_exact (bf16 branch).  With idx[m, :] = 0 .. V-1 it is
 * the stock bf16 head over the whole vocabulary (for recall measurements).
 *   x      [M, H]  bf16, 16-byte aligned                                      (input)
 *   W_bf16 [V, H]  bf16 head rows, 16-byte aligned                            (input)
 *   idx    [M, n]  int32 row ids; an id outside [0, V) gives -inf                (input)
 *   exact  [M, n]  fp32 exact logits                                         (output)
 * 1 <= M <= 128, H a positive multiple of 512, V >= 1, n >= 1, M n < 2^31.  Stream-ordered on
 * `stream`, no allocation, no synchronisation.  DH_ERR_NULL / DH_ERR_SHAPE / DH_ERR_ALIGN /
 * DH_ERR_CUDA as dh_forward.
 */
int dh_rerank(const uint16_t *x, const uint16_t *W_bf16, int M, int H, int V, const int32_t *idx,
              long long n, float *exact, void *stream);

/*
 * Vocabulary-parallel head: each rank holds rows [vocab_offset, vocab_offset + Vs) of the
 * head (its own packed/S/ZS and bf16 rows) and the result equals the unsharded dh_forward bit
 * for bit.  The pages deploy the head as per-rank vocabulary shards
 * (radiance_drafthead.py, _apply_head_int2 on a vocab-parallel lm_head); the exchange between
 * the steps below is the caller's (two all-gathers of M x RERANK entries per rank).
 *
 * 1. dh_shard_candidates: the shard's coarse pass, block top-KCAND and top-RERANK of its own
 *    candidates.  out_val [M, rerank] fp32 coarse values and out_idx [M, rerank] int32 GLOBAL
 *    vocabulary ids (local row + vocab_offset), in rank order (value descending, lower id
 *    first).
 *    vocab_offset must be a multiple of 64 (the selection blocks then coincide with the
 *    unsharded head's) and rerank must not exceed the shard's valid candidates.  Workspace:
 *    dh_workspace_bytes(M, H, Vs, kcand, rerank).  Status codes as dh_forward.
 *    Because every shard's top-RERANK contains every global top-RERANK candidate it owns, the
 *    global top-RERANK of all shards' lists is the unsharded selection.
 * 2. dh_shard_rerank: every rank passes the gathered lists all_val/all_idx [M, ncand_all]
 *    (ncand_all = P x rerank; any order, -1 ids ignored, ids distinct).  Writes the global
 *    top-RERANK ids to sel_idx [M, rerank] in rank order (identical on every rank: step 3
 *    merges position by position) and their exact logits
 *    x . W[id] to exact [M, rerank] for the ids this shard owns, -inf for the others.
 *    W_shard [Vs, H] bf16 holds the shard's rows.  Workspace:
 *    dh_shard_rerank_workspace_bytes(M, ncand_all, rerank) (0 = invalid sizes).
 * 3. dh_shard_topk: exact_parts [P, M, rerank] (every rank's `exact`, gathered) merged by
 *    max, then idx/logit [M, topk] exactly as dh_forward returns them.
 */
int dh_shard_candidates(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, int M, int H, int Vs, long long vocab_offset,
                        int kcand, int rerank, float *out_val, int32_t *out_idx,
                        void *workspace, size_t ws_bytes, void *stream);
size_t dh_shard_rerank_workspace_bytes(int M, long long ncand_all, int rerank);
int dh_shard_rerank(const uint16_t *x, const uint16_t *W_shard, int M, int H, int Vs,
                    long long vocab_offset, const float *all_val, const int32_t *all_idx,
                    long long ncand_all, int rerank, int32_t *sel_idx, float *exact,
                    void *workspace, size_t ws_bytes, void *stream);
int dh_shard_topk(const float *exact_parts, const int32_t *sel_idx, int P, int M, int rerank,
                  int topk, int32_t *idx, float *logit, void *stream);

/*
 * fp8 head: the bf16 head weight replaced by e4m3 rows with one fp32 scale per row.
 * Page: radiance_drafthead.py, _quantize_head_now (an fp8 lm_head's weight is pre-scaled by
 * its per-row scale before the group statistics) and _rerank_exact (FP8 branch: the selected
 * rows are dequantised to fp32 and dotted with x).
 *
 *   W_e4m3    [V, H]  u8: OCP e4m3 (float8_e4m3fn) codes, row n = vocabulary entry n; finite
 *                     codes only (0x7F / 0xFF, the NaN codes, are not a weight)     (input)
 *   row_scale [V]     fp32 scale of each row; weight w[n, k] = fp32(e4m3(W[n, k]) * row_scale[n]),
 *                     the product rounded once to nearest even                     (input)
 *
 * dh_quantize_fp8 -- dh_quantize of those fp32 weights: the same group steps, outputs and
 *   layout, bit-exact.  W_e4m3, packed, scales, zeros 16-byte aligned, row_scale 4-byte.
 * dh_forward_fp8w -- dh_forward whose rerank scores against the fp8 rows: logit =
 *   sum_k x[m, k] * w[idx, k] with w as above.  packed/scales/zeros are dh_quantize_fp8's
 *   output; the coarse pass, selection, workspace (dh_workspace_bytes), ranking rules and
 *   status codes are those of dh_forward.  The rerank reads H bytes per selected row instead
 *   of 2H.
 */
int dh_quantize_fp8(const uint8_t *W_e4m3, const float *row_scale, int V, int H, uint8_t *packed,
                    uint16_t *scales, uint16_t *zeros, void *stream);
int dh_forward_fp8w(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                    const uint16_t *zeros, const uint8_t *W_e4m3, const float *row_scale, int M,
                    int H, int V, int kcand, int rerank, int topk, int32_t *idx, float *logit,
                    void *workspace, size_t ws_bytes, void *stream);

/*
 * 4-bit head: the page's BITS = 4 variant (radiance_drafthead.py, _quantize_head_now with
 * BITS = 4; the coarse term with bias 16).  The page's note: at 4 bits KCAND = 1 already
 * recovers nearly every argmax, where 2 bits needs KCAND = 8.
 *
 * dh_quantize4 -- as dh_quantize with 15 levels and the half split:
 *   packed  [V, H/2]     u8: byte j of row n holds the 4-bit codes of k = j (bits 0-3) and
 *                        k = H/2 + j (bits 4-7)                                   (output)
 *   scales  [V, H/128]   bf16 S  = bf16(16 * sc)                                  (output)
 *   zeros   [V, H/128]   bf16 ZS = bf16(16 * sc + zp * sc)                        (output)
 *   with sc = max((hi - lo) / 15, 1e-8), zp = clamp(round(-lo / sc), 0, 15),
 *   q = clamp(round(w / sc + zp), 0, 15).  H % 512 == 0.  Bit-exact with that definition.
 * dh_forward4 / dh_forward4_debug / dh_forward4_timed -- dh_forward / _debug / _timed on that
 *   head: coarse value
 *   c = sum_g ( S_g sum_{k in g} x_k (1 + v_k/16) - ZS_g sum_{k in g} x_k ); selection,
 *   rerank (against W_bf16), workspace (dh_workspace_bytes) and ranking rules unchanged.
 *   Runs on the 8-bit tcgen05 coarse path only: DH_ERR_ARG when another path is forced by
 *   dh_set_coarse_path or the sizes do not fit it (two pipeline stages of 32 KB of packed
 *   bytes plus the staged x next to the fixed buffers, in launches of 16 rows: H <= 11264 at
 *   any M -- the check runs before any launch).
 */
int dh_quantize4(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                 uint16_t *zeros, void *stream);
int dh_forward4(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V, int kcand,
                int rerank, int topk, int32_t *idx, float *logit, void *workspace,
                size_t ws_bytes, void *stream);
int dh_forward4_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                      const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                      int kcand, int rerank, int topk, int32_t *idx, float *logit,
                      void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                      int32_t *cand_idx, int32_t *sel_idx, float *sel_exact, void *stream);
/* dh_forward4_timed -- dh_forward_timed on the 4-bit head (same events). */
int dh_forward4_timed(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                      const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                      int kcand, int rerank, int topk, int32_t *idx, float *logit,
                      void *workspace, size_t ws_bytes, void *const *events, void *stream);

/*
 * Contiguous-4 layout of the 2-bit head: the packing the page measured against the quarter
 * split (radiance_drafthead.py, module docstring, 'Quarter-split packing' bullet).  Kept as an
 * ablation: it gives the same coarse values and costs a byte transpose in the dequant.
 *
 * dh_quantize_c4 -- dh_quantize with packed [V, H/4] u8 holding k = 4j .. 4j+3 in byte j
 *   (code of k = 4j + f in bits 2f .. 2f+1); scales and zeros as dh_quantize.  Bit-exact.
 * dh_forward_c4_debug -- the forward on that packing (8-bit tcgen05 path only, H <= 15360;
 *   DH_ERR_ARG otherwise, before any launch), with dh_forward_debug's optional outputs and, when `events` is not NULL,
 *   dh_forward_timed's stage events.  Everything else as dh_forward.
 */
int dh_quantize_c4(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                   uint16_t *zeros, void *stream);
int dh_forward_c4_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                        int kcand, int rerank, int topk, int32_t *idx, float *logit,
                        void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                        int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                        void *const *events, void *stream);

/*
 * Groups of 64: the group size the page measured against 128 (radiance_drafthead.py, module
 * docstring, 'Group 128, not 64').  Kept as an ablation: twice the scale/zero pairs and twice
 * the per-group accumulator folds for the same packed bytes.
 *
 * dh_quantize_g64 -- dh_quantize with groups of 64 consecutive k: scales, zeros [V, H/64] bf16
 *   (S = bf16(4 sc), ZS = bf16(4 sc + zp sc) per 64-group); packed [V, H/4] quarter split.
 * dh_forward_g64_debug -- the forward on that head, M <= 16, H <= 7680, 8-bit tcgen05 path only
 *   (DH_ERR_ARG otherwise); optional debug outputs and stage events as dh_forward_c4_debug.
 */
int dh_quantize_g64(const uint16_t *W_bf16, int V, int H, uint8_t *packed, uint16_t *scales,
                    uint16_t *zeros, void *stream);
int dh_forward_g64_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                         const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                         int kcand, int rerank, int topk, int32_t *idx, float *logit,
                         void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                         int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                         void *const *events, void *stream);

/*
 * Weight-side dequant: the scale placement the page measured against (radiance_drafthead.py,
 * module docstring, 'The scale is applied to the accumulator, never to the weight tile').
 * Kept as an ablation.
 *
 * dh_forward_wside_debug -- the forward on dh_quantize's head with the coarse value
 *   c = sum_k x_k bf16(S_g (1 + v_k/4) - ZS_g): every weight dequantised with its group's
 *   scale and zero and rounded to bf16, one bf16 tcgen05 accumulation per tile (no per-group
 *   fold).  Runs on the bf16 tcgen05 path whatever dh_set_coarse_path selects; optional debug
 *   outputs and stage events as dh_forward_c4_debug.
 */
int dh_forward_wside_debug(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                           const uint16_t *zeros, const uint16_t *W_bf16, int M, int H, int V,
                           int kcand, int rerank, int topk, int32_t *idx, float *logit,
                           void *workspace, size_t ws_bytes, float *coarse, float *cand_val,
                           int32_t *cand_idx, int32_t *sel_idx, float *sel_exact,
                           void *const *events, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DH_H */
