/*
 * dh_oracle.c -- plain, slow CPU oracle for the 2-bit draft head with exact rerank
 * (and the page's 4-bit and fp8-weight variants).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or call this
 * file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Source of every step: the page "radiance_drafthead.py" (module docstring bullets and the
 * functions _quantize_head_now, _draft_head_int2, _emit, _apply_head_int2, _rerank_exact).
 * Precision: the quantiser runs in IEEE fp32 exactly as the page's torch code does
 * (correctly rounded division, no fused multiply-add, round half to even); everything the
 * page leaves to "the math" (coarse value, exact logit, exact head) runs in fp64.
 * Selection decisions are taken on fp32-rounded values, the precision the page's kernel
 * holds its accumulator in.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no -ffast-math, ever).
 *
 * Parity status per function (pins live in tests/test_oracle_pins.py):
 *   orc_quantize       pinned: hand-worked golden groups, invariants, error bound
 *   orc_pack/unpack    pinned: golden bytes, round trip, plane placement
 *   orc_coarse         pinned: collapsed form == direct dequant-and-dot (exact scales)
 *   orc_block_topk     pinned: brute force full sort on tiny inputs, KC=64 special case
 *   orc_select_topr    pinned: brute force, R = all candidates special case
 *   orc_rerank         pinned: exact integer arithmetic on scaled bf16 values
 *   orc_decode_e4m3    pinned: every finite code against torch's float8_e4m3fn conversion
 *   orc_quantize_fp8   pinned: power-of-two row scales reduce it to orc_quantize
 *   orc_rerank_fp8     pinned: power-of-two row scales reduce it to orc_rerank
 *   orc_exact_head     pinned: exact integer arithmetic; KC=64,R=V reduces forward to it
 *   orc_quantize4      pinned: hand-worked golden group, on-grid rows recovered exactly,
 *                      half-split byte placement, error bound
 *   orc_coarse4        pinned: collapsed form == direct dequant-and-dot (exact scales)
 *   orc_quantize_c4    pinned: hand-worked golden bytes; codes, S, ZS equal orc_quantize's
 *   orc_coarse_c4      pinned: equals orc_coarse of the quarter-split packing of the same head
 *   orc_quantize_g64   pinned: hand-worked golden groups at 64; each 64-group equals the
 *                      128-group quantiser on that group's values doubled in place
 *   orc_coarse_g64     pinned: collapsed form == direct dequant-and-dot over 64-groups
 *   orc_coarse_wside   pinned: equals orc_coarse where every dequantised weight is a bf16
 *                      value (power-of-two scales); a dequant-and-dot with torch's bf16 rounding
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

/* ------------------------------------------------------------------------------------- */
/* bf16 <-> fp32, written out from the IEEE definitions                                  */
/* ------------------------------------------------------------------------------------- */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round an fp32 value to bf16, nearest with ties to even (what torch's .to(bfloat16) does). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) /* NaN: keep it a NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* Round half to even on an fp32 value (torch.round semantics), written out explicitly. */
static float round_half_even(float x)
{
    float fl = floorf(x);
    float diff = x - fl; /* exact: x and floor(x) share the exponent range */
    if (diff > 0.5f) return fl + 1.0f;
    if (diff < 0.5f) return fl;
    /* exactly halfway: pick the even neighbour */
    double half = (double)fl * 0.5;
    return (floor(half) == half) ? fl : fl + 1.0f;
}

static float clampf(float v, float lo, float hi)
{
    if (v < lo) return lo;
    if (v > hi) return hi;
    return v;
}

/* ------------------------------------------------------------------------------------- */
/* Quantiser and packing: radiance_drafthead.py, _quantize_head_now                       */
/* ------------------------------------------------------------------------------------- */

#define GROUP 128
/* Per bit width (the page's BITS = 2 default and its BITS = 4 variant): the largest code
 * (1 << BITS) - 1, and the premultiplier 2^BITS of the bit-pattern dequant, whose bf16 bias is
 * 1 + v / 2^BITS (the code sits in mantissa slot 7 - BITS). */
static float levels_of(int bits) { return bits == 4 ? 15.0f : 3.0f; }
static float bias_of(int bits) { return bits == 4 ? 16.0f : 4.0f; }

/*
 * Per (row n, group gi of 128 consecutive k), in fp32:
 *   lo, hi = min, max of the group;   sc = max((hi - lo) / 3, 1e-8)
 *   zp = clamp(round(-lo / sc), 0, 3);   q_k = clamp(round(w_k / sc + zp), 0, 3)
 *   S = bf16(4 sc);   ZS = bf16(4 sc + zp sc)          (the premultiplied pair)
 * Packing (quarter split): byte j of a row holds q[j] | q[Q+j]<<2 | q[2Q+j]<<4 | q[3Q+j]<<6,
 * Q = H/4.  Optional outputs sc_out / zp_out expose the fp32 scale and zero point.
 * Returns 0, or -2 when H is not a multiple of 512 (whole groups in every quarter).
 */
/* e4m3 (fp8, "fn" variant) from its definition: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent 0 is subnormal, m/8 * 2^-6.  The codes with every exponent and
 * mantissa bit set (NaN in the format) are not given a special value: the page's decoder
 * does not test for them either, and the synthetic fp8 weights never contain them. */
static float e4m3_to_f32(uint8_t b)
{
    const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (float)(sgn ? -mag : mag);
}

void orc_decode_e4m3(const uint8_t *b, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_f32(b[i]);
}

/* One row of fp32 weights -> its packed bytes, S and ZS (the page's per-group steps).
 * bits = 2: quarter split, byte j = q[j] | q[H/4+j] << 2 | q[H/2+j] << 4 | q[3H/4+j] << 6;
 * bits = 4: half split, byte j = q[j] | q[H/2+j] << 4. */
static void quantize_row(const float *row, int64_t H, int bits, uint8_t *q, uint8_t *packed_row,
                         uint16_t *S_row, uint16_t *ZS_row, float *sc_row, float *zp_row,
                         int contiguous, int G)
{
    const int64_t NGt = H / G, Q = H / 4;
    const float LEVELS = levels_of(bits), BIAS = bias_of(bits);
    for (int64_t gi = 0; gi < NGt; ++gi) {
        float lo = row[gi * G], hi = lo;
        for (int t = 1; t < G; ++t) {
            float w = row[gi * G + t];
            if (w < lo) lo = w;
            if (w > hi) hi = w;
        }
        float sc = (hi - lo) / LEVELS;
        if (sc < 1e-8f) sc = 1e-8f;
        float zp = clampf(round_half_even((-lo) / sc), 0.0f, LEVELS);
        for (int t = 0; t < G; ++t) {
            float w = row[gi * G + t];
            float r = round_half_even(w / sc + zp);
            q[gi * G + t] = (uint8_t)clampf(r, 0.0f, LEVELS);
        }
        float s4 = BIAS * sc;
        float zsc = zp * sc;
        S_row[gi] = f32_to_bf16_rne(s4);
        ZS_row[gi] = f32_to_bf16_rne(s4 + zsc);
        if (sc_row) sc_row[gi] = sc;
        if (zp_row) zp_row[gi] = zp;
    }
    if (bits == 4) {
        for (int64_t j = 0; j < H / 2; ++j) packed_row[j] = (uint8_t)(q[j] | (q[H / 2 + j] << 4));
        return;
    }
    if (contiguous) { /* the page's rejected layout: byte j holds k = 4j .. 4j+3 */
        for (int64_t j = 0; j < Q; ++j)
            packed_row[j] = (uint8_t)(q[4 * j] | (q[4 * j + 1] << 2) | (q[4 * j + 2] << 4) |
                                      (q[4 * j + 3] << 6));
        return;
    }
    for (int64_t j = 0; j < Q; ++j)
        packed_row[j] = (uint8_t)(q[j] | (q[Q + j] << 2) | (q[2 * Q + j] << 4) | (q[3 * Q + j] << 6));
}

int orc_quantize(const uint16_t *W, int64_t V, int64_t H, uint8_t *packed, uint16_t *S,
                 uint16_t *ZS, float *sc_out, float *zp_out)
{
    if (H <= 0 || H % 512 != 0 || V <= 0) return -2;
    const int64_t NGt = H / GROUP, Q = H / 4;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *row = (float *)malloc((size_t)H * sizeof(float));
    if (!q || !row) {
        free(q);
        free(row);
        return -1;
    }
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) row[k] = bf16_to_f32(W[n * H + k]);
        quantize_row(row, H, 2, q, packed + n * Q, S + n * NGt, ZS + n * NGt,
                     sc_out ? sc_out + n * NGt : NULL, zp_out ? zp_out + n * NGt : NULL, 0, GROUP);
    }
    free(q);
    free(row);
    return 0;
}

/* The 2-bit head in the contiguous-4 layout the page measured against the quarter split
 * (byte j = q[4j] | q[4j+1] << 2 | q[4j+2] << 4 | q[4j+3] << 6); codes, S and ZS are those of
 * orc_quantize. */
int orc_quantize_c4(const uint16_t *W, int64_t V, int64_t H, uint8_t *packed, uint16_t *S,
                    uint16_t *ZS)
{
    if (H <= 0 || H % 512 != 0 || V <= 0) return -2;
    const int64_t NGt = H / GROUP, Q = H / 4;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *row = (float *)malloc((size_t)H * sizeof(float));
    if (!q || !row) {
        free(q);
        free(row);
        return -1;
    }
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) row[k] = bf16_to_f32(W[n * H + k]);
        quantize_row(row, H, 2, q, packed + n * Q, S + n * NGt, ZS + n * NGt, NULL, NULL, 1, GROUP);
    }
    free(q);
    free(row);
    return 0;
}

/* The group-size ablation the page measured (module docstring, 'Group 128, not 64'): the
 * 2-bit head with groups of 64 consecutive k, S and ZS [V, H/64]; quarter-split packing. */
int orc_quantize_g64(const uint16_t *W, int64_t V, int64_t H, uint8_t *packed, uint16_t *S,
                     uint16_t *ZS)
{
    if (H <= 0 || H % 512 != 0 || V <= 0) return -2;
    const int64_t NG64 = H / 64, Q = H / 4;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *row = (float *)malloc((size_t)H * sizeof(float));
    if (!q || !row) {
        free(q);
        free(row);
        return -1;
    }
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) row[k] = bf16_to_f32(W[n * H + k]);
        quantize_row(row, H, 2, q, packed + n * Q, S + n * NG64, ZS + n * NG64, NULL, NULL, 0,
                     64);
    }
    free(q);
    free(row);
    return 0;
}

/* The BITS = 4 variant of _quantize_head_now: levels 0..15, S = bf16(16 sc),
 * ZS = bf16(16 sc + zp sc), half-split packing into [V, H/2] bytes.  H % 256 == 0. */
int orc_quantize4(const uint16_t *W, int64_t V, int64_t H, uint8_t *packed, uint16_t *S,
                  uint16_t *ZS, float *sc_out, float *zp_out)
{
    if (H <= 0 || H % 256 != 0 || V <= 0) return -2;
    const int64_t NGt = H / GROUP;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *row = (float *)malloc((size_t)H * sizeof(float));
    if (!q || !row) {
        free(q);
        free(row);
        return -1;
    }
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) row[k] = bf16_to_f32(W[n * H + k]);
        quantize_row(row, H, 4, q, packed + n * (H / 2), S + n * NGt, ZS + n * NGt,
                     sc_out ? sc_out + n * NGt : NULL, zp_out ? zp_out + n * NGt : NULL, 0, GROUP);
    }
    free(q);
    free(row);
    return 0;
}

/* An fp8 head: e4m3 rows and a per-row fp32 scale.  The page widens the rows to fp32 and
 * multiplies by the row's scale (one fp32 rounding) before the same per-group steps. */
int orc_quantize_fp8(const uint8_t *W8, const float *wsc, int64_t V, int64_t H, uint8_t *packed,
                     uint16_t *S, uint16_t *ZS)
{
    if (H <= 0 || H % 512 != 0 || V <= 0) return -2;
    const int64_t NGt = H / GROUP, Q = H / 4;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *row = (float *)malloc((size_t)H * sizeof(float));
    if (!q || !row) {
        free(q);
        free(row);
        return -1;
    }
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) row[k] = e4m3_to_f32(W8[n * H + k]) * wsc[n];
        quantize_row(row, H, 2, q, packed + n * Q, S + n * NGt, ZS + n * NGt, NULL, NULL, 0, GROUP);
    }
    free(q);
    free(row);
    return 0;
}

void orc_unpack(const uint8_t *packed, int64_t V, int64_t H, uint8_t *codes)
{
    const int64_t Q = H / 4;
    for (int64_t n = 0; n < V; ++n)
        for (int64_t k = 0; k < H; ++k) {
            int64_t plane = k / Q, j = k % Q;
            codes[n * H + k] = (uint8_t)((packed[n * Q + j] >> (2 * plane)) & 3u);
        }
}

/* ------------------------------------------------------------------------------------- */
/* Coarse value: radiance_drafthead.py, docstring "Bit-pattern dequant" bullet and        */
/* _draft_head_int2.  c[m,n] = sum_gi ( S[n,gi] * p - ZS[n,gi] * xs ),                    */
/*   p  = sum_{k in gi} x[m,k] * (1 + v[n,k]/4),   xs = sum_{k in gi} x[m,k]              */
/* with S, ZS the stored bf16 values; fp64 throughout.                                    */
/* ------------------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *x;
    const uint8_t *packed;
    const uint16_t *S, *ZS;
    int M, bits, contiguous, group;
    int64_t H, V, n0, n1;
    double *c;
} coarse_job;

static void *coarse_worker(void *arg)
{
    coarse_job *jb = (coarse_job *)arg;
    const int bits = jb->bits;
    const int G = jb->group;
    const int64_t H = jb->H, NGt = H / G;
    const int64_t Q = H / (8 / bits); /* packed bytes per row: codes of k share byte k mod Q */
    const double bias = bits == 4 ? 16.0 : 4.0;
    const unsigned mask = (1u << bits) - 1u;
    double *v = (double *)malloc((size_t)H * sizeof(double));
    for (int64_t n = jb->n0; n < jb->n1; ++n) {
        const uint8_t *prow = jb->packed + n * Q;
        if (jb->contiguous) /* v[n,k]: field k mod 4 of the packed byte k / 4 */
            for (int64_t k = 0; k < H; ++k) v[k] = (double)((prow[k / 4] >> (2 * (k % 4))) & 3u);
        else /* v[n,k]: field k / Q of the packed byte k mod Q */
            for (int64_t k = 0; k < H; ++k) v[k] = (double)((prow[k % Q] >> (bits * (k / Q))) & mask);
        for (int m = 0; m < jb->M; ++m) {
            const uint16_t *xr = jb->x + (int64_t)m * H;
            double c = 0.0;
            for (int64_t gi = 0; gi < NGt; ++gi) {
                double p = 0.0, xs = 0.0;
                for (int t = 0; t < G; ++t) {
                    double xk = (double)bf16_to_f32(xr[gi * G + t]);
                    p += xk * (1.0 + v[gi * G + t] / bias);
                    xs += xk;
                }
                c += (double)bf16_to_f32(jb->S[n * NGt + gi]) * p -
                     (double)bf16_to_f32(jb->ZS[n * NGt + gi]) * xs;
            }
            jb->c[(int64_t)m * jb->V + n] = c;
        }
    }
    free(v);
    return NULL;
}

/* c is [M, V] fp64.  nthreads <= 1 runs on the calling thread.  bits: 2 (packed [V, H/4],
 * bias 4) or 4 (packed [V, H/2], bias 16). */
static void coarse_bits(const uint16_t *x, const uint8_t *packed, const uint16_t *S,
                        const uint16_t *ZS, int M, int64_t H, int64_t V, double *c, int nthreads,
                        int bits, int contiguous, int group)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    coarse_job jobs[256];
    int64_t chunk = (V + nthreads - 1) / nthreads;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        int64_t n0 = (int64_t)i * chunk, n1 = n0 + chunk;
        if (n1 > V) n1 = V;
        if (n0 >= n1) break;
        jobs[i] = (coarse_job){x, packed, S, ZS, M, bits, contiguous, group, H, V, n0, n1, c};
        if (nthreads == 1) {
            coarse_worker(&jobs[i]);
        } else {
            pthread_create(&th[i], NULL, coarse_worker, &jobs[i]);
            ++started;
        }
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
}

void orc_coarse(const uint16_t *x, const uint8_t *packed, const uint16_t *S, const uint16_t *ZS,
                int M, int64_t H, int64_t V, double *c, int nthreads)
{
    coarse_bits(x, packed, S, ZS, M, H, V, c, nthreads, 2, 0, GROUP);
}

/* The 2-bit head with groups of 64 (S, ZS [V, H/64]): the same group term per 64-group. */
void orc_coarse_g64(const uint16_t *x, const uint8_t *packed, const uint16_t *S,
                    const uint16_t *ZS, int M, int64_t H, int64_t V, double *c, int nthreads)
{
    coarse_bits(x, packed, S, ZS, M, H, V, c, nthreads, 2, 0, 64);
}

/* The 2-bit head in the contiguous-4 layout (same group term). */
void orc_coarse_c4(const uint16_t *x, const uint8_t *packed, const uint16_t *S,
                   const uint16_t *ZS, int M, int64_t H, int64_t V, double *c, int nthreads)
{
    coarse_bits(x, packed, S, ZS, M, H, V, c, nthreads, 2, 1, GROUP);
}

/* The BITS = 4 head: group term S p - ZS xs with p = sum x (1 + v/16). */
void orc_coarse4(const uint16_t *x, const uint8_t *packed, const uint16_t *S, const uint16_t *ZS,
                 int M, int64_t H, int64_t V, double *c, int nthreads)
{
    coarse_bits(x, packed, S, ZS, M, H, V, c, nthreads, 4, 0, GROUP);
}

/* The weight-side variant the page measured against (module docstring, 'The scale is applied
 * to the accumulator, never to the weight tile'): every weight is dequantised on its own to
 * the bf16 value bf16(S (1 + v/4) - ZS) and dotted with x.  S (1 + v/4) - ZS is exact in fp64
 * (and in fp32) for stored bf16 S and ZS, so the only rounding is the bf16 one.
 * c[m, n] = sum_k x[m, k] * w'[n, k], fp64. */
void orc_coarse_wside(const uint16_t *x, const uint8_t *packed, const uint16_t *S,
                      const uint16_t *ZS, int M, int64_t H, int64_t V, double *c)
{
    const int64_t Q = H / 4, NGt = H / GROUP;
    double *w = (double *)malloc((size_t)H * sizeof(double));
    for (int64_t n = 0; n < V; ++n) {
        for (int64_t k = 0; k < H; ++k) {
            const double v = (double)((packed[n * Q + k % Q] >> (2 * (k / Q))) & 3u);
            const double s = (double)bf16_to_f32(S[n * NGt + k / GROUP]);
            const double z = (double)bf16_to_f32(ZS[n * NGt + k / GROUP]);
            w[k] = (double)bf16_to_f32(f32_to_bf16_rne((float)(s * (1.0 + v / 4.0) - z)));
        }
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < H; ++k) acc += (double)bf16_to_f32(x[(int64_t)m * H + k]) * w[k];
            c[(int64_t)m * V + n] = acc;
        }
    }
    free(w);
}

/* ------------------------------------------------------------------------------------- */
/* Selection.  Order everywhere: value descending, equal values -> lower vocab index      */
/* (the first maximum, as the page's argmax returns).                                     */
/* ------------------------------------------------------------------------------------- */

typedef struct {
    float val;
    int32_t idx;
} cand;

static int cand_cmp(const void *a, const void *b)
{
    const cand *x = (const cand *)a, *y = (const cand *)b;
    if (x->val > y->val) return -1;
    if (x->val < y->val) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/*
 * Block candidates: radiance_drafthead.py, _emit.  For each row m and each block b of 64
 * columns [64b, min(64b+64, V)), the KC best columns by fp32 coarse value.  A block with
 * fewer than KC valid columns emits only those.  Output slots are [M, nblk*KC] in block
 * order, best first inside a block; unused slots get idx -1 and val -inf.
 * Returns the number of valid candidates per row.
 */
int64_t orc_block_topk(const float *cf, int M, int64_t V, int kcand, float *cval, int32_t *cidx)
{
    const int64_t nblk = (V + 63) / 64;
    int64_t nvalid = 0;
    cand buf[64];
    for (int m = 0; m < M; ++m) {
        nvalid = 0;
        for (int64_t b = 0; b < nblk; ++b) {
            int64_t c0 = 64 * b, c1 = c0 + 64 < V ? c0 + 64 : V;
            int cnt = (int)(c1 - c0);
            for (int i = 0; i < cnt; ++i) {
                buf[i].val = cf[(int64_t)m * V + c0 + i];
                buf[i].idx = (int32_t)(c0 + i);
            }
            qsort(buf, (size_t)cnt, sizeof(cand), cand_cmp);
            for (int s = 0; s < kcand; ++s) {
                int64_t o = (int64_t)m * nblk * kcand + b * kcand + s;
                if (s < cnt) {
                    cval[o] = buf[s].val;
                    cidx[o] = buf[s].idx;
                    ++nvalid;
                } else {
                    cval[o] = -INFINITY;
                    cidx[o] = -1;
                }
            }
        }
    }
    return nvalid;
}

/*
 * Global top-R: radiance_drafthead.py, _apply_head_int2 (BI gathered at BM.topk(RERANK)).
 * Per row, the R best of the ncand slots (slots with idx < 0 are skipped).
 * Returns 0, or -3 when a row has fewer than R valid candidates.
 */
int orc_select_topr(const float *cval, const int32_t *cidx, int M, int64_t ncand, int R,
                    int32_t *sel_idx, float *sel_val)
{
    cand *buf = (cand *)malloc((size_t)ncand * sizeof(cand));
    if (!buf) return -1;
    for (int m = 0; m < M; ++m) {
        int64_t cnt = 0;
        for (int64_t i = 0; i < ncand; ++i) {
            int32_t id = cidx[(int64_t)m * ncand + i];
            if (id < 0) continue;
            buf[cnt].val = cval[(int64_t)m * ncand + i];
            buf[cnt].idx = id;
            ++cnt;
        }
        if (cnt < R) {
            free(buf);
            return -3;
        }
        qsort(buf, (size_t)cnt, sizeof(cand), cand_cmp);
        for (int j = 0; j < R; ++j) {
            sel_idx[(int64_t)m * R + j] = buf[j].idx;
            if (sel_val) sel_val[(int64_t)m * R + j] = buf[j].val;
        }
    }
    free(buf);
    return 0;
}

/*
 * Exact rerank: radiance_drafthead.py, _rerank_exact (bf16 branch).
 * e[m,j] = sum_k x[m,k] * W[idx[m,j], k], fp64.
 */
void orc_rerank(const uint16_t *x, const uint16_t *W, int M, int64_t H, const int32_t *idx, int R,
                double *e)
{
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < R; ++j) {
            const uint16_t *wr = W + (int64_t)idx[(int64_t)m * R + j] * H;
            const uint16_t *xr = x + (int64_t)m * H;
            double s = 0.0;
            for (int64_t k = 0; k < H; ++k)
                s += (double)bf16_to_f32(xr[k]) * (double)bf16_to_f32(wr[k]);
            e[(int64_t)m * R + j] = s;
        }
}

/* The page's fp8 rerank arm: weight k of row n is the fp32 product e4m3(b) * scale[n]; the
 * exact logit sums x_k times that weight, here in fp64. */
void orc_rerank_fp8(const uint16_t *x, const uint8_t *W8, const float *wsc, int M, int64_t H,
                    const int32_t *idx, int R, double *e)
{
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < R; ++j) {
            const int64_t n = idx[(int64_t)m * R + j];
            const uint8_t *wr = W8 + n * H;
            const uint16_t *xr = x + (int64_t)m * H;
            double s = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                const float w = e4m3_to_f32(wr[k]) * wsc[n];
                s += (double)bf16_to_f32(xr[k]) * (double)w;
            }
            e[(int64_t)m * R + j] = s;
        }
}

/*
 * Result: the top-k of the R reranked entries (only reranked entries are eligible, the
 * reading of the top-k caller in _apply_head_int2; argmax is k = 1).  Ranked on the
 * fp32-rounded exact value, ties -> lower vocab index.  out_val receives the fp64 value.
 */
void orc_topk(const double *e, const int32_t *idx, int M, int R, int topk, int32_t *out_idx,
              double *out_val)
{
    cand *buf = (cand *)malloc((size_t)R * sizeof(cand));
    for (int m = 0; m < M; ++m) {
        for (int j = 0; j < R; ++j) {
            buf[j].val = (float)e[(int64_t)m * R + j];
            buf[j].idx = idx[(int64_t)m * R + j];
        }
        qsort(buf, (size_t)R, sizeof(cand), cand_cmp);
        for (int t = 0; t < topk; ++t) {
            out_idx[(int64_t)m * topk + t] = buf[t].idx;
            /* recover the fp64 value of that index */
            for (int j = 0; j < R; ++j)
                if (idx[(int64_t)m * R + j] == buf[t].idx) {
                    out_val[(int64_t)m * topk + t] = e[(int64_t)m * R + j];
                    break;
                }
        }
    }
    free(buf);
}

/* ------------------------------------------------------------------------------------- */
/* Exact bf16 head, for recall: logits[m,n] = sum_k x[m,k] W[n,k], fp64.                  */
/* ------------------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *x, *W;
    int M;
    int64_t H, V, n0, n1;
    double *out;
} head_job;

static void *head_worker(void *arg)
{
    head_job *jb = (head_job *)arg;
    for (int64_t n = jb->n0; n < jb->n1; ++n) {
        const uint16_t *wr = jb->W + n * jb->H;
        for (int m = 0; m < jb->M; ++m) {
            const uint16_t *xr = jb->x + (int64_t)m * jb->H;
            double s = 0.0;
            for (int64_t k = 0; k < jb->H; ++k)
                s += (double)bf16_to_f32(xr[k]) * (double)bf16_to_f32(wr[k]);
            jb->out[(int64_t)m * jb->V + n] = s;
        }
    }
    return NULL;
}

void orc_exact_head(const uint16_t *x, const uint16_t *W, int M, int64_t H, int64_t V,
                    double *out, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    head_job jobs[256];
    int64_t chunk = (V + nthreads - 1) / nthreads;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        int64_t n0 = (int64_t)i * chunk, n1 = n0 + chunk;
        if (n1 > V) n1 = V;
        if (n0 >= n1) break;
        jobs[i] = (head_job){x, W, M, H, V, n0, n1, out};
        if (nthreads == 1) {
            head_worker(&jobs[i]);
        } else {
            pthread_create(&th[i], NULL, head_worker, &jobs[i]);
            ++started;
        }
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
}
