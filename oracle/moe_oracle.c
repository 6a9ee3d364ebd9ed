/*
 * moe_oracle.c -- plain CPU oracle of the fused block-scaled MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, call or
 * link this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (one forward of the layer, per token row t):
 *   ROCm/aiter PR #6881 "[FlyDSL] MegaMoEV2: fuse Dispatch, GEMM1, GEMM2 and
 *   Combine into one kernel" (Title / Technical Details): quantise the BF16
 *   row, dispatch it to its top-k experts, GEMM1 against W13 with the SwiGLU
 *   epilogue, GEMM2 against W2, weighted combine back to a BF16 row.
 *   ROCm/aiter PR #6154 "Add full-expert DeepSeek V4.1 Flash MegaMoE tuning for
 *   gfx950" (Summary): W13 -> clamp-10 SwiGLU -> FP8 intermediate quantisation
 *   -> MXFP4 W2 -> weighted combine.
 *
 * The formulation is the plainest one: a dense loop over the token's k slots,
 * every dot product accumulated in double (the aiter #6881 commit that adds the
 * mega_moe op: its reference accumulates the experts' sum in double precision)
 * and rounded to float.  No blocking, no fusion, no reordering.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   Q8  MXFP8 block quantisation (E4M3 codes, one E8M0 scale per 32): OCP MX
 *       rule, scale exponent X = floor(log2 amax) - 8, E8M0 code clamp(X+127,
 *       0, 254), zero block -> code 0; element = RNE_E4M3(x / 2^(code-127)),
 *       saturating to +-448.
 *   SwiGLU a = G[0:I) (gate), b = G[I:2I) (up); with clamp L > 0:
 *       a = min(a, L), b = clamp(b, -L, L); h = a * (1/(1+exp(-a))) * b in float.
 *   y   GEMM2 rows are rounded to BF16 per route before the combine (the main
 *       path's BF16 rows, aiter #6881 Technical Details); `y_mode` 1 keeps them
 *       float; `y_mode` 2 sends them as MXFP8 in the main path's 1x32 format
 *       (aiter #6881 Technical Details, small input: GEMM2 rows go to the
 *       combine as FP8 instead of BF16), quantised from the float value with
 *       rule Q8 along H and dequantised for the combine.
 *   out Sum over valid slots in ascending k in float, rounded to BF16 once
 *       (ROCm/ATOM PR #2725 "route before the rows move", last commit note:
 *       the routed terms are added in single precision and rounded one time).
 *   A slot is valid iff its row t < num_valid_rows and 0 <= id < E
 *       (ATOM #2725 "Per-pass real row counts"; the linked aiter fix commit:
 *       a negative id takes no slot).  Invalid rows give +0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

/* ------------------------------------------------------------------ formats */

/* E2M1: sign | 2-bit exponent (bias 1) | 1-bit mantissa; exponent 0 is subnormal (0.5*m). */
double orc_e2m1_value(int nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (fn): sign | 4-bit exponent (bias 7) | 3-bit mantissa; S.1111.111 is NaN, no infinities. */
double orc_e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E8M0: unsigned power of two 2^(c-127); 0xFF is NaN. */
double orc_e8m0_value(int code) {
    if (code == 255) return NAN;
    return ldexp(1.0, code - 127);
}

float orc_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> BF16, round to nearest even (inputs are finite). */
uint16_t orc_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* value -> E4M3 code: nearest finite code, ties to the even code, so values
 * beyond 448 saturate to 448.  The 127 non-negative finite codes 0x00..0x7E are
 * ascending in value; the search finds the largest one not above |v|. */
int orc_e4m3_encode(double v) {
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    int lo = 0, hi = 126;
    if (a >= orc_e4m3_value(126)) return sign | 126;
    while (lo < hi) {          /* invariant: value(lo) <= a, answer in [lo, hi] */
        int mid = (lo + hi + 1) / 2;
        if (orc_e4m3_value(mid) <= a) lo = mid; else hi = mid - 1;
    }
    {
        double dlo = a - orc_e4m3_value(lo), dhi = orc_e4m3_value(lo + 1) - a;
        int c = lo;
        if (dhi < dlo) c = lo + 1;
        else if (dhi == dlo) c = (lo & 1) ? lo + 1 : lo;
        return sign | c;
    }
}

/* Q8: one 32-element block -> 32 E4M3 codes + one E8M0 scale code. */
void orc_quant_mxfp8_block(const float* x, uint8_t* codes, uint8_t* scale_code) {
    float amax = 0.0f;
    int i, code;
    double scale;
    for (i = 0; i < 32; ++i) if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    if (amax == 0.0f) {
        code = 0;
    } else {
        int ex;
        frexp((double)amax, &ex);            /* amax = m * 2^ex, m in [0.5,1) */
        code = (ex - 1) - 8 + 127;           /* floor(log2 amax) - emax(E4M3) + bias */
        if (code < 0) code = 0;
        if (code > 254) code = 254;
    }
    scale = orc_e8m0_value(code);
    for (i = 0; i < 32; ++i) codes[i] = (uint8_t)orc_e4m3_encode((double)x[i] / scale);
    *scale_code = (uint8_t)code;
}

/* Q8 over rows of BF16: codes [rows, cols], scales [rows, cols/32]. */
int orc_quant_mxfp8_rows(const uint16_t* x, int64_t rows, int cols, uint8_t* codes, uint8_t* scales) {
    int64_t r;
    if (cols <= 0 || cols % 32) return ORC_EINVAL;
    for (r = 0; r < rows; ++r) {
        float blk[32];
        int j, i;
        for (j = 0; j < cols / 32; ++j) {
            for (i = 0; i < 32; ++i) blk[i] = orc_bf16_to_float(x[r * cols + j * 32 + i]);
            orc_quant_mxfp8_block(blk, codes + r * cols + j * 32, scales + r * (cols / 32) + j);
        }
    }
    return ORC_OK;
}

/* ----------------------------------------------------------------- dispatch */

static int clamp_nvr(const int32_t* nvr, int T) {
    int v = nvr ? *nvr : T;
    if (v < 0) v = 0;
    if (v > T) v = T;
    return v;
}

static int slot_valid(const int32_t* ids, int t, int k, int K, int E, int nvr) {
    int e = ids[(int64_t)t * K + k];
    return t < nvr && e >= 0 && e < E;
}

/* Compact dispatch (vLLM PR #61262 (a second, fixed-slot MegaMoEV2 runtime): the compact
 * scheme packs tokens before dispatch).  counts[e] = valid slots with id e;
 * offsets = exclusive scan (E+1 entries); perm lists the valid flat slot ids
 * t*K+k grouped by expert, ascending flat id inside an expert;
 * route_row[t*K+k] = offsets[e] + rank, -1 for an invalid slot. */
int orc_dispatch_compact(const int32_t* ids, int T, int K, int E, const int32_t* num_valid_rows,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* route_row) {
    int nvr = clamp_nvr(num_valid_rows, T), t, k, e;
    int32_t* fill;
    if (T < 0 || K <= 0 || E <= 0) return ORC_EINVAL;
    for (e = 0; e < E; ++e) counts[e] = 0;
    for (t = 0; t < T; ++t)
        for (k = 0; k < K; ++k)
            if (slot_valid(ids, t, k, K, E, nvr)) counts[ids[(int64_t)t * K + k]]++;
    offsets[0] = 0;
    for (e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!fill) return ORC_ENOMEM;
    for (t = 0; t < T; ++t)
        for (k = 0; k < K; ++k) {
            int64_t s = (int64_t)t * K + k;
            if (slot_valid(ids, t, k, K, E, nvr)) {
                int ee = ids[s];
                int p = offsets[ee] + fill[ee]++;
                perm[p] = (int32_t)s;
                route_row[s] = p;
            } else {
                route_row[s] = -1;
            }
        }
    free(fill);
    return ORC_OK;
}

/* Fixed-slot dispatch (vLLM PR #61262: a token goes directly to a slot reserved
 * per rank, without a separate prepare step; on one GPU the slot belongs to the
 * expert).
 * Slot of (t,k) = e*mtpr + t; occ holds one bit per (e,t) in words of 32 tokens
 * ([E][ceil(mtpr/32)]); counts[e] = occupied slots of expert e (a row that names
 * the same expert twice occupies one slot); route_slot = -1 for invalid slots. */
int orc_dispatch_fixed(const int32_t* ids, int T, int K, int E, const int32_t* num_valid_rows, int mtpr,
                       uint32_t* occ, int32_t* counts, int32_t* route_slot) {
    int nvr = clamp_nvr(num_valid_rows, T), t, k, e;
    int words = (mtpr + 31) / 32;
    if (T < 0 || K <= 0 || E <= 0 || T > mtpr) return ORC_EINVAL;
    memset(occ, 0, sizeof(uint32_t) * (size_t)E * words);
    for (t = 0; t < T; ++t)
        for (k = 0; k < K; ++k) {
            int64_t s = (int64_t)t * K + k;
            if (slot_valid(ids, t, k, K, E, nvr)) {
                e = ids[s];
                occ[(int64_t)e * words + t / 32] |= 1u << (t % 32);
                route_slot[s] = e * mtpr + t;
            } else {
                route_slot[s] = -1;
            }
        }
    for (e = 0; e < E; ++e) {
        int n = 0, w;
        for (w = 0; w < words; ++w) {
            uint32_t v = occ[(int64_t)e * words + w];
            while (v) { n += (int)(v & 1u); v >>= 1; }
        }
        counts[e] = n;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ experts */

typedef struct {
    int H, I, E;
    const uint8_t *w13, *w13s, *w2, *w2s;
} orc_weights;

/* Dequantised MXFP4 weight element: E2M1 code (element 2j in the low nibble of
 * byte j) times the E8M0 scale of its 32-block along K. */
static double dq4(const uint8_t* codes, const uint8_t* scales, int64_t row, int Kdim, int k) {
    uint8_t byte = codes[row * (Kdim / 2) + k / 2];
    int nib = (k & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_value(nib) * orc_e8m0_value(scales[row * (Kdim / 32) + k / 32]);
}

/* One route: xdq = dequantised MXFP8 row [H]; writes y [H] (float) and, when
 * asked, the intermediates g [2I] and the requantised h codes/scales [I], [I/32]. */
static void expert_route(const orc_weights* W, int e, const double* xdq, float swiglu_limit,
                         float* y, float* g_out, uint8_t* hq_out, uint8_t* hs_out,
                         float* g, float* h, uint8_t* hq, uint8_t* hs, double* hdq) {
    const int H = W->H, I = W->I;
    int n, i, m;
    /* GEMM1: g[n] = sum_h xdq[h] * W13[e][n][h], n in [0, 2I) */
    for (n = 0; n < 2 * I; ++n) {
        double acc = 0.0;
        int64_t row = (int64_t)e * 2 * I + n;
        int hh;
        for (hh = 0; hh < H; ++hh) acc += xdq[hh] * dq4(W->w13, W->w13s, row, H, hh);
        g[n] = (float)acc;
    }
    /* SwiGLU with the optional clamp */
    for (i = 0; i < I; ++i) {
        float a = g[i], b = g[I + i];
        if (swiglu_limit > 0.0f) {
            if (a > swiglu_limit) a = swiglu_limit;
            if (b > swiglu_limit) b = swiglu_limit;
            if (b < -swiglu_limit) b = -swiglu_limit;
        }
        h[i] = a * (1.0f / (1.0f + expf(-a))) * b;
    }
    /* FP8 1x32 re-quantisation of h along I, then dequantise for GEMM2 */
    for (i = 0; i < I / 32; ++i) orc_quant_mxfp8_block(h + 32 * i, hq + 32 * i, hs + i);
    for (i = 0; i < I; ++i) hdq[i] = orc_e4m3_value(hq[i]) * orc_e8m0_value(hs[i / 32]);
    /* GEMM2: y[m] = sum_i hdq[i] * W2[e][m][i], m in [0, H) */
    for (m = 0; m < H; ++m) {
        double acc = 0.0;
        int64_t row = (int64_t)e * H + m;
        for (i = 0; i < I; ++i) acc += hdq[i] * dq4(W->w2, W->w2s, row, I, i);
        y[m] = (float)acc;
    }
    if (g_out) memcpy(g_out, g, sizeof(float) * 2 * I);
    if (hq_out) memcpy(hq_out, hq, (size_t)I);
    if (hs_out) memcpy(hs_out, hs, (size_t)I / 32);
}

typedef struct {
    float *g, *h, *y, *acc;
    uint8_t *hq, *hs, *xq, *xs, *yq, *ys;
    double *xdq, *hdq;
} orc_scratch;

static int scratch_alloc(orc_scratch* s, int H, int I) {
    s->g = (float*)malloc(sizeof(float) * 2 * I);
    s->h = (float*)malloc(sizeof(float) * I);
    s->y = (float*)malloc(sizeof(float) * H);
    s->acc = (float*)malloc(sizeof(float) * H);
    s->hq = (uint8_t*)malloc((size_t)I);
    s->hs = (uint8_t*)malloc((size_t)I / 32);
    s->xq = (uint8_t*)malloc((size_t)H);
    s->xs = (uint8_t*)malloc((size_t)H / 32);
    s->yq = (uint8_t*)malloc((size_t)H);
    s->ys = (uint8_t*)malloc((size_t)H / 32);
    s->xdq = (double*)malloc(sizeof(double) * H);
    s->hdq = (double*)malloc(sizeof(double) * I);
    return (s->g && s->h && s->y && s->acc && s->hq && s->hs && s->xq && s->xs && s->yq && s->ys && s->xdq && s->hdq)
               ? ORC_OK : ORC_ENOMEM;
}

static void scratch_free(orc_scratch* s) {
    free(s->g); free(s->h); free(s->y); free(s->acc); free(s->hq); free(s->hs);
    free(s->xq); free(s->xs); free(s->yq); free(s->ys); free(s->xdq); free(s->hdq);
}

/* One output row. */
static void forward_row(const orc_weights* W, const uint16_t* x, const int32_t* ids, const float* wts,
                        int t, int K, int nvr, float swiglu_limit, int y_mode, uint16_t* out_row,
                        orc_scratch* s) {
    const int H = W->H;
    int k, j, hh, any = 0;
    for (hh = 0; hh < H; ++hh) s->acc[hh] = 0.0f;
    if (t < nvr) {
        /* Q8 of the input row, then its dequantised values */
        orc_quant_mxfp8_rows(x + (int64_t)t * H, 1, H, s->xq, s->xs);
        for (hh = 0; hh < H; ++hh) s->xdq[hh] = orc_e4m3_value(s->xq[hh]) * orc_e8m0_value(s->xs[hh / 32]);
        for (k = 0; k < K; ++k) {
            int e = ids[(int64_t)t * K + k];
            float wk = wts[(int64_t)t * K + k];
            if (e < 0 || e >= W->E) continue;
            any = 1;
            expert_route(W, e, s->xdq, swiglu_limit, s->y, NULL, NULL, NULL, s->g, s->h, s->hq, s->hs, s->hdq);
            if (y_mode == 2)
                for (j = 0; j < H / 32; ++j) orc_quant_mxfp8_block(s->y + 32 * j, s->yq + 32 * j, s->ys + j);
            for (j = 0; j < H; ++j) {
                float yv = y_mode == 1   ? s->y[j]
                           : y_mode == 2 ? (float)(orc_e4m3_value(s->yq[j]) * orc_e8m0_value(s->ys[j / 32]))
                                         : orc_bf16_to_float(orc_float_to_bf16(s->y[j]));
                float prod = wk * yv;
                s->acc[j] = s->acc[j] + prod;
            }
        }
    }
    for (j = 0; j < H; ++j) out_row[j] = any ? orc_float_to_bf16(s->acc[j]) : (uint16_t)0;
}

/* Full forward, or a subset of rows.
 *   x [T,H] bf16; ids [T,K] int32; wts [T,K] float; num_valid_rows: NULL = T.
 *   y_mode: 0 BF16 GEMM2 rows, 1 float, 2 MXFP8 (see the file comment).
 *   rows/nrows: the token rows to compute (NULL = all T, in order); out is
 *   [nrows, H] bf16 in the order of `rows`.
 *   nthreads <= 0: the OpenMP default. */
int orc_moe_forward(const uint16_t* x, const int32_t* ids, const float* wts, int T, int H, int I, int E, int K,
                    const int32_t* num_valid_rows, const uint8_t* w13, const uint8_t* w13s,
                    const uint8_t* w2, const uint8_t* w2s, float swiglu_limit, int y_mode,
                    const int32_t* rows, int nrows, uint16_t* out, int nthreads) {
    orc_weights W;
    int nvr = clamp_nvr(num_valid_rows, T), n = rows ? nrows : T, r, err = ORC_OK;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || K <= 0 || H % 32 || I % 32) return ORC_EINVAL;
    W.H = H; W.I = I; W.E = E; W.w13 = w13; W.w13s = w13s; W.w2 = w2; W.w2s = w2s;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        orc_scratch s;
        int ok = scratch_alloc(&s, H, I) == ORC_OK;
        if (!ok) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORC_ENOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (r = 0; r < n; ++r) {
            int t = rows ? rows[r] : r;
            if (!ok) continue;
            if (t < 0 || t >= T) { memset(out + (int64_t)r * H, 0, sizeof(uint16_t) * H); continue; }
            forward_row(&W, x, ids, wts, t, K, nvr, swiglu_limit, y_mode, out + (int64_t)r * H, &s);
        }
        scratch_free(&s);
    }
    return err;
}

/* Intermediates of one (token, expert) route, for diagnosis: g [2I] float,
 * h codes [I], h scales [I/32], y [H] float (before the BF16 rounding). */
int orc_route_intermediates(const uint16_t* x_row, int H, int I, int E, int e,
                            const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s,
                            float swiglu_limit, float* g_out, uint8_t* hq_out, uint8_t* hs_out, float* y_out) {
    orc_weights W;
    orc_scratch s;
    int hh;
    if (e < 0 || e >= E || H % 32 || I % 32) return ORC_EINVAL;
    W.H = H; W.I = I; W.E = E; W.w13 = w13; W.w13s = w13s; W.w2 = w2; W.w2s = w2s;
    if (scratch_alloc(&s, H, I) != ORC_OK) { scratch_free(&s); return ORC_ENOMEM; }
    orc_quant_mxfp8_rows(x_row, 1, H, s.xq, s.xs);
    for (hh = 0; hh < H; ++hh) s.xdq[hh] = orc_e4m3_value(s.xq[hh]) * orc_e8m0_value(s.xs[hh / 32]);
    expert_route(&W, e, s.xdq, swiglu_limit, y_out, g_out, hq_out, hs_out, s.g, s.h, s.hq, s.hs, s.hdq);
    scratch_free(&s);
    return ORC_OK;
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Router top-k with softmax weights, the step in front of dispatch (ROCm/ATOM
 * PR #2725, linked commits on the Triton softmax top-k routing: an optional
 * valid-row count on the device gives every row from that count on ids -1 and
 * weight 0; an expert once picked is cleared to -inf and picks use a strict
 * greater-than scan, so ties go to the lowest id and a row with no finite
 * logit left picks expert 0 again with weight 0; weights are renormalised over the
 * picked experts unless `renormalize` is 0).
 *
 * Per row t < nvr, with m = max_e logit[t,e]:
 *   p_e = exp(l_e - m) / sum_e' exp(l_e' - m)             (double)
 *   pick k = 0..K-1: the first e with the largest remaining logit; its logit
 *   becomes -inf; weight_k = exp(l_pick - m) of the value before clearing
 *   (0 if it was already -inf), divided by sum_e' exp(l_e' - m), or by the sum
 *   of the K picked numerators when renormalising.
 * A row whose logits are all -inf has m = -inf and NaN weights (the formula as
 * written; out of the layer's contract).  Logits are float32 here; BF16 logits
 * are widened exactly by the caller. */
int orc_topk_softmax(const float* logits, int T, int E, int K, const int32_t* num_valid_rows, int renormalize,
                     int32_t* ids, float* weights) {
    int t, e, k;
    int nvr;
    double* v;
    double* num;
    if (T < 0 || E < 1 || K < 1 || K > E) return ORC_EINVAL;
    nvr = clamp_nvr(num_valid_rows, T);
    v = (double*)malloc(sizeof(double) * (size_t)E);
    num = (double*)malloc(sizeof(double) * (size_t)K);
    if (!v || !num) {
        free(v);
        free(num);
        return ORC_ENOMEM;
    }
    for (t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        double m = -INFINITY, all = 0.0, picked = 0.0;
        if (t >= nvr) {
            for (k = 0; k < K; ++k) {
                ids[(int64_t)t * K + k] = -1;
                weights[(int64_t)t * K + k] = 0.0f;
            }
            continue;
        }
        for (e = 0; e < E; ++e) {
            v[e] = (double)l[e];
            if (v[e] > m) m = v[e];
        }
        for (e = 0; e < E; ++e) all += exp((double)l[e] - m);
        for (k = 0; k < K; ++k) {
            int best = 0;
            for (e = 1; e < E; ++e)
                if (v[e] > v[best]) best = e;
            num[k] = v[best] == -INFINITY ? 0.0 : exp(v[best] - m);
            picked += num[k];
            ids[(int64_t)t * K + k] = best;
            v[best] = -INFINITY;
        }
        for (k = 0; k < K; ++k)
            weights[(int64_t)t * K + k] = (float)(num[k] / (renormalize ? picked : all));
    }
    free(v);
    free(num);
    return ORC_OK;
}
