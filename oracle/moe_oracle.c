/*
 * moe_oracle.c -- plain, slow CPU statement of the local Mixture-of-Experts
 * FFN forward (softmax top-k routing, compact dispatch, bias-free SwiGLU
 * experts, weighted combine, residual Add + RMSNorm).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the timed CPU
 * baseline of the benchmark load this file's library. It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (page title, section):
 *   [ruDNN-4]  ruDNN user guide, section 4 "Routing contract" (German and
 *              Chinese editions): FP32 softmax over all E experts before
 *              top-k; ties favour the lower expert id; optional
 *              renormalisation of the selected weights, then a cast to the
 *              logits dtype; rows holding NaN or +inf, or only -inf, keep NaN
 *              weights; indices are U32 of shape [T, top_k].
 *   [ruDNN-5]  ruDNN user guide, section 5 "Expert weights and dispatch":
 *              x [T,H], gate/up [E,I,H], down [E,H,I], one float dtype;
 *              dispatch drops nothing; order inside an expert is unspecified;
 *              a saved map restores token order.
 *   [ruDNN-3]  ruDNN user guide, section 3 "MoE workflow": logits ->
 *              softmax/top-k -> compact dispatch -> SwiGLU experts ->
 *              weighted combine; bias-free experts.
 *   [ruDNN-10] ruDNN user guide, section 10 "Group-limited sigmoid MoE
 *              routing" (Chinese edition): sigmoid scores; an optional FP32
 *              correction bias that only affects the selection; experts in
 *              equal consecutive groups; a group scored by its best (or two
 *              best) corrected scores; selected_groups groups kept, top_k
 *              experts picked inside them; weights are the raw scores,
 *              optionally renormalised, times a finite positive scale; equal
 *              scores favour the lower id; limits E 1..1024, groups 1..128,
 *              top_k 1..64.
 *   [ruDNN-7]  ruDNN user guide, section 7 "LayerNorm, RMSNorm and Softmax":
 *              last-axis RMSNorm, epsilon finite and > 0, FP32 statistics,
 *              output in the input dtype.
 *   [Ascend-CARN] aclnnMoeDistributeCombineAddRmsNormV2, "Function" formula:
 *              combineOut = sum_k(expertScales * expert output),
 *              x = combineOut + residualX,
 *              y = x / sqrt(mean(x^2) + normEps) * gamma; outputs yOut, xOut
 *              (residual dtype) and rstdOut (FP32, one per token).
 *   [Ascend-CARN-V2] the same operator's formula and parameter list:
 *              combineOut = Sum(expertScales * ataOut + expertScales *
 *              sharedExpertX); special experts by id range after the
 *              moeExpertNum routed experts: zero (output 0), copy (output
 *              oriX), const (alpha1 * oriX + alpha2 * V); xActiveMask 1-D
 *              [BS] (kept tokens first) or 2-D [BS, K].
 *   [aclnnFFN] aclnnFFN, "Formula": y = activation(x W1 + b1) W2 + b2; the
 *              experts here are its bias-free, SwiGLU-activated case.
 *   [ruDNN-12] ruDNN user guide, section 12 "MoE first-order training"
 *              (Chinese edition): FP32 weights of a fixed selection
 *              (softmax or sigmoid scoring, optional renormalisation of the
 *              selected weights, then a finite positive scale) and their
 *              logits gradient; repeated indices act as a gather; an illegal
 *              index makes the whole row NaN; no derivative through the
 *              selection. Backward order: combine backward (expert-output
 *              gradient and FP32 weight gradient), expert backward (input
 *              rows and FP32 gate/up/down gradients), dispatch backward (the
 *              selected rows summed back to their token without the routing
 *              weight), then the router backward.
 *
 * Precision. Routing follows [ruDNN-4] literally: the softmax is computed in
 * float (FP32) with libm expf. Everything the pages leave open (expert GEMMs,
 * combine, norm statistics) is computed in double and left unrounded unless
 * the pages name an output dtype.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - selection ranks experts by their FP32 logit, highest first, lower id on
 *     equal logits; softmax is strictly increasing in the logit, so this is
 *     the top-k of the exact softmax;
 *   - the k outputs of a row are written in selection order;
 *   - an invalid row (NaN, +inf, or all -inf) gets indices 0..k-1 (every key
 *     ties, so the lower ids win) and NaN weights; it is still dispatched;
 *   - weights are cast to the logits dtype with or without renormalisation;
 *   - order inside an expert segment is the assignment order t*k+j here;
 *     any order is valid, so tests compare per-expert sets;
 *   - an expert index >= E handed to dispatch gets no row (row_of = -1) and
 *     makes the token's combined output NaN;
 *   - RMSNorm statistics are taken on x after it is rounded to the output
 *     dtype, so the fused op equals RMSNorm applied to xOut.
 *
 * Element type codes: 0 = f32, 1 = bf16, 2 = f16 (both stored as raw 16-bit
 * words), 3 = f64 (oracle-internal arrays only).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_F64 = 3 };

/* ---- element conversions (IEEE 754 binary32 / bfloat16 / binary16) ----- */

/* bfloat16 is the top half of a binary32 word, so the upcast is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
static uint16_t float_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* binary16 conversions go through the compiler's IEEE _Float16 type. */
static float f16_bits_to_float(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, sizeof h);
    return (float)h;
}

static uint16_t float_to_f16_bits(float f)
{
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, sizeof b);
    return b;
}

static double load_elem(const void *p, int dt, int64_t i)
{
    switch (dt) {
    case OR_F32: return (double)((const float *)p)[i];
    case OR_BF16: return (double)bf16_bits_to_float(((const uint16_t *)p)[i]);
    case OR_F16: return (double)f16_bits_to_float(((const uint16_t *)p)[i]);
    default: return ((const double *)p)[i];
    }
}

/* Store v rounded once to dtype dt. For the 16-bit types the value is first
 * rounded to binary32; doubles that reach this point are already float-exact
 * (routing weights) or the double rounding is inside every stated tolerance. */
static void store_elem(void *p, int dt, int64_t i, double v)
{
    switch (dt) {
    case OR_F32: ((float *)p)[i] = (float)v; break;
    case OR_BF16: ((uint16_t *)p)[i] = float_to_bf16_bits((float)v); break;
    case OR_F16: ((uint16_t *)p)[i] = float_to_f16_bits((float)v); break;
    default: ((double *)p)[i] = v; break;
    }
}

/* Exposed so tests can pin the conversions against library routines. */
void oracle_convert(const void *src, int sdt, void *dst, int ddt, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        store_elem(dst, ddt, i, load_elem(src, sdt, i));
}

/* ---- routing [ruDNN-4] -------------------------------------------------- */

/*
 * For every token t: upcast the E logits to FP32; classify the row; FP32
 * softmax over all E (max-subtracted, summed in ascending expert order);
 * pick top_k experts one at a time, each pick the highest remaining FP32
 * logit with the lower id kept on equal logits; optionally divide the picked
 * probabilities by their FP32 sum (taken in slot order); cast to the logits
 * dtype. Returns the number of invalid rows, or -1 on bad arguments.
 */
int64_t oracle_route(const void *logits, int ldt, int64_t T, int64_t E,
                     int64_t top_k, int renormalize, uint32_t *idx, void *w)
{
    if (T < 0 || E < 1 || top_k < 1 || top_k > E)
        return -1;
    float *l = (float *)malloc((size_t)E * sizeof(float));
    float *p = (float *)malloc((size_t)E * sizeof(float));
    float *sel = (float *)malloc((size_t)top_k * sizeof(float));
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    int64_t invalid_rows = 0;

    for (int64_t t = 0; t < T; ++t) {
        int has_nan_or_pinf = 0, all_ninf = 1;
        for (int64_t e = 0; e < E; ++e) {
            l[e] = (float)load_elem(logits, ldt, t * E + e);
            if (isnan(l[e]) || (isinf(l[e]) && l[e] > 0.0f))
                has_nan_or_pinf = 1;
            if (!(isinf(l[e]) && l[e] < 0.0f))
                all_ninf = 0;
        }
        if (has_nan_or_pinf || all_ninf) {
            for (int64_t j = 0; j < top_k; ++j) {
                idx[t * top_k + j] = (uint32_t)j;
                store_elem(w, ldt, t * top_k + j, (double)NAN);
            }
            ++invalid_rows;
            continue;
        }

        float m = l[0];
        for (int64_t e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        float s = 0.0f;
        for (int64_t e = 0; e < E; ++e)
            s += expf(l[e] - m);
        for (int64_t e = 0; e < E; ++e)
            p[e] = expf(l[e] - m) / s;

        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            idx[t * top_k + j] = (uint32_t)best;
            sel[j] = p[best];
        }
        if (renormalize) {
            float z = 0.0f;
            for (int64_t j = 0; j < top_k; ++j) z += sel[j];
            for (int64_t j = 0; j < top_k; ++j) sel[j] = sel[j] / z;
        }
        for (int64_t j = 0; j < top_k; ++j)
            store_elem(w, ldt, t * top_k + j, (double)sel[j]);
    }
    free(l); free(p); free(sel); free(taken);
    return invalid_rows;
}

/* ---- grouped sigmoid routing [ruDNN-10] --------------------------------- */

/* Sigmoid of a binary32 value, correctly rounded to binary32: evaluated in
 * double (whose error is far below half a binary32 ulp) and rounded once. */
static float sigmoid_f32(float x)
{
    return (float)(1.0 / (1.0 + exp(-(double)x)));
}

/*
 * For every token t, in the order the section gives:
 *   s_e = sigmoid(l_e) as an FP32 score; c_e = s_e + bias_e (FP32; the bias
 *   only steers the selection);
 *   the E experts form `groups` groups of E/groups consecutive experts; a
 *   group's score is its largest c, or the FP32 sum of its two largest c when
 *   group_top_two is set;
 *   the `selected_groups` best groups are kept (higher score first, lower
 *   group id on equal scores);
 *   top_k experts of the kept groups are picked by c (higher first, lower id
 *   on equal scores);
 *   their weights are the raw scores s, divided by their FP32 sum (slot
 *   order) when renormalize is set, times `scale`, cast to the logits dtype.
 * A row whose corrected scores hold a NaN (a NaN logit or bias) gets indices
 * 0..k-1 and NaN weights, as in the softmax contract. bias may be NULL
 * (all zero). Returns the number of such rows, or -1 on arguments outside
 * the section's limits.
 */
int64_t oracle_route_sigmoid_grouped(const void *logits, int ldt, int64_t T, int64_t E,
                                     const float *bias, int64_t top_k, int64_t groups,
                                     int64_t selected_groups, int group_top_two,
                                     int renormalize, float scale, uint32_t *idx, void *w)
{
    if (T < 0 || E < 1 || E > 1024 || groups < 1 || groups > 128 || E % groups != 0 ||
        selected_groups < 1 || selected_groups > groups || top_k < 1 || top_k > 64 ||
        top_k > selected_groups * (E / groups) || (group_top_two && E / groups < 2) ||
        !isfinite(scale) || !(scale > 0.0f))
        return -1;
    const int64_t gs = E / groups;
    float *sc = (float *)malloc((size_t)E * sizeof(float));
    float *c = (float *)malloc((size_t)E * sizeof(float));
    float *gscore = (float *)malloc((size_t)groups * sizeof(float));
    unsigned char *gkept = (unsigned char *)malloc((size_t)groups);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    float *pick = (float *)malloc((size_t)top_k * sizeof(float));
    int64_t invalid_rows = 0;

    for (int64_t t = 0; t < T; ++t) {
        int has_nan = 0;
        for (int64_t e = 0; e < E; ++e) {
            sc[e] = sigmoid_f32((float)load_elem(logits, ldt, t * E + e));
            c[e] = sc[e] + (bias ? bias[e] : 0.0f);
            if (isnan(c[e])) has_nan = 1;
        }
        if (has_nan) {
            for (int64_t j = 0; j < top_k; ++j) {
                idx[t * top_k + j] = (uint32_t)j;
                store_elem(w, ldt, t * top_k + j, (double)NAN);
            }
            ++invalid_rows;
            continue;
        }

        for (int64_t g = 0; g < groups; ++g) {
            float first = -INFINITY, second = -INFINITY;
            for (int64_t e = g * gs; e < (g + 1) * gs; ++e) {
                if (c[e] > first) { second = first; first = c[e]; }
                else if (c[e] > second) second = c[e];
            }
            gscore[g] = group_top_two ? first + second : first;
        }
        memset(gkept, 0, (size_t)groups);
        for (int64_t n = 0; n < selected_groups; ++n) {
            int64_t best = -1;
            for (int64_t g = 0; g < groups; ++g) {
                if (gkept[g]) continue;
                if (best < 0 || gscore[g] > gscore[best]) best = g;
            }
            gkept[best] = 1;
        }

        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e] || !gkept[e / gs]) continue;
                if (best < 0 || c[e] > c[best]) best = e;
            }
            taken[best] = 1;
            idx[t * top_k + j] = (uint32_t)best;
            pick[j] = sc[best];
        }
        if (renormalize) {
            float zsum = 0.0f;
            for (int64_t j = 0; j < top_k; ++j) zsum += pick[j];
            for (int64_t j = 0; j < top_k; ++j) pick[j] = pick[j] / zsum;
        }
        for (int64_t j = 0; j < top_k; ++j)
            store_elem(w, ldt, t * top_k + j, (double)(pick[j] * scale));
    }
    free(sc); free(c); free(gscore); free(gkept); free(taken); free(pick);
    return invalid_rows;
}

/* ---- dispatch [ruDNN-5] ------------------------------------------------- */

/*
 * Count assignments per expert, take the exclusive prefix sum, and give each
 * assignment a = t*top_k + j the next free row of its expert's segment, in
 * ascending a. row_of[a] is that row; src_of[row] = a is its inverse. An
 * index >= E gets no row (row_of = -1). src_of entries past the last row are
 * set to -1. Returns the number of such bad indices, or -1 on bad arguments.
 */
int64_t oracle_dispatch(const uint32_t *idx, int64_t T, int64_t top_k, int64_t E,
                        int32_t *counts, int32_t *offsets, int32_t *row_of,
                        int32_t *src_of)
{
    if (T < 0 || E < 1 || top_k < 1)
        return -1;
    int64_t A = T * top_k, bad = 0;
    int64_t *next = (int64_t *)malloc((size_t)E * sizeof(int64_t));
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < A; ++a) {
        if ((int64_t)idx[a] >= E) ++bad;
        else ++counts[idx[a]];
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) {
        offsets[e + 1] = offsets[e] + counts[e];
        next[e] = offsets[e];
    }
    for (int64_t r = 0; r < A; ++r) src_of[r] = -1;
    for (int64_t a = 0; a < A; ++a) {
        int64_t e = (int64_t)idx[a];
        if (e >= E) { row_of[a] = -1; continue; }
        int64_t r = next[e]++;
        row_of[a] = (int32_t)r;
        src_of[r] = (int32_t)a;
    }
    free(next);
    return bad;
}

/* x_disp[r, :] = x[src_of[r] / top_k, :] for every row r < rows; rows with
 * src_of < 0 are left untouched. Same dtype on both sides (a copy). */
void oracle_gather(const void *x, int dt, int64_t H, int64_t top_k,
                   const int32_t *src_of, int64_t rows, void *x_disp)
{
    for (int64_t r = 0; r < rows; ++r) {
        if (src_of[r] < 0) continue;
        int64_t t = src_of[r] / top_k;
        for (int64_t h = 0; h < H; ++h)
            store_elem(x_disp, dt, r * H + h, load_elem(x, dt, t * H + h));
    }
}

/* ---- experts [ruDNN-3], [ruDNN-5], [aclnnFFN] --------------------------- */

/*
 * For each of nrows input rows x_r with expert e = expert_of_row[r]:
 *   g = Wg[e] x_r, u = Wu[e] x_r          (Wg, Wu are [E, I, H]; length I)
 *   h = SiLU(g) * u, SiLU(z) = z / (1 + exp(-z))
 *   out_r = Wd[e] h                       (Wd is [E, H, I]; length H)
 * in double, unrounded. x and the weights share dtype dt.
 * Returns 0, or -1 when an expert id is out of range.
 */
int oracle_swiglu_rows(const void *xrows, int dt, int64_t nrows,
                       const int32_t *expert_of_row, const void *gate,
                       const void *up, const void *down, int64_t E, int64_t H,
                       int64_t I, double *out)
{
    double *xr = (double *)malloc((size_t)H * sizeof(double));
    double *hv = (double *)malloc((size_t)I * sizeof(double));
    int rc = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t e = expert_of_row[r];
        if (e < 0 || e >= E) { rc = -1; break; }
        for (int64_t k = 0; k < H; ++k) xr[k] = load_elem(xrows, dt, r * H + k);
        for (int64_t i = 0; i < I; ++i) {
            double g = 0.0, u = 0.0;
            int64_t wrow = (e * I + i) * H;
            for (int64_t k = 0; k < H; ++k) {
                g += load_elem(gate, dt, wrow + k) * xr[k];
                u += load_elem(up, dt, wrow + k) * xr[k];
            }
            hv[i] = g / (1.0 + exp(-g)) * u;
        }
        for (int64_t o = 0; o < H; ++o) {
            double acc = 0.0;
            int64_t wrow = (e * H + o) * I;
            for (int64_t i = 0; i < I; ++i)
                acc += load_elem(down, dt, wrow + i) * hv[i];
            out[r * H + o] = acc;
        }
    }
    free(xr); free(hv);
    return rc;
}

/* The dispatched form: rows [offsets[e], offsets[e+1]) belong to expert e. */
int oracle_experts_dispatched(const void *x_disp, int dt, const int32_t *offsets,
                              int64_t E, const void *gate, const void *up,
                              const void *down, int64_t H, int64_t I, double *out)
{
    int64_t rows = offsets[E];
    int32_t *owner = (int32_t *)malloc((size_t)(rows > 0 ? rows : 1) * sizeof(int32_t));
    for (int64_t e = 0; e < E; ++e)
        for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) owner[r] = (int32_t)e;
    int rc = oracle_swiglu_rows(x_disp, dt, rows, owner, gate, up, down, E, H, I, out);
    free(owner);
    return rc;
}

/* ---- combine [ruDNN-3], [Ascend-CARN] ----------------------------------- */

/*
 * y[t, :] = sum over slots j < top_k, in slot order, of
 *           w[t, j] * out_disp[row_of[t*top_k + j], :]
 * in double, unrounded. A slot with row_of < 0 makes the whole row NaN.
 */
void oracle_combine(const void *out_disp, int odt, const void *w, int wdt,
                    const int32_t *row_of, int64_t T, int64_t top_k, int64_t H,
                    double *y)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t j = 0; j < top_k; ++j) {
                int64_t r = row_of[t * top_k + j];
                if (r < 0) { acc = NAN; break; }
                acc += load_elem(w, wdt, t * top_k + j) * load_elem(out_disp, odt, r * H + h);
            }
            y[t * H + h] = acc;
        }
    }
}

/* ---- combine with special experts, shared expert, active mask
 *      [Ascend-CARN-V2] -------------------------------------------------- */

/*
 * The combine of aclnnMoeDistributeCombineAddRmsNormV2 on one device. For
 * each token t and each slot j that the active mask keeps (mask_dims 0: all;
 * 1: mask[t] keeps or drops the token's every slot; 2: mask[t*k+j]), with
 * id = ids[t*k+j] and scale s = w[t*k+j]:
 *   id < E                        o = the dispatched row out_disp[row_of[.]]
 *   E <= id < E+zero              o = 0                      (zero expert)
 *   ... < E+zero+copy             o = ori_x[t]               (copy expert)
 *   ... < E+zero+copy+const_n     o = alpha1[c]*ori_x[t] + alpha2[c]*V[c],
 *                                 c = id - E - zero - copy   (const expert)
 * and combineOut[t] = sum_j (s*o + s*shared_x[t]), the formula's shared term
 * taken as printed (one per kept slot, scaled like it; no term without
 * shared_x). ids may be NULL when no special experts are configured (every
 * slot is then a dispatched expert). A slot with a dispatched id but no row
 * (row_of < 0), or an id past the last special expert, makes the token's
 * output NaN. ori_x, alpha1/2, V and shared_x are in dtype xdt. Sums in
 * double. Returns -1 on missing inputs for the configured special experts or
 * a bad mask_dims, -2 if a 1-D mask keeps a token after dropping one (the
 * operator requires the kept tokens first), else 0.
 */
int oracle_combine_v2(const void *out_disp, int odt, const void *w, int wdt,
                      const int32_t *row_of, const uint32_t *ids, int64_t E, int64_t zero_n,
                      int64_t copy_n, int64_t const_n, const void *ori_x,
                      const void *alpha1, const void *alpha2, const void *const_v,
                      const void *shared_x, const uint8_t *mask, int mask_dims, int xdt,
                      int64_t T, int64_t top_k, int64_t H, double *y)
{
    const int64_t special = zero_n + copy_n + const_n;
    if (zero_n < 0 || copy_n < 0 || const_n < 0 || mask_dims < 0 || mask_dims > 2 ||
        (mask_dims && !mask) || (special > 0 && !ids) ||
        ((copy_n > 0 || const_n > 0) && !ori_x) ||
        (const_n > 0 && (!alpha1 || !alpha2 || !const_v)))
        return -1;
    if (mask_dims == 1)
        for (int64_t t = 1; t < T; ++t)
            if (mask[t] && !mask[t - 1]) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t j = 0; j < top_k; ++j) {
                const int64_t a = t * top_k + j;
                if (mask_dims == 1 && !mask[t]) continue;
                if (mask_dims == 2 && !mask[a]) continue;
                const int64_t id = ids ? (int64_t)ids[a] : 0;
                const double sc = load_elem(w, wdt, a);
                double o;
                if (!ids || id < E) {
                    const int64_t r = row_of[a];
                    if (r < 0) { acc = NAN; break; }
                    o = load_elem(out_disp, odt, r * H + h);
                } else if (id < E + zero_n) {
                    o = 0.0;
                } else if (id < E + zero_n + copy_n) {
                    o = load_elem(ori_x, xdt, t * H + h);
                } else if (id < E + special) {
                    const int64_t c = id - E - zero_n - copy_n;
                    o = load_elem(alpha1, xdt, c) * load_elem(ori_x, xdt, t * H + h) +
                        load_elem(alpha2, xdt, c) * load_elem(const_v, xdt, c * H + h);
                } else {
                    acc = NAN;
                    break;
                }
                acc += sc * o;
                if (shared_x) acc += sc * load_elem(shared_x, xdt, t * H + h);
            }
            y[t * H + h] = acc;
        }
    }
    return 0;
}

/* ---- RMSNorm [ruDNN-7], Add + RMSNorm [Ascend-CARN] --------------------- */

/* y = x / sqrt(mean over H of x^2 + eps) * gamma, rstd = 1/sqrt(mean + eps).
 * Returns -1 when eps is not finite and positive. */
int oracle_rmsnorm(const void *x, int xdt, const void *gamma, int gdt, float eps,
                   int64_t T, int64_t H, void *y, int ydt, float *rstd)
{
    if (!(isfinite(eps) && eps > 0.0f)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double v = load_elem(x, xdt, t * H + h);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)H + (double)eps);
        if (rstd) rstd[t] = (float)r;
        for (int64_t h = 0; h < H; ++h)
            store_elem(y, ydt, t * H + h,
                       load_elem(x, xdt, t * H + h) * r * load_elem(gamma, gdt, h));
    }
    return 0;
}

/*
 * x = combine + residual, rounded to the residual dtype -> x_out;
 * rstd = 1/sqrt(mean(x_out^2) + eps) -> rstd (FP32);
 * y = x_out * rstd * gamma -> y (residual dtype).
 * combine is the unrounded double result of oracle_combine.
 */
int oracle_add_rmsnorm(const double *combine, const void *residual, int rdt,
                       const void *gamma, int gdt, float eps, int64_t T,
                       int64_t H, void *y, void *x_out, float *rstd)
{
    if (!(isfinite(eps) && eps > 0.0f)) return -1;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h)
            store_elem(x_out, rdt, t * H + h,
                       combine[t * H + h] + load_elem(residual, rdt, t * H + h));
    return oracle_rmsnorm(x_out, rdt, gamma, gdt, eps, T, H, y, rdt, rstd);
}

/* ---- first-order training [ruDNN-12] ------------------------------------ */

/*
 * Score of every expert of row t under a fixed selection: softmax over all E
 * logits (scoring 0) or the element-wise sigmoid (scoring 1), in double.
 * Returns 0 when the softmax row is invalid under the routing contract (a NaN
 * or +inf logit, or every logit -inf), else 1. For the sigmoid, scores of
 * NaN logits are NaN and +-inf give 1 and 0.
 */
static int row_scores(const void *logits, int ldt, int64_t t, int64_t E, int scoring,
                      double *p)
{
    if (scoring == 1) {
        for (int64_t e = 0; e < E; ++e)
            p[e] = 1.0 / (1.0 + exp(-load_elem(logits, ldt, t * E + e)));
        return 1;
    }
    int bad = 0, all_ninf = 1;
    double m = -INFINITY;
    for (int64_t e = 0; e < E; ++e) {
        double l = load_elem(logits, ldt, t * E + e);
        if (isnan(l) || (isinf(l) && l > 0.0)) bad = 1;
        if (!(isinf(l) && l < 0.0)) all_ninf = 0;
        if (l > m) m = l;
    }
    if (bad || all_ninf) return 0;
    double s = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        p[e] = exp(load_elem(logits, ldt, t * E + e) - m);
        s += p[e];
    }
    for (int64_t e = 0; e < E; ++e) p[e] /= s;
    return 1;
}

/*
 * Weights of a fixed selection: for slot j of token t, s_j = score of expert
 * idx[t,j] (a repeated id is gathered again); with renormalize, s_j / sum_i s_i
 * (the sum over the k slots); times scale; rounded once to wdt (FP32 in the
 * section; f64 for derivative checks). A slot id outside [0, E) makes the
 * row NaN, and so does an invalid softmax row. Returns the number of NaN
 * rows so made, or -1 on bad arguments.
 */
int64_t oracle_router_weights(const void *logits, int ldt, int64_t T, int64_t E,
                              const int64_t *idx, int64_t top_k, int scoring,
                              int renormalize, double scale, void *w, int wdt)
{
    if (T < 0 || E < 1 || top_k < 1 || top_k > E || top_k > 64 ||
        (scoring != 0 && scoring != 1) || !isfinite(scale) || !(scale > 0.0))
        return -1;
    double *p = (double *)malloc((size_t)E * sizeof(double));
    double sel[64];
    int64_t nan_rows = 0;
    for (int64_t t = 0; t < T; ++t) {
        int ok = row_scores(logits, ldt, t, E, scoring, p);
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = idx[t * top_k + j];
            if (e < 0 || e >= E) ok = 0;
            else sel[j] = p[e];
        }
        if (!ok) {
            for (int64_t j = 0; j < top_k; ++j) store_elem(w, wdt, t * top_k + j, (double)NAN);
            ++nan_rows;
            continue;
        }
        double z = 0.0;
        for (int64_t j = 0; j < top_k; ++j) z += sel[j];
        for (int64_t j = 0; j < top_k; ++j) {
            double v = renormalize ? sel[j] / z : sel[j];
            store_elem(w, wdt, t * top_k + j, v * scale);
        }
    }
    free(p);
    return nan_rows;
}

/*
 * Logits gradient of the weights above for an upstream gradient gw [T,k]
 * (FP32 in the section), by the chain rule in double:
 *   ds_j = scale * gw_j                                  without renormalize,
 *   ds_j = scale * (gw_j - sum_i gw_i s_i / Z) / Z,  Z = sum_i s_i, with it;
 *   G_e  = sum of ds_j over the slots j that hold expert e (gather adjoint);
 *   softmax: dl_e = p_e * (G_e - sum_f p_f G_f);
 *   sigmoid: dl_e = G_e * sigma_e * (1 - sigma_e) for the selected experts,
 *            0 for the others.
 * Rounded once to dldt (the logits dtype in the section). Rows that the
 * forward makes NaN (illegal id, invalid softmax row) are NaN. Returns the
 * number of such rows, or -1 on bad arguments.
 */
int64_t oracle_router_backward(const void *logits, int ldt, int64_t T, int64_t E,
                               const int64_t *idx, int64_t top_k, const void *gw, int gwdt,
                               int scoring, int renormalize, double scale, void *dl,
                               int dldt)
{
    if (T < 0 || E < 1 || top_k < 1 || top_k > E || top_k > 64 ||
        (scoring != 0 && scoring != 1) || !isfinite(scale) || !(scale > 0.0))
        return -1;
    double *p = (double *)malloc((size_t)E * sizeof(double));
    double *G = (double *)malloc((size_t)E * sizeof(double));
    double sel[64], ds[64];
    int64_t nan_rows = 0;
    for (int64_t t = 0; t < T; ++t) {
        int ok = row_scores(logits, ldt, t, E, scoring, p);
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = idx[t * top_k + j];
            if (e < 0 || e >= E) ok = 0;
            else sel[j] = p[e];
        }
        if (!ok) {
            for (int64_t e = 0; e < E; ++e) store_elem(dl, dldt, t * E + e, (double)NAN);
            ++nan_rows;
            continue;
        }
        if (renormalize) {
            double z = 0.0, gbar = 0.0;
            for (int64_t j = 0; j < top_k; ++j) z += sel[j];
            for (int64_t j = 0; j < top_k; ++j)
                gbar += load_elem(gw, gwdt, t * top_k + j) * sel[j];
            gbar /= z;
            for (int64_t j = 0; j < top_k; ++j)
                ds[j] = scale * (load_elem(gw, gwdt, t * top_k + j) - gbar) / z;
        } else {
            for (int64_t j = 0; j < top_k; ++j)
                ds[j] = scale * load_elem(gw, gwdt, t * top_k + j);
        }
        for (int64_t e = 0; e < E; ++e) G[e] = 0.0;
        for (int64_t j = 0; j < top_k; ++j) G[idx[t * top_k + j]] += ds[j];
        if (scoring == 0) {
            double c = 0.0;
            for (int64_t e = 0; e < E; ++e) c += p[e] * G[e];
            for (int64_t e = 0; e < E; ++e) store_elem(dl, dldt, t * E + e, p[e] * (G[e] - c));
        } else {
            /* only the selected logits move a sigmoid weight: the others get an
             * exact 0, even where their own logit is NaN */
            for (int64_t e = 0; e < E; ++e) store_elem(dl, dldt, t * E + e, 0.0);
            for (int64_t j = 0; j < top_k; ++j) {
                const int64_t e = idx[t * top_k + j];
                store_elem(dl, dldt, t * E + e, G[e] * p[e] * (1.0 - p[e]));
            }
        }
    }
    free(p); free(G);
    return nan_rows;
}

/*
 * Backward of the combine y[t] = sum_j w[t,j] * out_disp[row_of[t*k+j]]:
 *   dexpert[row_of[t*k+j]] = w[t,j] * gy[t]          (the routing weight
 *                                                     scales the gradient)
 *   dw[t,j] = sum_h gy[t,h] * out_disp[row_of[t*k+j], h]
 * in double. A slot with no row (row_of < 0) writes no dexpert row and gets
 * dw = NaN. dexpert rows no slot names stay 0.
 */
void oracle_combine_backward(const void *out_disp, int odt, const void *w, int wdt,
                             const int32_t *row_of, const void *gy, int gdt, int64_t T,
                             int64_t top_k, int64_t H, int64_t rows, double *dexpert,
                             double *dw)
{
    for (int64_t i = 0; i < rows * H; ++i) dexpert[i] = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < top_k; ++j) {
            const int64_t a = t * top_k + j;
            const int64_t r = row_of[a];
            if (r < 0) { dw[a] = NAN; continue; }
            const double wj = load_elem(w, wdt, a);
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const double g = load_elem(gy, gdt, t * H + h);
                dexpert[r * H + h] = wj * g;
                acc += g * load_elem(out_disp, odt, r * H + h);
            }
            dw[a] = acc;
        }
    }
}

/*
 * Backward of the bias-free SwiGLU expert o = Wd (silu(Wg x) * (Wu x)) for
 * every dispatched row r of expert e, given do = dout[r]:
 *   g = Wg x, u = Wu x, s = sigmoid(g), h = g s u      (recomputed)
 *   dh    = Wd^T do
 *   dg    = dh * u * s * (1 + g (1 - s))               (d silu / dg)
 *   du    = dh * g * s
 *   dx    = Wg^T dg + Wu^T du
 *   dWd  += do h^T,  dWg += dg x^T,  dWu += du x^T
 * All in double. dx is [nrows,H]; dgate, dup are [E,I,H] and ddown [E,H,I],
 * zeroed here and summed over every row of the expert. Returns -1 on an
 * expert id out of range.
 */
int oracle_swiglu_backward_rows(const void *xrows, int dt, int64_t nrows,
                                const int32_t *expert_of_row, const void *gate,
                                const void *up, const void *down, int64_t E, int64_t H,
                                int64_t I, const void *dout, int ddt, double *dx,
                                double *dgate, double *dup, double *ddown)
{
    for (int64_t i = 0; i < E * I * H; ++i) { dgate[i] = 0.0; dup[i] = 0.0; ddown[i] = 0.0; }
    double *xr = (double *)malloc((size_t)H * sizeof(double));
    double *dor = (double *)malloc((size_t)H * sizeof(double));
    double *hv = (double *)malloc((size_t)I * sizeof(double));
    double *dgv = (double *)malloc((size_t)I * sizeof(double));
    double *duv = (double *)malloc((size_t)I * sizeof(double));
    int rc = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t e = expert_of_row[r];
        if (e < 0 || e >= E) { rc = -1; break; }
        for (int64_t k = 0; k < H; ++k) {
            xr[k] = load_elem(xrows, dt, r * H + k);
            dor[k] = load_elem(dout, ddt, r * H + k);
        }
        for (int64_t i = 0; i < I; ++i) {
            double g = 0.0, u = 0.0, dh = 0.0;
            const int64_t wr = (e * I + i) * H;
            for (int64_t k = 0; k < H; ++k) {
                g += load_elem(gate, dt, wr + k) * xr[k];
                u += load_elem(up, dt, wr + k) * xr[k];
            }
            for (int64_t o = 0; o < H; ++o)
                dh += load_elem(down, dt, (e * H + o) * I + i) * dor[o];
            const double s = 1.0 / (1.0 + exp(-g));
            hv[i] = g * s * u;
            dgv[i] = dh * u * s * (1.0 + g * (1.0 - s));
            duv[i] = dh * g * s;
        }
        for (int64_t o = 0; o < H; ++o)
            for (int64_t i = 0; i < I; ++i)
                ddown[(e * H + o) * I + i] += dor[o] * hv[i];
        for (int64_t i = 0; i < I; ++i)
            for (int64_t k = 0; k < H; ++k) {
                dgate[(e * I + i) * H + k] += dgv[i] * xr[k];
                dup[(e * I + i) * H + k] += duv[i] * xr[k];
            }
        for (int64_t k = 0; k < H; ++k) {
            double acc = 0.0;
            for (int64_t i = 0; i < I; ++i)
                acc += load_elem(gate, dt, (e * I + i) * H + k) * dgv[i] +
                       load_elem(up, dt, (e * I + i) * H + k) * duv[i];
            dx[r * H + k] = acc;
        }
    }
    free(xr); free(dor); free(hv); free(dgv); free(duv);
    return rc;
}

/*
 * What the training forward keeps per dispatched row r of expert e: the gate
 * and up products g = Wg[e] x_r and u = Wu[e] x_r, and h = SiLU(g) * u, each
 * [nrows, I] in double. Returns -1 on an expert id out of range.
 */
int oracle_swiglu_cache_rows(const void *xrows, int dt, int64_t nrows,
                             const int32_t *expert_of_row, const void *gate, const void *up,
                             int64_t E, int64_t H, int64_t I, double *g_out, double *u_out,
                             double *h_out)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t e = expert_of_row[r];
        if (e < 0 || e >= E) return -1;
        for (int64_t i = 0; i < I; ++i) {
            double gv = 0.0, uv = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                const double xv = load_elem(xrows, dt, r * H + k);
                gv += load_elem(gate, dt, (e * I + i) * H + k) * xv;
                uv += load_elem(up, dt, (e * I + i) * H + k) * xv;
            }
            g_out[r * I + i] = gv;
            u_out[r * I + i] = uv;
            h_out[r * I + i] = gv / (1.0 + exp(-gv)) * uv;
        }
    }
    return 0;
}

/*
 * Backward of the dispatch gather: dx[t] = sum over slots j (slot order) of
 * dinput[row_of[t*k+j]], in double, without the routing weight (the combine
 * backward already applied it). A slot with no row contributes nothing (the
 * gather never copied x for it).
 */
void oracle_dispatch_backward(const void *dinput, int dt, const int32_t *row_of, int64_t T,
                              int64_t top_k, int64_t H, double *dx)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t j = 0; j < top_k; ++j) {
                const int64_t r = row_of[t * top_k + j];
                if (r >= 0) acc += load_elem(dinput, dt, r * H + h);
            }
            dx[t * H + h] = acc;
        }
}
