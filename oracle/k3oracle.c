/*
 * k3oracle.c -- the plain, slow, fp64 CPU oracle for the MXFP4 routed-expert
 * MoE layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: the E2M1 table below is
 * spelled out here by hand and nowhere else in the repository.
 *
 * Every result is computed from its plain definition in double precision:
 * the packed weights are dequantised element by element with a 16-entry table
 * and the rule scale = 2^(e-127), then multiplied row by row in fp64.  The
 * only blocked/grouped form is orc_matvec_groupwise, which restates the
 * group-wise order described on the explainer page (ai.thesatyajit.com,
 * "kimi-k3-in-c", section "Reduction one: the experts already ship at half a
 * byte") so that a test can check the two orders agree to the bound stated in
 * that page's section "A floating-point contract, not a convention".
 *
 * Readings of the pages taken here (where they are silent or garbled):
 *  - E2M1 values: the OCP Microscaling v1.0 set {0, .5, 1, 1.5, 2, 3, 4, 6}
 *    with a sign bit; the pages name a "16-entry E2M1 table" but do not print
 *    it ("kimi-k3-in-c: A 176 KB Engine...", section "What byte-identical
 *    actually costs").  Code 8 is -0 and contributes 0.
 *  - E8M0 values: 2^(e-127); byte 255 is NaN and the whole 32-group then
 *    contributes 0 (same section; explainer, "Reduction one").
 *  - Nibble order: the low nibble is the even-index weight, the high nibble
 *    the odd one ("Running Kimi K3 locally", section "What are the four
 *    reductions, and why is the answer unchanged?").
 *  - Combine weights: softmax over the selected experts' UNBIASED logits; the
 *    selection bias only steers which experts are chosen ("Running Kimi K3
 *    locally", section "How is the C engine actually built?", invariant 3).
 *  - Ties in top-k selection go to the lower expert id; selected ids are
 *    returned in ascending id order with their weights aligned.
 *  - RMSNorm: y = x / sqrt(mean(x^2) + eps), epsilon inside the square root
 *    ("kimi-k3-in-c: A 176 KB Engine...", "What byte-identical actually
 *    costs"); unit gain.
 *  - Gated activation: SwiGLU, h = silu(g) * u with silu(z) = z / (1 + e^-z).
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ format */

/* The 16 E2M1 values, indexed by the 4-bit code (bit 3 = sign). */
static const double ORC_E2M1[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

typedef struct {
    const uint8_t *packed;  /* [rows][in/2]: two 4-bit codes per byte          */
    const uint8_t *scales;  /* [rows][in/32]: one E8M0 exponent per 32 weights */
    int rows;
    int in;
} orc_mat;

typedef struct {
    orc_mat gate;  /* [f x d] */
    orc_mat up;    /* [f x d] */
    orc_mat down;  /* [d x f] */
} orc_expert;

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double orc_e2m1_value(int code) { return ORC_E2M1[code & 15]; }

/* 2^(e-127); NaN for the reserved byte 255. */
double orc_e8m0_value(int e)
{
    if (e == 255) return NAN;
    return ldexp(1.0, e - 127);
}

/* 4-bit code of element j of row r: low nibble for even j, high for odd j. */
int orc_code(const orc_mat *W, int r, int j)
{
    const uint8_t b = W->packed[(size_t)r * (size_t)(W->in / 2) + (size_t)(j / 2)];
    return (j & 1) ? (b >> 4) : (b & 15);
}

/* Dequantised weight W[r][j]; a NaN scale zeroes its group. */
double orc_weight(const orc_mat *W, int r, int j)
{
    const int e = W->scales[(size_t)r * (size_t)(W->in / 32) + (size_t)(j / 32)];
    if (e == 255) return 0.0;
    return ORC_E2M1[orc_code(W, r, j)] * ldexp(1.0, e - 127);
}

/* Whole dense matrix in fp64, row-major [rows][in].  Rows are independent
 * (OpenMP over rows only; every element is orc_weight's value). */
void orc_dequant(double *Wd, const orc_mat *W)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < W->rows; r++)
        for (int j = 0; j < W->in; j++)
            Wd[(size_t)r * W->in + j] = orc_weight(W, r, j);
}

/* y = W x by the definition: dequantise row r, then sum_j W[r][j] x[j] in
 * fp64 with j ascending.  Rows are independent (OpenMP over rows only). */
void orc_matvec(double *y, const orc_mat *W, const double *x)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < W->rows; r++) {
        double acc = 0.0;
        for (int j = 0; j < W->in; j++) acc += orc_weight(W, r, j) * x[j];
        y[r] = acc;
    }
}

/* The group-wise order of the explainer page: for each 32-group, the dot
 * product of the table values with x, then that group's scale applied once;
 * a NaN-scale group is skipped; group results summed in fp64. */
void orc_matvec_groupwise(double *y, const orc_mat *W, const double *x)
{
    const int ngrp = W->in / 32;
    for (int r = 0; r < W->rows; r++) {
        double acc = 0.0;
        for (int g = 0; g < ngrp; g++) {
            const int e = W->scales[(size_t)r * ngrp + g];
            if (e == 255) continue;
            double sub = 0.0;
            for (int t = 0; t < 32; t++) {
                const int j = g * 32 + t;
                sub += ORC_E2M1[orc_code(W, r, j)] * x[j];
            }
            acc += sub * ldexp(1.0, e - 127);
        }
        y[r] = acc;
    }
}

/* Packed size of a rows x in matrix: in/2 nibble bytes + in/32 scale bytes a
 * row (0.53125 bytes per weight). */
int64_t orc_matrix_bytes(int64_t rows, int64_t in) { return rows * (in / 2 + in / 32); }

/* One expert: gate and up [f x d], down [d x f]. */
int64_t orc_expert_bytes(int64_t d, int64_t f) { return 3 * orc_matrix_bytes(f, d); }

/* ------------------------------------------------------------------ expert */

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* bf16 round-to-nearest-even of a double, returned as a double (used only for
 * the prefill contract where the SwiGLU output is handed to the down product
 * in bf16).  Written from the definition: keep 8 significant bits. */
double orc_round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    int ex;
    double m = frexp(fabs(v), &ex);          /* |v| = m * 2^ex, m in [0.5, 1) */
    double scaled = ldexp(m, 8);             /* 8 significant bits -> [128, 256) */
    double fl = floor(scaled), rem = scaled - fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = ldexp(fl, ex - 8);
    /* bf16 keeps fp32's exponent range; below 2^-126 it is subnormal with the
     * fixed spacing 2^-133.  Inputs here never go that small; guard anyway. */
    if (fabs(v) < ldexp(1.0, -126)) {
        double q = v / ldexp(1.0, -133);
        double qf = floor(q), qr = q - qf;
        if (qr > 0.5 || (qr == 0.5 && fmod(qf, 2.0) != 0.0)) qf += 1.0;
        return qf * ldexp(1.0, -133);
    }
    return copysign(r, v);
}

/* orc_silu and orc_round_bf16 over an array, in place: v[i] = silu(v[i]) *
 * u[i], rounded to bf16 if h_bf16 != 0 (the SwiGLU step of
 * orc_expert_forward_ex for many rows at once). */
void orc_swiglu_n(double *v, const double *u, int64_t n, int h_bf16)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        const double h = orc_silu(v[i]) * u[i];
        v[i] = h_bf16 ? orc_round_bf16(h) : h;
    }
}

/* y = W_d (silu(W_g x) * (W_u x)).  If h_bf16 != 0, h is rounded to bf16
 * before the down product.  h_out (optional) receives h [f]. */
void orc_expert_forward_ex(double *y, const orc_expert *E, const double *x, int h_bf16,
                           double *h_out)
{
    const int f = E->gate.rows;
    double *g = (double *)malloc(sizeof(double) * (size_t)f);
    double *u = (double *)malloc(sizeof(double) * (size_t)f);
    orc_matvec(g, &E->gate, x);
    orc_matvec(u, &E->up, x);
    for (int i = 0; i < f; i++) {
        double h = orc_silu(g[i]) * u[i];
        g[i] = h_bf16 ? orc_round_bf16(h) : h;
    }
    if (h_out) memcpy(h_out, g, sizeof(double) * (size_t)f);
    orc_matvec(y, &E->down, g);
    free(g);
    free(u);
}

void orc_expert_forward(double *y, const orc_expert *E, const double *x)
{
    orc_expert_forward_ex(y, E, x, 0, NULL);
}

/* ------------------------------------------- MXFP4 activations (mode B) */

/* Quantisation of activations to MXFP4 for a block-scaled product whose B
 * operand is E2M1 too.  The pages store only weights this way; the rule for
 * activations is the OCP Microscaling v1.0 conversion (a reading, not the
 * pages'): per 32-block the shared exponent is floor(log2(amax)) minus the
 * largest E2M1 exponent (2), as an E8M0 byte clamped to [0, 254]; each value
 * divided by 2^(e-127) is rounded to the nearest E2M1 magnitude, ties to the
 * even code, values above 6 saturating to 6.  A block holding a non-finite
 * value gets scale byte 255 and decodes to NaN.  codes[i] carries the sign in
 * bit 3 (a negative value that rounds to 0 gets code 8, -0).  Returns the
 * scale byte. */
int orc_mx_quant_block(uint8_t *codes, const float *x)
{
    double amax = 0.0;
    int bad = 0;
    for (int i = 0; i < 32; i++) {
        if (!isfinite(x[i])) bad = 1;
        else amax = fmax(amax, fabs((double)x[i]));
    }
    if (bad) {
        for (int i = 0; i < 32; i++) codes[i] = 0;
        return 255;
    }
    int e = 0;
    if (amax > 0.0) {
        int E;
        frexp(amax, &E);        /* amax = m 2^E, m in [0.5, 1): floor(log2 amax) = E - 1 */
        e = (E - 1) - 2 + 127;
        if (e < 0) e = 0;
        if (e > 254) e = 254;
    }
    const double inv = ldexp(1.0, 127 - e);
    for (int i = 0; i < 32; i++) {
        const double v = fabs((double)x[i]) * inv;  /* exact: a power-of-two scaling */
        /* midpoints of the magnitudes 0 .5 1 1.5 2 3 4 6; at a midpoint the
         * even code wins: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2,
         * 2.5 -> 2, 3.5 -> 4, 5 -> 4 */
        int c = (v > 0.25) + (v >= 0.75) + (v > 1.25) + (v >= 1.75) + (v > 2.5) + (v >= 3.5) +
                (v > 5.0);
        if (signbit(x[i])) c |= 8;
        codes[i] = (uint8_t)c;
    }
    return e;
}

/* xq[i] = the value of x[i]'s MXFP4 code, n a multiple of 32.  codes and
 * scales (n and n/32 bytes) may be null. */
void orc_mx_quantize(double *xq, uint8_t *codes, uint8_t *scales, const float *x, int n)
{
    uint8_t c[32];
    for (int b = 0; b < n / 32; b++) {
        const int e = orc_mx_quant_block(c, x + 32 * b);
        for (int i = 0; i < 32; i++) {
            xq[32 * b + i] = (e == 255) ? NAN : ORC_E2M1[c[i]] * ldexp(1.0, e - 127);
            if (codes) codes[32 * b + i] = c[i];
        }
        if (scales) scales[b] = (uint8_t)e;
    }
}

/* One expert with MXFP4 activations: x is quantised, g and u are computed
 * from it in fp64, h = silu(g) u is rounded to fp32 (the precision in which a
 * kernel holds h before it quantises it) and quantised, and y = W_down h. */
void orc_expert_forward_mxq(double *y, const orc_expert *E, const float *x)
{
    const int d = E->gate.in, f = E->gate.rows;
    double *xq = (double *)malloc(sizeof(double) * (size_t)d);
    double *g = (double *)malloc(sizeof(double) * (size_t)f);
    double *u = (double *)malloc(sizeof(double) * (size_t)f);
    float *h = (float *)malloc(sizeof(float) * (size_t)f);
    orc_mx_quantize(xq, NULL, NULL, x, d);
    orc_matvec(g, &E->gate, xq);
    orc_matvec(u, &E->up, xq);
    for (int i = 0; i < f; i++) h[i] = (float)(orc_silu(g[i]) * u[i]);
    orc_mx_quantize(g, NULL, NULL, h, f);
    orc_matvec(y, &E->down, g);
    free(xq);
    free(g);
    free(u);
    free(h);
}

/* ------------------------------------------------------------------ router */

/* bf16 bit pattern -> its exact value (bf16 is the top half of an fp32). */
double orc_bf16_value(uint16_t b)
{
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)b << 16;
    return (double)c.f;
}

/* logits[t][e] = sum_i W_r[e][i] x[t][i], W_r bf16 [E x d] row-major. */
void orc_router_logits(double *logits, const double *x, const uint16_t *Wr, int T, int E, int d)
{
#pragma omp parallel for schedule(static) collapse(2)
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            const uint16_t *w = Wr + (size_t)e * d;
            const double *xt = x + (size_t)t * d;
            for (int i = 0; i < d; i++) acc += orc_bf16_value(w[i]) * xt[i];
            logits[(size_t)t * E + e] = acc;
        }
}

/* Top-k of one token by repeated selection of the largest score (logit +
 * bias), ties to the lower id.  ids come out ascending, w[j] the softmax of
 * the UNBIASED logits over the chosen set.  Returns the selection margin:
 * score of rank k minus score of rank k+1 (+inf when k == E). */
double orc_topk_one(int32_t *ids, double *w, const double *logit, const double *bias, int E, int k)
{
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    double kth = 0.0, next = INFINITY;
    for (int r = 0; r < k + 1 && r < E; r++) {
        int best = -1;
        double bs = 0.0;
        for (int e = 0; e < E; e++) {
            if (taken[e]) continue;
            double s = logit[e] + (bias ? bias[e] : 0.0);
            if (best < 0 || s > bs) { best = e; bs = s; }
        }
        if (r < k) { taken[best] = 1; kth = bs; }
        else next = bs;
    }
    int n = 0;
    for (int e = 0; e < E; e++)
        if (taken[e]) ids[n++] = e;
    double mx = -INFINITY;
    for (int j = 0; j < k; j++) mx = fmax(mx, logit[ids[j]]);
    double s = 0.0;
    for (int j = 0; j < k; j++) { w[j] = exp(logit[ids[j]] - mx); s += w[j]; }
    for (int j = 0; j < k; j++) w[j] /= s;
    free(taken);
    return (k < E) ? kth - next : INFINITY;
}

void orc_topk(int32_t *ids, double *w, double *margin, const double *logits, const double *bias,
              int T, int E, int k)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        double m = orc_topk_one(ids + (size_t)t * k, w + (size_t)t * k, logits + (size_t)t * E,
                                bias, E, k);
        if (margin) margin[t] = m;
    }
}

/* Sigmoid router variant ("Running Kimi K3 locally", "How is the C engine
 * actually built?", invariant 3: top-k is taken on the biased score and the
 * combine weights are the UNBIASED sigmoid scores).  Per expert the score is
 * s_e = 1 / (1 + e^-logit_e); the k largest s_e + bias_e are chosen, ties to
 * the lower id, ids ascending.  w[j] = s_{ids[j]} when normalize == 0; the
 * pages do not say whether the weights are renormalised over the chosen set,
 * so normalize == 1 gives w[j] = s_{ids[j]} / sum_j s_{ids[j]} as the other
 * reading.  Returns the margin on s + bias (rank k minus rank k+1). */
double orc_topk_sigmoid_one(int32_t *ids, double *w, const double *logit, const double *bias, int E,
                            int k, int normalize)
{
    double *score = (double *)malloc(sizeof(double) * (size_t)E);
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    for (int e = 0; e < E; e++) score[e] = 1.0 / (1.0 + exp(-logit[e]));
    double kth = 0.0, next = INFINITY;
    for (int r = 0; r < k + 1 && r < E; r++) {
        int best = -1;
        double bs = 0.0;
        for (int e = 0; e < E; e++) {
            if (taken[e]) continue;
            double s = score[e] + (bias ? bias[e] : 0.0);
            if (best < 0 || s > bs) { best = e; bs = s; }
        }
        if (r < k) { taken[best] = 1; kth = bs; }
        else next = bs;
    }
    int n = 0;
    for (int e = 0; e < E; e++)
        if (taken[e]) ids[n++] = e;
    double sum = 0.0;
    for (int j = 0; j < k; j++) { w[j] = score[ids[j]]; sum += w[j]; }
    if (normalize)
        for (int j = 0; j < k; j++) w[j] /= sum;
    free(score);
    free(taken);
    return (k < E) ? kth - next : INFINITY;
}

void orc_topk_sigmoid(int32_t *ids, double *w, double *margin, const double *logits,
                      const double *bias, int T, int E, int k, int normalize)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        double m = orc_topk_sigmoid_one(ids + (size_t)t * k, w + (size_t)t * k,
                                        logits + (size_t)t * E, bias, E, k, normalize);
        if (margin) margin[t] = m;
    }
}

/* ------------------------------------------------------------------- layer */

/* out[t] = sum_j w[t][j] * expert_{ids[t][j]}(x[t]) for given routing (j in
 * ascending-id order).  experts[] has one entry per expert id; only the
 * selected ones are read.  h_bf16 as in orc_expert_forward_ex. */
void orc_combine(double *out, const double *x, int T, int d, const int32_t *ids, const double *w,
                 int k, const orc_expert *experts, int h_bf16)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int t = 0; t < T; t++) {
        double *o = out + (size_t)t * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        for (int j = 0; j < k; j++) {
            const int e = ids[(size_t)t * k + j];
            orc_expert_forward_ex(y, &experts[e], x + (size_t)t * d, h_bf16, NULL);
            const double wj = w[(size_t)t * k + j];
            for (int i = 0; i < d; i++) o[i] += wj * y[i];
        }
    }
    free(y);
}

/* The whole layer: router logits -> top-k -> weighted sum of expert outputs. */
void orc_layer_forward(double *out, int32_t *ids, double *w, double *margin, const double *x,
                       int T, int d, int E, int k, const uint16_t *Wr, const double *bias,
                       const orc_expert *experts, int h_bf16)
{
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * E);
    orc_router_logits(logits, x, Wr, T, E, d);
    orc_topk(ids, w, margin, logits, bias, T, E, k);
    orc_combine(out, x, T, d, ids, w, k, experts, h_bf16);
    free(logits);
}

/* ------------------------------------------- shared (always-on) experts */

/* One shared expert of the dense trunk, kept in bf16 (the pages keep the
 * trunk at 16 bits on purpose, "kimi-k3-in-c" explainer, "Why the trunk stays
 * at 16 bits"; each MoE layer has two shared experts that run on every token,
 * "Running Kimi K3 locally", "What are the four reductions, and why is the
 * answer unchanged?").  The same SwiGLU form as a routed expert:
 * y = W_down (silu(W_gate x) * (W_up x)), every bf16 weight exact in fp64,
 * each row sum in fp64 with j ascending.  gate, up: [f][d]; down: [d][f],
 * row-major bf16 bit patterns. */
void orc_shared_expert(double *y, const uint16_t *gate, const uint16_t *up, const uint16_t *down,
                       const double *x, int d, int f)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp parallel for schedule(static)
    for (int r = 0; r < f; r++) {
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; j++) {
            g += orc_bf16_value(gate[(size_t)r * d + j]) * x[j];
            u += orc_bf16_value(up[(size_t)r * d + j]) * x[j];
        }
        h[r] = orc_silu(g) * u;
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; c++) {
        double acc = 0.0;
        for (int r = 0; r < f; r++) acc += orc_bf16_value(down[(size_t)c * f + r]) * h[r];
        y[c] = acc;
    }
    free(h);
}

/* out[t] = sum over the n shared experts of shared_expert_s(x[t]): the
 * shared experts' outputs are added to the layer's output with weight 1 (a
 * reading: the pages name the shared experts but not how they combine; an
 * always-on expert has no router weight). */
void orc_shared_forward(double *out, const double *x, int T, int d, int f, int n,
                        const uint16_t *const *gates, const uint16_t *const *ups,
                        const uint16_t *const *downs)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int t = 0; t < T; t++) {
        double *o = out + (size_t)t * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        for (int s = 0; s < n; s++) {
            orc_shared_expert(y, gates[s], ups[s], downs[s], x + (size_t)t * d, d, f);
            for (int i = 0; i < d; i++) o[i] += y[i];
        }
    }
    free(y);
}

/* ----------------------------------------------------------------- rmsnorm */

void orc_rmsnorm(double *y, const double *x, int n, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    const double inv = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; i++) y[i] = x[i] * inv;
}

/* ------------------------------------------------------------------- cache */

/* Replay of an expert cache over a trace of batches (one batch = the keys one
 * layer of one token needs at the same time, so a batch's keys never evict
 * one another).  Policy: a present key is a hit and becomes most recently
 * used; a missing key takes an empty slot if one exists, else evicts the
 * least recently used slot that is neither pinned nor used by the current
 * batch.  Keys listed in `pinned` are loaded first and never evicted.
 * hit[i] receives 1/0 per trace entry.  Returns the hit count, or -1 when a
 * batch cannot be placed (no evictable slot). */
long long orc_cache_lru(uint8_t *hit, const int64_t *keys, const int32_t *batch_len, int nbatch,
                        int capacity, const int64_t *pinned, int npinned)
{
    int64_t *slot_key = (int64_t *)malloc(sizeof(int64_t) * (size_t)(capacity > 0 ? capacity : 1));
    long long *last = (long long *)malloc(sizeof(long long) * (size_t)(capacity > 0 ? capacity : 1));
    unsigned char *pin = (unsigned char *)calloc((size_t)(capacity > 0 ? capacity : 1), 1);
    long long *inbatch = (long long *)malloc(sizeof(long long) * (size_t)(capacity > 0 ? capacity : 1));
    long long hits = 0, now = 0;
    size_t pos = 0;
    if (npinned > capacity) { hits = -1; goto out; }
    for (int s = 0; s < capacity; s++) { slot_key[s] = -1; last[s] = -1; inbatch[s] = -1; }
    for (int p = 0; p < npinned; p++) { slot_key[p] = pinned[p]; pin[p] = 1; }
    for (int b = 0; b < nbatch; b++) {
        const int n = batch_len[b];
        /* hits first: the whole batch is needed at once */
        for (int i = 0; i < n; i++) {
            hit[pos + i] = 0;
            for (int s = 0; s < capacity; s++)
                if (slot_key[s] == keys[pos + i]) { hit[pos + i] = 1; last[s] = now; inbatch[s] = b; break; }
        }
        for (int i = 0; i < n; i++) {
            if (hit[pos + i]) { hits++; continue; }
            /* a key repeated inside one batch is a hit the second time */
            int dup = -1;
            for (int s = 0; s < capacity; s++)
                if (slot_key[s] == keys[pos + i]) { dup = s; break; }
            if (dup >= 0) { hit[pos + i] = 1; hits++; last[dup] = now; continue; }
            int v = -1;
            for (int s = 0; s < capacity; s++)
                if (slot_key[s] < 0) { v = s; break; }
            if (v < 0)
                for (int s = 0; s < capacity; s++) {
                    if (pin[s] || inbatch[s] == b) continue;
                    if (v < 0 || last[s] < last[v]) v = s;
                }
            if (v < 0) { hits = -1; goto out; }
            slot_key[v] = keys[pos + i];
            last[v] = now;
            inbatch[v] = b;
        }
        now++;
        pos += (size_t)n;
    }
out:
    free(slot_key); free(last); free(pin); free(inbatch);
    return hits;
}

/* Belady's offline policy on the same trace: a miss evicts the resident key
 * (not used by the current batch) whose next use is farthest in the future.
 * Returns the hit count (-1 if a batch cannot be placed). */
long long orc_cache_belady(const int64_t *keys, const int32_t *batch_len, int nbatch, int capacity)
{
    size_t total = 0;
    for (int b = 0; b < nbatch; b++) total += (size_t)batch_len[b];
    int *bidx = (int *)malloc(sizeof(int) * (total ? total : 1));
    size_t pos = 0;
    for (int b = 0; b < nbatch; b++)
        for (int i = 0; i < batch_len[b]; i++) bidx[pos++] = b;
    int64_t *slot_key = (int64_t *)malloc(sizeof(int64_t) * (size_t)(capacity > 0 ? capacity : 1));
    for (int s = 0; s < capacity; s++) slot_key[s] = -1;
    long long hits = 0;
    pos = 0;
    for (int b = 0; b < nbatch; b++) {
        const int n = batch_len[b];
        for (int i = 0; i < n; i++) {
            const int64_t kk = keys[pos + i];
            int found = -1;
            for (int s = 0; s < capacity; s++)
                if (slot_key[s] == kk) { found = s; break; }
            if (found >= 0) { hits++; continue; }
            int v = -1;
            for (int s = 0; s < capacity; s++)
                if (slot_key[s] < 0) { v = s; break; }
            if (v < 0) {
                size_t far = 0;
                for (int s = 0; s < capacity; s++) {
                    /* not evictable if the current batch uses it */
                    int used_now = 0;
                    for (int q = 0; q < n; q++)
                        if (keys[pos + q] == slot_key[s]) { used_now = 1; break; }
                    if (used_now) continue;
                    size_t nx = pos + (size_t)n;
                    while (nx < total && keys[nx] != slot_key[s]) nx++;
                    if (v < 0 || nx > far) { v = s; far = nx; }
                }
            }
            if (v < 0) { hits = -1; goto out; }
            slot_key[v] = kk;
        }
        pos += (size_t)n;
    }
out:
    free(bidx); free(slot_key);
    return hits;
}
