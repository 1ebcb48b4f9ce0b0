/*
 * moe_oracle.c -- plain, slow CPU oracle for the forward pass of one
 * mixture-of-experts (MoE) feed-forward layer with top-k gating, an optional
 * expert capacity, an always-on shared expert and the load-balancing loss.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this file.  The CUDA library
 * never calls it, shares no code, header, table or helper with it, and does
 * not fall back to it.
 *
 * Precision: fp32 inputs are widened exactly to double; every dot product,
 * softmax, SiLU, weight and sum is taken in double (fp64).  Loops run over
 * tokens, then experts, in the order the definitions below are written.
 *
 * Sources (page titles; the section or equation follows each citation):
 *   [M17]  "Mixture of Experts" (transformers-and-math, module 17)
 *   [SFR]  "Mixture of Experts: Sparse FFNs, Routers, and Shared Experts"
 *   [AEV]  "Mixture of experts" (AI engineering visualised)
 *   [MPF]  "Mixture of Experts: More Parameters, Same FLOPs"
 *   [FRT]  "Mixture of experts" (frontiers track)
 *
 * Parity pins (the tests that tie this file to the pages, not to itself):
 *   - worked example of [MPF] "The router": probabilities (0.50, 0.30, 0.15,
 *     0.05) at top-2 give weights 0.625 / 0.375;
 *   - softmax-over-selected weights sum to 1 ([M17] 17.2, [FRT] gate eq.);
 *   - closed forms of the balance loss ([M17] 17.4 and its exercise,
 *     [MPF] "Keeping the load even", [FRT] balance eq.);
 *   - the capacity exercise of [M17] 17.5 (C = 640) and the capacity
 *     invariants (per-expert kept count <= C, token-order priority checked by
 *     an independent recount);
 *   - one expert with k = 1 equals the dense SwiGLU MLP ([MPF] "A bug worth
 *     knowing about");
 *   - a dense "run every expert on every token, mask by routing" brute force
 *     on tiny inputs, and top-k selection against a full sort;
 *   - permuting the experts permutes the indices and leaves y unchanged;
 *   - E4M3 decode and encode against PyTorch's float8_e4m3fn (every code,
 *     every tie and its neighbours, random values), the row quantizer against
 *     its defining properties, and the E4M3 expert against the fp32 expert on
 *     weights that dequantize exactly;
 *   - the E4M3-activation expert against a recomputation with PyTorch's
 *     float8_e4m3fn casts and numpy matrix products, and, with an identity
 *     down projection, against the E4M3-weight expert and the row quantizer
 *     composed by hand.
 * Every exported function below is pinned by at least one of these.
 *
 * Weight layout: W_gate and W_up hold, per expert, F rows of D values
 * (row f = the coefficients of hidden unit f); W_down holds D rows of F
 * values.  [MPF] "An MoE tiny GPT" stores the transposes ([E,D,F], [E,F,D]);
 * the arithmetic is the same.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEMORY (-2)
#define ORACLE_NONFINITE (-3)

/* Gating modes.
 *   0: softmax over the k selected scores ([M17] 17.2 "Mixtral";
 *      [FRT] "Where the experts live", gate equation; [SFR] Router);
 *   1: softmax over all E scores, keep the k largest, no renormalisation
 *      ([M17] 17.2 "Switch Transformer and Qwen2"); with k = 1 this is the
 *      raw top-1 probability ([MPF] "The router", last remark);
 *   2: softmax over all E, renormalised over the chosen k
 *      ([MPF] "The router", equation MoE(x));
 *   3: sigmoid of each score, normalised over the chosen k ([MPF] "The
 *      router", closing remark: DeepSeek-V3 scores experts with a sigmoid
 *      rather than a softmax, normalised over the chosen ones).  For the
 *      balance loss's P_e the sigmoids are normalised over all E experts
 *      (reading: the "router probability" of a sigmoid router). */
#define MODE_SOFTMAX_SELECTED 0
#define MODE_SOFTMAX_ALL 1
#define MODE_SOFTMAX_ALL_RENORM 2
#define MODE_SIGMOID_SELECTED 3

/* Router scores: s[t][e] = sum_d x[t][d] * W_r[e][d] (+ bias[e]).
 * [MPF] "The router" (one score per expert, x W_r); [FRT] "Where the experts
 * live" (s = W_r x); [SFR] Router (a bias-free linear layer).  The optional
 * per-expert bias is part of the synthetic workloads, not of the pages. */
static void router_logits_f64(int64_t T, int64_t D, int64_t E, const double *x,
                              const float *W_r, const float *bias, double *s)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += x[t * D + d] * (double)W_r[e * D + d];
            if (bias)
                acc += (double)bias[e];
            s[t * E + e] = acc;
        }
    }
}

void oracle_router_logits(int64_t T, int64_t D, int64_t E, const float *x,
                          const float *W_r, const float *bias, double *s)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)(T * D > 0 ? T * D : 1));
    if (!xd)
        return;
    for (int64_t i = 0; i < T * D; ++i)
        xd[i] = (double)x[i];
    router_logits_f64(T, D, E, xd, W_r, bias, s);
    free(xd);
}

/* Softmax of one row of scores over all E experts, largest score subtracted
 * first ([MPF] "The router": a softmax turns the scores into probabilities). */
static void softmax_row(int64_t E, const double *s, double *p)
{
    double m = s[0];
    for (int64_t e = 1; e < E; ++e)
        if (s[e] > m)
            m = s[e];
    double z = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        p[e] = exp(s[e] - m);
        z += p[e];
    }
    for (int64_t e = 0; e < E; ++e)
        p[e] /= z;
}

/* Logistic sigmoid 1 / (1 + e^{-a}). */
static double sigmoid(double a)
{
    return 1.0 / (1.0 + exp(-a));
}

/* Top-k selection: k rounds, each taking the largest key not yet taken; on
 * equal keys the lower expert index wins (the pages leave tie order open;
 * this is the reading the whole build uses).  idx[0] has the largest key. */
static void topk_row(int64_t E, int64_t k, const double *s, unsigned char *taken,
                     int32_t *idx)
{
    memset(taken, 0, (size_t)E);
    for (int64_t j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || s[e] > s[best])
                best = e;
        }
        idx[j] = (int32_t)best;
        taken[best] = 1;
    }
}

/* Routing of T tokens from their scores s[T][E]:
 *   idx[t][0..k-1]  chosen experts, largest selection key first;
 *   w[t][0..k-1]    gate weights for the given mode;
 *   P_sum[e]        sum over tokens of the router probability of e (the
 *                   full softmax; mode 3: the sigmoids normalised over all E);
 *                   the balance loss's P_e is P_sum[e] / T;
 *   counts[e]       assignments (t, j) with idx[t][j] == e, before capacity.
 * sel_bias (nullable, [E]): a bias that only selection sees ([MPF] "Keeping
 * the load even", bias balancing: added to the scores only when choosing the
 * top k, never in the weights).  The selection key is then the score plus the
 * bias rounded to fp32, as the scores and biases are fp32 on the GPU; without
 * it the key is the score itself.  The weights always use the scores.
 * Returns ORACLE_OK, ORACLE_BAD_ARG or ORACLE_NONFINITE (a score is NaN/Inf). */
int oracle_route(int64_t T, int64_t E, int64_t k, int mode, const double *s,
                 const float *sel_bias, int32_t *idx, double *w, double *P_sum,
                 int64_t *counts)
{
    if (T < 0 || E < 1 || k < 1 || k > E || mode < 0 || mode > 3)
        return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < T * E; ++i)
        if (!isfinite(s[i]))
            return ORACLE_NONFINITE;
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double *key = (double *)malloc(sizeof(double) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!p || !key || !taken) {
        free(p);
        free(key);
        free(taken);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t e = 0; e < E; ++e) {
        P_sum[e] = 0.0;
        counts[e] = 0;
    }
    for (int64_t t = 0; t < T; ++t) {
        const double *st = s + t * E;
        int32_t *it = idx + t * k;
        double *wt = w + t * k;
        if (mode == MODE_SIGMOID_SELECTED) {
            double z = 0.0;
            for (int64_t e = 0; e < E; ++e) {
                p[e] = sigmoid(st[e]);
                z += p[e];
            }
            for (int64_t e = 0; e < E; ++e)
                p[e] /= z;
        } else {
            softmax_row(E, st, p);
        }
        for (int64_t e = 0; e < E; ++e)
            key[e] = sel_bias ? (double)(float)((float)st[e] + sel_bias[e]) : st[e];
        topk_row(E, k, key, taken, it);
        if (mode == MODE_SOFTMAX_SELECTED) {
            /* g_i = e^{s_i} / sum_{j in top-k} e^{s_j}; the largest selected
             * score is subtracted for range only. */
            double m = st[it[0]], z = 0.0;
            for (int64_t j = 1; j < k; ++j)
                if (st[it[j]] > m)
                    m = st[it[j]];
            for (int64_t j = 0; j < k; ++j)
                z += exp(st[it[j]] - m);
            for (int64_t j = 0; j < k; ++j)
                wt[j] = exp(st[it[j]] - m) / z;
        } else if (mode == MODE_SIGMOID_SELECTED) {
            /* w_i = sigmoid(s_i) / sum_{j in top-k} sigmoid(s_j) */
            double z = 0.0;
            for (int64_t j = 0; j < k; ++j)
                z += sigmoid(st[it[j]]);
            for (int64_t j = 0; j < k; ++j)
                wt[j] = sigmoid(st[it[j]]) / z;
        } else if (mode == MODE_SOFTMAX_ALL) {
            for (int64_t j = 0; j < k; ++j)
                wt[j] = p[it[j]];
        } else {
            /* w_e = p_e / sum_{e' in top-k} p_{e'} */
            double z = 0.0;
            for (int64_t j = 0; j < k; ++j)
                z += p[it[j]];
            for (int64_t j = 0; j < k; ++j)
                wt[j] = p[it[j]] / z;
        }
        for (int64_t e = 0; e < E; ++e)
            P_sum[e] += p[e];
        for (int64_t j = 0; j < k; ++j)
            counts[it[j]] += 1;
    }
    free(p);
    free(key);
    free(taken);
    return ORACLE_OK;
}

/* Expert capacity C = ceil(gamma * k * T / E) ([M17] 17.5 equation;
 * [AEV] "Capacity": phi times the fair share Tk/E; [MPF] "Keeping the load
 * even": a capacity factor times kN/E).  gamma <= 0 means dropless: -1. */
int64_t oracle_capacity(int64_t T, int64_t k, int64_t E, double gamma)
{
    if (gamma <= 0.0)
        return -1;
    const double c = ceil(gamma * (double)(T * k) / (double)E);
    /* no expert can be asked for more than T*k rows, so a capacity too large
     * for int64 drops nothing: saturate rather than overflow the cast */
    return c >= 9.2e18 ? INT64_MAX : (int64_t)c;
}

/* Capacity truncation in token order: walk t = 0..T-1 and j = 0..k-1; the
 * assignment (t, j) is kept iff fewer than C earlier assignments were kept by
 * expert idx[t][j].  An over-capacity assignment is dropped by that expert
 * only; the token keeps its other experts and its weights are not
 * renormalised ([M17] 17.5; [SFR] "Capacity factor": tokens arriving at a full
 * expert skip it; [AEV] "Capacity").  C < 0: nothing is dropped.
 * dropped[t][j] = 1 for a dropped assignment; kept[e] = assignments kept. */
void oracle_apply_capacity(int64_t T, int64_t k, int64_t E, int64_t C,
                           const int32_t *idx, uint8_t *dropped, int64_t *kept)
{
    for (int64_t e = 0; e < E; ++e)
        kept[e] = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            if (C < 0 || kept[e] < C) {
                kept[e] += 1;
                dropped[t * k + j] = 0;
            } else {
                dropped[t * k + j] = 1;
            }
        }
    }
}

/* Load-balancing loss aux = alpha * E * sum_e f_e * P_e with
 *   f_e = counts[e] / (T * k)   (fraction of token assignments, [FRT]
 *                                "Keeping the load balanced"; sums to 1),
 *   P_e = P_sum[e] / T          (mean router probability).
 * [M17] 17.4 equation; [SFR] "Auxiliary load-balancing loss"; [MPF] "Keeping
 * the load even".  T = 0 gives 0 (no tokens, no loss). */
double oracle_aux_loss(int64_t T, int64_t k, int64_t E, double alpha,
                       const int64_t *counts, const double *P_sum)
{
    if (T <= 0)
        return 0.0;
    double acc = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        double f = (double)counts[e] / (double)(T * k);
        double P = P_sum[e] / (double)T;
        acc += f * P;
    }
    return alpha * (double)E * acc;
}

/* SiLU(a) = a * sigmoid(a) = a / (1 + e^{-a}). */
static double silu(double a)
{
    return a / (1.0 + exp(-a));
}

/* One SwiGLU feed-forward network on one token:
 *   h_f = silu(sum_d W_gate[f][d] x_d) * (sum_d W_up[f][d] x_d),
 *   out_d = sum_f W_down[d][f] h_f
 * ([MPF] "An MoE tiny GPT": (silu(h G) * (h U)) D; [FRT] "Counting the
 * parameters yourself": three weight matrices per gated expert).
 * h is caller scratch of F doubles. */
static void swiglu_token(int64_t D, int64_t F, const double *x, const float *Wg,
                         const float *Wu, const float *Wd, double *h, double *out)
{
    for (int64_t f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            g += (double)Wg[f * D + d] * x[d];
            u += (double)Wu[f * D + d] * x[d];
        }
        h[f] = silu(g) * u;
    }
    for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t f = 0; f < F; ++f)
            acc += (double)Wd[d * F + f] * h[f];
        out[d] = acc;
    }
}

/* One SwiGLU expert applied to n token rows x[n][D] (fp64) -> out[n][D].
 * Rows are independent; OpenMP (when compiled in) splits them over host
 * threads without changing any row's arithmetic. */
int oracle_swiglu_rows(int64_t n, int64_t D, int64_t F, const double *x,
                       const float *Wg, const float *Wu, const float *Wd,
                       double *out)
{
    if (n < 0 || D < 1 || F < 1)
        return ORACLE_BAD_ARG;
    int err = 0;
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)F);
        if (!h) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; ++r)
            if (h)
                swiglu_token(D, F, x + r * D, Wg, Wu, Wd, h, out + r * D);
        free(h);
    }
    return err ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* A linear map of n rows: out[r][o] = sum_i in[r][i] * W[o][i], W [N_out][N_in]
 * (fp32, each output's coefficients contiguous), in and out fp64.  Used for
 * two projections of a latent MoE ([SFR], the Nemotron 3 Super variant after
 * 'The 2026 configuration table': the layer works at width 1024 inside a
 * 4096-wide model, x_lat = x W_in^T before it and y = y_lat W_out^T after). */
void oracle_linear(int64_t n, int64_t n_in, int64_t n_out, const double *in,
                   const float *W, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t o = 0; o < n_out; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < n_in; ++i)
                acc += in[r * n_in + i] * (double)W[o * n_in + i];
            out[r * n_out + o] = acc;
        }
}

/* The whole layer ([M17] 17.2 equation with the shared expert):
 *   y_t = FFN_shared(x_t) + sum_{j < k, kept} w_tj * FFN_{idx_tj}(x_t)
 * computed token by token.  The residual connection is the caller's: y
 * excludes x ([SFR] "Capacity factor": dropped tokens pass on the residual).
 *
 * s_in: scores to route on (e.g. another implementation's fp32 scores widened
 * to double); NULL to use the oracle's own oracle_router_logits().  The scores
 * used are written to s_out.  S = 0: no shared expert (Wsg/Wsu/Wsd unused).
 * bias_selection_only: 0 = the bias is part of the scores (selection and
 * weights); 1 = the bias only shifts the selection keys (oracle_route's
 * sel_bias) and the scores exclude it.
 * Output arrays: s_out[T][E], idx[T][k], w[T][k], dropped[T][k], counts[E],
 * kept[E], aux[1], y[T][D]. */
static int moe_forward_core(int64_t T, int64_t D, int64_t E, int64_t F, int64_t k,
                       int64_t S, int mode, double gamma, double alpha,
                       int bias_selection_only,
                       const double *x, const float *W_r, const float *bias,
                       const float *Wg, const float *Wu, const float *Wd,
                       const float *Wsg, const float *Wsu, const float *Wsd,
                       const double *s_in, double *s_out, int32_t *idx,
                       double *w, uint8_t *dropped, int64_t *counts,
                       int64_t *kept, double *aux, double *y)
{
    if (T < 0 || D < 1 || E < 1 || F < 1 || k < 1 || k > E || S < 0)
        return ORACLE_BAD_ARG;
    if (s_in)
        memcpy(s_out, s_in, sizeof(double) * (size_t)(T * E));
    else
        router_logits_f64(T, D, E, x, W_r, bias_selection_only ? NULL : bias, s_out);

    double *P_sum = (double *)malloc(sizeof(double) * (size_t)E);
    if (!P_sum)
        return ORACLE_NO_MEMORY;
    int rc = oracle_route(T, E, k, mode, s_out, bias_selection_only ? bias : NULL, idx, w,
                          P_sum, counts);
    if (rc != ORACLE_OK) {
        free(P_sum);
        return rc;
    }
    int64_t C = oracle_capacity(T, k, E, gamma);
    oracle_apply_capacity(T, k, E, C, idx, dropped, kept);
    *aux = oracle_aux_loss(T, k, E, alpha, counts, P_sum);
    free(P_sum);

    int err = 0;
#pragma omp parallel
    {
        int64_t hmax = F > S ? F : S;
        double *h = (double *)malloc(sizeof(double) * (size_t)hmax);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        if (!h || !o) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            if (!h || !o)
                continue;
            double *yt = y + t * D;
            for (int64_t d = 0; d < D; ++d)
                yt[d] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                if (dropped[t * k + j])
                    continue;
                int64_t e = idx[t * k + j];
                swiglu_token(D, F, x + t * D, Wg + e * F * D, Wu + e * F * D,
                             Wd + e * D * F, h, o);
                for (int64_t d = 0; d < D; ++d)
                    yt[d] += w[t * k + j] * o[d];
            }
            if (S > 0) {
                swiglu_token(D, S, x + t * D, Wsg, Wsu, Wsd, h, o);
                for (int64_t d = 0; d < D; ++d)
                    yt[d] += o[d];
            }
        }
        free(h);
        free(o);
    }
    return err ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* The layer on fp32 inputs (widened exactly to fp64). */
int oracle_moe_forward(int64_t T, int64_t D, int64_t E, int64_t F, int64_t k,
                       int64_t S, int mode, double gamma, double alpha,
                       int bias_selection_only,
                       const float *x, const float *W_r, const float *bias,
                       const float *Wg, const float *Wu, const float *Wd,
                       const float *Wsg, const float *Wsu, const float *Wsd,
                       const double *s_in, double *s_out, int32_t *idx,
                       double *w, uint8_t *dropped, int64_t *counts,
                       int64_t *kept, double *aux, double *y)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)(T * D > 0 ? T * D : 1));
    if (!xd)
        return ORACLE_NO_MEMORY;
    for (int64_t i = 0; i < T * D; ++i)
        xd[i] = (double)x[i];
    int rc = moe_forward_core(T, D, E, F, k, S, mode, gamma, alpha, bias_selection_only, xd, W_r,
                              bias, Wg, Wu, Wd, Wsg, Wsu, Wsd, s_in, s_out, idx, w, dropped,
                              counts, kept, aux, y);
    free(xd);
    return rc;
}

/* A latent MoE ([SFR], the Nemotron 3 Super variant after 'The 2026
 * configuration table': the whole layer runs at a narrower width L between
 * a projection down to L and one back up to the model width):
 *   x_lat = x W_in^T      (W_in [L][D_outer]),
 *   y_lat = the layer above on x_lat (everything at width L),
 *   y     = y_lat W_out^T (W_out [D_outer][L]).
 * Arguments as oracle_moe_forward with D = L, plus D_outer, W_in, W_out and
 * y [T][D_outer]; x [T][D_outer]. */
int oracle_latent_forward(int64_t T, int64_t D_outer, int64_t L, int64_t E, int64_t F,
                          int64_t k, int64_t S, int mode, double gamma, double alpha,
                          int bias_selection_only, const float *x, const float *W_in,
                          const float *W_out, const float *W_r, const float *bias,
                          const float *Wg, const float *Wu, const float *Wd,
                          const float *Wsg, const float *Wsu, const float *Wsd,
                          const double *s_in, double *s_out, int32_t *idx, double *w,
                          uint8_t *dropped, int64_t *counts, int64_t *kept, double *aux,
                          double *y)
{
    if (T < 0 || D_outer < 1 || L < 1)
        return ORACLE_BAD_ARG;
    const size_t nT = (size_t)(T > 0 ? T : 1);
    double *xd = (double *)malloc(sizeof(double) * nT * (size_t)D_outer);
    double *xl = (double *)malloc(sizeof(double) * nT * (size_t)L);
    double *yl = (double *)malloc(sizeof(double) * nT * (size_t)L);
    if (!xd || !xl || !yl) {
        free(xd);
        free(xl);
        free(yl);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t i = 0; i < T * D_outer; ++i)
        xd[i] = (double)x[i];
    oracle_linear(T, D_outer, L, xd, W_in, xl);
    int rc = moe_forward_core(T, L, E, F, k, S, mode, gamma, alpha, bias_selection_only, xl, W_r,
                              bias, Wg, Wu, Wd, Wsg, Wsu, Wsd, s_in, s_out, idx, w, dropped,
                              counts, kept, aux, yl);
    if (rc == ORACLE_OK)
        oracle_linear(T, L, D_outer, yl, W_out, y);
    free(xd);
    free(xl);
    free(yl);
    return rc;
}

/* ------------------------------------------------------------------------
 * e4m3 (FP8) expert weights.
 *
 * [MPF] "What experts cost at serving time" sizes serving memory at 8 bits
 * per weight and shows that decoding reads each expert weight for about two
 * FLOPs; the pages fix no 8-bit format.  Reading used here (and by the CUDA
 * path): the OCP FP8 E4M3 format -- sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, exponent field 0 holding subnormals m/8 * 2^-6, no
 * infinities, S.1111.111 = NaN, largest finite value 448 -- with one fp32
 * scale per weight row (output feature):
 *   scale_r = max_c |W[r][c]| / 448 (fp32 division; 1 for an all-zero row),
 *   q[r][c] = E4M3(W[r][c] / scale_r) (fp32 division, round to nearest,
 *             ties to even, magnitudes above 448 saturate to 448),
 * and the layer computes with W[r][c] = decode(q[r][c]) * scale_r.
 * ------------------------------------------------------------------------ */

/* Value of one E4M3 code. */
static double e4m3_value(uint8_t b)
{
    const int e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = (double)m * ldexp(1.0, -9);          /* m/8 * 2^-6 */
    else
        v = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    return (b & 0x80) ? -v : v;
}

/* E4M3 code of a fp32 value: round to nearest (ties to even) on the E4M3
 * grid, saturating to +-448; NaN stays NaN.  The grid spacing is 2^(e-3) for
 * a value in [2^e, 2^(e+1)) with e >= -6, and 2^-9 below 2^-6. */
static uint8_t e4m3_code(float v)
{
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    const double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int ex;
    frexp(a, &ex);                        /* a = f * 2^ex, f in [0.5, 1) */
    const int e = a == 0.0 ? -6 : (ex - 1 < -6 ? -6 : ex - 1);
    const double quantum = ldexp(1.0, e - 3);
    const double k = rint(a / quantum);   /* exact quotient; ties to even */
    const double r = k * quantum;
    if (r < ldexp(1.0, -6))               /* subnormal (k = 8 is 2^-6, code 8) */
        return (uint8_t)(sign | (uint8_t)k);
    frexp(r, &ex);
    const int er = ex - 1;                /* rounding may reach the next binade */
    const int mant = (int)((r / ldexp(1.0, er) - 1.0) * 8.0);
    return (uint8_t)(sign | ((er + 7) << 3) | mant);
}

void oracle_e4m3_decode(int64_t n, const uint8_t *codes, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_value(codes[i]);
}

void oracle_e4m3_encode(int64_t n, const float *v, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = e4m3_code(v[i]);
}

/* Row-wise quantization of W [rows][cols] (fp32 values of the bf16 weights)
 * by the definition above. */
void oracle_quantize_e4m3_rows(int64_t rows, int64_t cols, const float *W, uint8_t *q,
                               float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *w = W + r * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c)
            amax = fabsf(w[c]) > amax ? fabsf(w[c]) : amax;
        const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int64_t c = 0; c < cols; ++c)
            q[r * cols + c] = e4m3_code(w[c] / s);
    }
}

/* swiglu_token with W = decode(q) * scale (one scale per weight row); each
 * dequantized weight is exact in double. */
static void swiglu_token_q8(int64_t D, int64_t F, const double *x, const uint8_t *qg,
                            const float *sg, const uint8_t *qu, const float *su,
                            const uint8_t *qd, const float *sd, double *h, double *out)
{
    for (int64_t f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            g += e4m3_value(qg[f * D + d]) * (double)sg[f] * x[d];
            u += e4m3_value(qu[f * D + d]) * (double)su[f] * x[d];
        }
        h[f] = silu(g) * u;
    }
    for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t f = 0; f < F; ++f)
            acc += e4m3_value(qd[d * F + f]) * (double)sd[d] * h[f];
        out[d] = acc;
    }
}

/* oracle_swiglu_rows with e4m3 weights: qg, qu [F][D], qd [D][F] codes,
 * sg, su [F], sd [D] row scales. */
int oracle_swiglu_rows_q8(int64_t n, int64_t D, int64_t F, const double *x, const uint8_t *qg,
                          const float *sg, const uint8_t *qu, const float *su,
                          const uint8_t *qd, const float *sd, double *out)
{
    if (n < 0 || D < 1 || F < 1)
        return ORACLE_BAD_ARG;
    int err = 0;
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)F);
        if (!h) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; ++r)
            if (h)
                swiglu_token_q8(D, F, x + r * D, qg, sg, qu, su, qd, sd, h, out + r * D);
        free(h);
    }
    return err ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * E4M3 activations as well as E4M3 weights.
 *
 * [MPF] "What experts cost at serving time", in its arithmetic of published
 * configurations: DeepSeek-V3 sends the dispatched token rows in FP8.  The
 * pages fix no format or scaling for activations either.  Reading used here
 * (and by the CUDA path): every token row entering an expert, and the
 * expert's hidden row h between its two projections, is quantized with the
 * row rule above (one fp32 scale per row, scale = max|row| / 448); h is first
 * rounded to fp32 (the precision it is quantized in).  With dequantized
 * values x~ = decode(qx) * s_x and h~ = decode(qh) * s_h:
 *   h_f   = silu(sum_d Wg~[f][d] x~_d) * (sum_d Wu~[f][d] x~_d)   (fp64),
 *   out_d = sum_f Wd~[d][f] h~_f                                   (fp64),
 *   h~    = dequant(quantize(fp32(h))).
 * ------------------------------------------------------------------------ */

/* A row of n fp32 values replaced by its dequantized E4M3 values. */
static void dequantized_row(int64_t n, const float *v, double *out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        amax = fabsf(v[i]) > amax ? fabsf(v[i]) : amax;
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_value(e4m3_code(v[i] / s)) * (double)s;
}

/* The value of every E4M3 code (e4m3_value), looked up in the expert loops
 * below. */
static double e4m3_table[256];

static void swiglu_token_w8a8(int64_t D, int64_t F, const double *x, const uint8_t *qg,
                              const float *sg, const uint8_t *qu, const float *su,
                              const uint8_t *qd, const float *sd, float *v32, double *xq,
                              double *h, double *out)
{
    for (int64_t d = 0; d < D; ++d)
        v32[d] = (float)x[d];          /* exact for bf16 and fp32 inputs */
    dequantized_row(D, v32, xq);
    for (int64_t f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            g += e4m3_table[qg[f * D + d]] * (double)sg[f] * xq[d];
            u += e4m3_table[qu[f * D + d]] * (double)su[f] * xq[d];
        }
        v32[f] = (float)(silu(g) * u);
    }
    dequantized_row(F, v32, h);
    for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t f = 0; f < F; ++f)
            acc += e4m3_table[qd[d * F + f]] * (double)sd[d] * h[f];
        out[d] = acc;
    }
}

/* oracle_swiglu_rows_q8 with the token rows and the hidden rows quantized
 * too: x [n][D] (values of fp32 or bf16 inputs), codes and scales as there. */
int oracle_swiglu_rows_w8a8(int64_t n, int64_t D, int64_t F, const double *x,
                            const uint8_t *qg, const float *sg, const uint8_t *qu,
                            const float *su, const uint8_t *qd, const float *sd, double *out)
{
    if (n < 0 || D < 1 || F < 1)
        return ORACLE_BAD_ARG;
    const int64_t W = D > F ? D : F;
    for (int c = 0; c < 256; ++c)
        e4m3_table[c] = e4m3_value((uint8_t)c);
    int err = 0;
#pragma omp parallel
    {
        float *v32 = (float *)malloc(sizeof(float) * (size_t)W);
        double *xq = (double *)malloc(sizeof(double) * (size_t)D);
        double *h = (double *)malloc(sizeof(double) * (size_t)F);
        const int ok = v32 && xq && h;
        if (!ok) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; ++r)
            if (ok)
                swiglu_token_w8a8(D, F, x + r * D, qg, sg, qu, su, qd, sd, v32, xq, h,
                                  out + r * D);
        free(v32);
        free(xq);
        free(h);
    }
    return err ? ORACLE_NO_MEMORY : ORACLE_OK;
}
