/*
 * oracle.c -- plain, slow CPU oracle for the FastMTP verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (jina-ocr-v1, "Jina AI's jina-ocr-v1 Is Selling
 * Throughput", section "The speed comes from three layers working together";
 * evolve.pub review, "Summary" and "Scope & Claims", Section 3.1 / Eq. 2):
 *   - one DeepSeek-style MoE FFN layer: a router product x.W_r^T, a softmax
 *     gate over all E routed experts (not renormalised over the selection),
 *     the top-k experts by router score (ties to the lower expert index),
 *     SwiGLU experts down(silu(gate.x) * up.x), S always-on shared experts of
 *     weight 1, and the gate-weighted sum;
 *   - greedy verification: the longest draft prefix that matches the
 *     verifier's greedy tokens is committed, followed by the verifier's own
 *     token at the first mismatch (a correction) or after the last draft (the
 *     "bonus token when all drafts match").  The committed tokens are then
 *     exactly what plain greedy decoding emits ("lossless").
 *
 * Precision: expert arithmetic and the gate are evaluated in double from the
 * exact bf16 inputs with no intermediate rounding.  The router scores that
 * decide the top-k selection are accumulated in float (the CUDA kernel's
 * precision), in plain index order, because floating point decides an
 * integer there; the workloads keep consecutive router places at least 1e-3
 * apart so that the order of summation cannot flip a decision.
 *
 * bf16 values are passed as their uint16 bit patterns.
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bff(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* silu(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------ router */

/* Router scores of one token: logit[e] = sum_h x[h] * W_r[e,h], float
 * accumulation in increasing h. */
static void router_scores(const uint16_t *x, const uint16_t *w_router, int H, int E, float *logit) {
    for (int e = 0; e < E; ++e) {
        float acc = 0.0f;
        const uint16_t *w = w_router + (size_t)e * H;
        for (int h = 0; h < H; ++h) {
            float p = bff(x[h]) * bff(w[h]);
            acc = acc + p;
        }
        logit[e] = acc;
    }
}

/* Top-k by router score, descending; among equal scores the lower expert
 * index comes first.  Picks the best remaining expert k times. */
static void select_topk(const float *logit, int E, int k, int32_t *idx) {
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    for (int s = 0; s < k; ++s) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || logit[e] > logit[best]) best = e;
        }
        idx[s] = best;
        taken[best] = 1;
    }
    free(taken);
}

/* Routing of T tokens: topk_idx [T,k], topk_w [T,k] = softmax probability of
 * the selected expert (softmax over all E, no renormalisation); logits [T,E]
 * optional. */
int oracle_route(const uint16_t *x, const uint16_t *w_router, int T, int H, int E, int k,
                 int32_t *topk_idx, double *topk_w, float *logits_out) {
    if (T < 0 || H <= 0 || E <= 0 || k < 0 || k > E) return -1;
    float *logit = (float *)malloc(sizeof(float) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        router_scores(x + (size_t)t * H, w_router, H, E, logit);
        if (logits_out) memcpy(logits_out + (size_t)t * E, logit, sizeof(float) * (size_t)E);
        double m = logit[0];
        for (int e = 1; e < E; ++e) if (logit[e] > m) m = logit[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp((double)logit[e] - m);
        select_topk(logit, E, k, topk_idx + (size_t)t * k);
        for (int s = 0; s < k; ++s) {
            int e = topk_idx[(size_t)t * k + s];
            topk_w[(size_t)t * k + s] = exp((double)logit[e] - m) / z;
        }
    }
    free(logit);
    return 0;
}

/* Smallest distance between consecutive router places 1..min(k+1,E) of each
 * token, from router scores computed exactly (double) on the bf16 inputs.
 * Used to keep only well-posed selections in the test workloads. */
int oracle_route_gaps(const uint16_t *x, const uint16_t *w_router, int T, int H, int E, int k,
                      double *gap) {
    if (T < 0 || H <= 0 || E <= 0 || k < 0 || k > E) return -1;
    double *v = (double *)malloc(sizeof(double) * (size_t)E);
    int places = k < E ? k + 1 : E;
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (size_t)t * H;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            const uint16_t *w = w_router + (size_t)e * H;
            for (int h = 0; h < H; ++h) acc += bf(xt[h]) * bf(w[h]);
            v[e] = acc;
        }
        /* partial selection sort of the first `places` places */
        for (int p = 0; p < places; ++p) {
            int best = p;
            for (int e = p + 1; e < E; ++e) if (v[e] > v[best]) best = e;
            double tmp = v[p]; v[p] = v[best]; v[best] = tmp;
        }
        double g = INFINITY;
        for (int p = 0; p + 1 < places; ++p) if (v[p] - v[p + 1] < g) g = v[p] - v[p + 1];
        gap[t] = g;
    }
    free(v);
    return 0;
}

/* --------------------------------------------------------------- permutation */

/* Expert-contiguous order of the T*k (token, slot) pairs.  Entry i = t*k+s.
 * counts[e] = number of pairs routed to e; offsets = exclusive prefix sum
 * (offsets[E] = T*k); perm_src lists the pairs expert by expert, each
 * expert's pairs in increasing token order; inv is its inverse.
 * Returns -2 if an index lies outside [0,E). */
int oracle_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                   int32_t *offsets, int32_t *perm_src, int32_t *inv) {
    if (T < 0 || k < 0 || E <= 0) return -1;
    size_t n = (size_t)T * (size_t)k;
    for (size_t i = 0; i < n; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return -2;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < n; ++i) counts[topk_idx[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    size_t pos = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int s = 0; s < k; ++s) {
                size_t i = (size_t)t * k + s;
                if (topk_idx[i] == e) {
                    perm_src[pos] = (int32_t)i;
                    inv[i] = (int32_t)pos;
                    ++pos;
                }
            }
    return 0;
}

/* ------------------------------------------------------------------ experts */

/* One SwiGLU expert on one token:
 *   y[h] = sum_j Wd[h, j] * silu(sum_c Wg[j,c] x[c]) * (sum_c Wu[j,c] x[c])
 * gate rows Wg[j] = wg + j*H, up rows Wu[j] = wu + j*H, down element
 * Wd[h,j] = wd[h*ld_down + j].  Accumulates into y (double, length H). */
static void swiglu_expert(const uint16_t *x, const uint16_t *wg, const uint16_t *wu,
                          const uint16_t *wd, int ld_down, int H, int I, double *y, double *a) {
    for (int j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        const uint16_t *rg = wg + (size_t)j * H, *ru = wu + (size_t)j * H;
        for (int c = 0; c < H; ++c) {
            double xc = bf(x[c]);
            g += bf(rg[c]) * xc;
            u += bf(ru[c]) * xc;
        }
        a[j] = silu(g) * u;
    }
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        const uint16_t *rd = wd + (size_t)h * ld_down;
        for (int j = 0; j < I; ++j) acc += bf(rd[j]) * a[j];
        y[h] += acc;
    }
}

/* Routed expert e applied to token row x: w_gate_up [E,2I,H] (rows 0..I-1
 * gate, I..2I-1 up), w_down [E,H,I].  y = E_e(x), overwritten. */
static void routed_expert(const uint16_t *x, const uint16_t *w_gate_up, const uint16_t *w_down,
                          int e, int H, int I, double *y, double *a) {
    const uint16_t *base = w_gate_up + (size_t)e * 2 * I * H;
    for (int h = 0; h < H; ++h) y[h] = 0.0;
    swiglu_expert(x, base, base + (size_t)I * H, w_down + (size_t)e * H * I, I, H, I, y, a);
}

/* Sum of the S shared experts on x: ws_gate_up [2SI,H] holds the S gate
 * blocks (rows s*I..), then the S up blocks (rows S*I + s*I..); ws_down
 * [H,S*I] holds expert s's down matrix in columns s*I..s*I+I-1. */
static void shared_experts(const uint16_t *x, const uint16_t *ws_gate_up, const uint16_t *ws_down,
                           int S, int H, int I, double *y, double *a) {
    for (int h = 0; h < H; ++h) y[h] = 0.0;
    for (int s = 0; s < S; ++s)
        swiglu_expert(x, ws_gate_up + (size_t)s * I * H, ws_gate_up + ((size_t)S * I + (size_t)s * I) * H,
                      ws_down + (size_t)s * I, S * I, H, I, y, a);
}

/* Routed expert outputs for a list of (token, expert) rows:
 * y[r,:] = E_{expert[r]}(x[token[r],:]).  y is [n,H] double. */
int oracle_expert_rows(const uint16_t *x, const uint16_t *w_gate_up, const uint16_t *w_down,
                       int H, int I, int E, const int32_t *token, const int32_t *expert, int n,
                       double *y) {
    if (H <= 0 || I <= 0 || n < 0) return -1;
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
    for (int r = 0; r < n; ++r) {
        if (expert[r] < 0 || expert[r] >= E) { free(a); return -2; }
        routed_expert(x + (size_t)token[r] * H, w_gate_up, w_down, expert[r], H, I, y + (size_t)r * H, a);
    }
    free(a);
    return 0;
}

/* Shared-expert sum for a list of tokens: y[r,:] = sum_s S_s(x[token[r],:]). */
int oracle_shared_rows(const uint16_t *x, const uint16_t *ws_gate_up, const uint16_t *ws_down,
                       int H, int I, int S, const int32_t *token, int n, double *y) {
    if (H <= 0 || I <= 0 || S < 0 || n < 0) return -1;
    double *a = (double *)malloc(sizeof(double) * (size_t)(I > 0 ? I : 1));
    for (int r = 0; r < n; ++r)
        shared_experts(x + (size_t)token[r] * H, ws_gate_up, ws_down, S, H, I, y + (size_t)r * H, a);
    free(a);
    return 0;
}

/* Gate-weighted combine: out[t,:] = sum_s w[t,s] * y_perm[inv[t*k+s],:] + y_shared[t,:],
 * summed in slot order, then the shared term.  Inputs float, output double. */
int oracle_combine(const float *y_perm, const int32_t *inv, const float *topk_w,
                   const float *y_shared, int T, int k, int H, double *out) {
    if (T < 0 || k < 0 || H <= 0) return -1;
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int s = 0; s < k; ++s) {
                size_t r = (size_t)inv[(size_t)t * k + s];
                acc += (double)topk_w[(size_t)t * k + s] * (double)y_perm[r * H + h];
            }
            if (y_shared) acc += (double)y_shared[(size_t)t * H + h];
            out[(size_t)t * H + h] = acc;
        }
    return 0;
}

/* The whole MoE layer for the listed tokens (all T when token == NULL):
 *   out[r,:] = sum_{s<k} p[t, idx[t,s]] * E_{idx[t,s]}(x_t) + sum_{s<S} S_s(x_t)
 * Routing (idx, p) as in oracle_route.  out [n,H] double; idx_out [n,k] and
 * w_out [n,k] optional. */
int oracle_moe_layer(const uint16_t *x, const uint16_t *w_router, const uint16_t *w_gate_up,
                     const uint16_t *w_down, const uint16_t *ws_gate_up, const uint16_t *ws_down,
                     int T, int H, int E, int k, int S, int I, const int32_t *token, int n,
                     double *out, int32_t *idx_out, double *w_out) {
    if (T < 0 || H <= 0 || E <= 0 || k < 0 || k > E || S < 0 || I <= 0) return -1;
    if (token == NULL) n = T;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
    for (int r = 0; r < n; ++r) {
        int t = token ? token[r] : r;
        if (t < 0 || t >= T) { free(idx); free(p); free(y); free(a); return -2; }
        const uint16_t *xt = x + (size_t)t * H;
        oracle_route(xt, w_router, 1, H, E, k, idx, p, NULL);
        double *o = out + (size_t)r * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int s = 0; s < k; ++s) {
            routed_expert(xt, w_gate_up, w_down, idx[s], H, I, y, a);
            for (int h = 0; h < H; ++h) o[h] += p[s] * y[h];
        }
        if (S > 0) {
            shared_experts(xt, ws_gate_up, ws_down, S, H, I, y, a);
            for (int h = 0; h < H; ++h) o[h] += y[h];
        }
        if (idx_out) memcpy(idx_out + (size_t)r * k, idx, sizeof(int32_t) * (size_t)k);
        if (w_out) memcpy(w_out + (size_t)r * k, p, sizeof(double) * (size_t)k);
    }
    free(idx); free(p); free(y); free(a);
    return 0;
}

/* Residual update and normalisation between stacked layers:
 *   x_next = bf16(x + y),   h_next = x_next / sqrt(mean(x_next^2) + eps)
 * x_next is returned as double holding the rounded bf16 value (rounded to
 * nearest even), h_next in double without rounding. */
static double round_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t r = ((u >> 16) & 1u) + 0x7FFFu;
    u = (u + r) & 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_rmsnorm_residual(const uint16_t *x, const uint16_t *y, int T, int H, double eps,
                            double *x_next, double *h_next) {
    if (T < 0 || H <= 0) return -1;
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            double v = round_bf16(bf(x[(size_t)t * H + h]) + bf(y[(size_t)t * H + h]));
            x_next[(size_t)t * H + h] = v;
            ss += v * v;
        }
        double scale = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) h_next[(size_t)t * H + h] = x_next[(size_t)t * H + h] * scale;
    }
    return 0;
}

/* -------------------------------------------------------------- verification */

/* Greedy verification of B sequences with K drafts each.
 * logits [B, K+1, V] (bf16 bits): row j is the verifier's prediction for the
 * position after input j, where input 0 is the last committed token and input
 * j >= 1 is draft j.  drafts [B, K].
 *   g[b,j]       = first index attaining the maximum of row (b,j)
 *   accept_len_b = largest L <= K with drafts[b,i] == g[b,i] for all i < L
 *   committed[b] = drafts[b,0..L-1], then g[b,L], then -1 up to K+1 entries
 * A draft outside [0,V) can equal no greedy token, so it is a mismatch. */
int oracle_accept(const uint16_t *logits, const int32_t *drafts, int B, int K, int V,
                  int32_t *argmax, int32_t *accept_len, int32_t *committed) {
    if (B < 0 || K < 0 || V <= 0) return -1;
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j <= K; ++j) {
            const uint16_t *row = logits + ((size_t)b * (K + 1) + j) * (size_t)V;
            int best = 0;
            float bv = bff(row[0]);
            for (int v = 1; v < V; ++v) {
                float f = bff(row[v]);
                if (f > bv) { bv = f; best = v; }
            }
            argmax[(size_t)b * (K + 1) + j] = best;
        }
        int L = 0;
        while (L < K && drafts[(size_t)b * K + L] == argmax[(size_t)b * (K + 1) + L]) ++L;
        accept_len[b] = L;
        int32_t *c = committed + (size_t)b * (K + 1);
        for (int i = 0; i < L; ++i) c[i] = drafts[(size_t)b * K + i];
        c[L] = argmax[(size_t)b * (K + 1) + L];
        for (int i = L + 1; i <= K; ++i) c[i] = -1;
    }
    return 0;
}
