/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU statement of one MoE layer
 * of the Colibri GLM-5.2 engine: Route -> Union -> expert FFN (int4 SwiGLU,
 * routed + shared) -> score-weighted combine -> Learn (hit counters).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code.  It shares nothing with the
 * CUDA library (no headers, helpers, tables or constants) and the CUDA library
 * never calls it.
 *
 * Arithmetic: every floating-point step is fp64; inputs arrive as fp32 (the
 * pages keep activations and gate parameters in fp32: "Public Colibri
 * Observation and Revision Ledger", section "Exact Architecture and Data-Flow
 * Reconstruction").  Loops are written in the order of the definitions below,
 * with no blocking, fusion or reordering; OpenMP only splits independent
 * (token) or (output row) work and never a reduction, so results do not depend
 * on the thread count.
 *
 * Sources (page title, section):
 *  [arch]  "Public Colibri Observation and Revision Ledger", "Exact Architecture
 *         and Data-Flow Reconstruction": sigmoid router with n_group=1 over the
 *         experts of a layer; a routed expert's three weight matrices sit
 *         next to each other in one int4 block; a shared expert that every
 *         token uses; router parameters in fp32.
 *  [stages] same page and section: the five per-layer stages Route, Union,
 *         Place, Overlap, Learn; routing and precision are unchanged by them.
 *  [hits]  same section: per-expert hit counters updated after each token.
 *  [union] same page, "Cache/Prefetch Design Comparison" figure caption: the
 *         batch-union reads each unique expert once per batched decode.
 *  [R-idea] colibri README, "The idea": ~11 GB of routed experts change per
 *         token, which with 75 layers and ~19 MB experts means 8 experts per
 *         token and layer (k = 8).
 *  [R-path] colibri README, "How it works / The per-token path": placement only
 *         decides speed; router decisions and weight precision are identical.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - int4 values are symmetric two's complement in [-8, 7]; element 2i of a row
 *    is the low nibble of byte i, element 2i+1 the high nibble; rows are
 *    row-major [rows][cols/2].
 *  - one fp32 scale per G consecutive elements along the input (reduction) axis
 *    of every output row: scales are [rows][cols/G].
 *  - per expert the three matrices are gate [f][d], up [f][d], down [d][f], in
 *    that order: first all packed bytes, then all scales.
 *  - FFN(x) = down( silu(gate x) * (up x) ), silu(g) = g * sigmoid(g).
 *  - selection key = sigmoid(logit) + bias[e]; the bias only selects, the
 *    combine weight uses the unbiased sigmoid score.
 *  - top-k order: key descending, equal keys -> lower expert id first.
 *  - weights: normalize = 0 -> w_j = s_j;  normalize = 1 ->
 *    w_j = route_scale * s_j / sum_j' s_j'.
 *  - out_t = res_t + shared(x_t) + sum_{j<k} w_tj FFN_{e_tj}(x_t), summed left
 *    to right in slot order.
 *  - union: counts per expert, offsets = exclusive scan over ascending expert
 *    id, pairs p = t*k + j stably ordered by (expert, p), perm[p] = position of
 *    pair p in that order, sorted_pair[position] = p, uniq = experts with a
 *    non-zero count in ascending order.
 *  - hits[e] += counts[e] (one count per routed (token, slot) pair).
 *  - top-p pruning (lossy, off at top_p = 1): of the k chosen experts in
 *    selection order, the shortest prefix whose scores reach top_p times the
 *    scores of all k is kept; the other slots hold id -1 and weight 0, join no
 *    union group and add nothing to the output or the hit counters.
 *
 * Pins: every function here is pinned by the CPU test suite (closed forms,
 * invariants, brute force, exhaustive enumeration).  Nothing printed on the
 * pages fixes the GLM-5.2 bias / normalisation semantics themselves: those two
 * readings are "parity unpinned" against the real model, although the code that
 * states them is pinned to their definitions.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- int4 ---- */

/* Signed value of element `i` of a packed int4 row (two's complement nibble). */
static int nibble_value(const uint8_t *row, int64_t i)
{
    uint8_t byte = row[i / 2];
    int v = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    if (v >= 8)
        v -= 16;
    return v;
}

/* Unpack n int4 elements into int8 values in [-8, 7]. */
ORACLE_API void oracle_int4_unpack(const uint8_t *q, int64_t n, int8_t *v)
{
    for (int64_t i = 0; i < n; i++)
        v[i] = (int8_t)nibble_value(q, i);
}

/* Pack n int8 values (each must be in [-8, 7]) into n/2 bytes; returns the
 * number of values that were out of range (they are stored modulo 16). */
ORACLE_API int64_t oracle_int4_pack(const int8_t *v, int64_t n, uint8_t *q)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; i += 2) {
        int lo = v[i], hi = (i + 1 < n) ? v[i + 1] : 0;
        if (lo < -8 || lo > 7) bad++;
        if (hi < -8 || hi > 7) bad++;
        q[i / 2] = (uint8_t)(((unsigned)lo & 0x0F) | (((unsigned)hi & 0x0F) << 4));
    }
    return bad;
}

/* deq(W)[r, i] = q[r, i] * s[r, floor(i / G)] for a [rows][cols] matrix. */
static double deq(const uint8_t *q, const float *s, int64_t cols, int G,
                  int64_t r, int64_t i)
{
    return (double)nibble_value(q + r * (cols / 2), i) *
           (double)s[r * (cols / G) + i / G];
}

/* Dequantise a whole [rows][cols] matrix to fp64 (used by tiny-size tests). */
ORACLE_API void oracle_dequant(const uint8_t *q, const float *s, int64_t rows,
                               int64_t cols, int G, double *w)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t i = 0; i < cols; i++)
            w[r * cols + i] = deq(q, s, cols, G, r, i);
}

/* Bytes of one expert block: packed nibbles of gate, up, down, then scales. */
ORACLE_API int64_t oracle_expert_q_bytes(int64_t d, int64_t f)
{
    return 3 * d * f / 2;
}

ORACLE_API int64_t oracle_expert_s_count(int64_t d, int64_t f, int G)
{
    return 3 * d * f / G;
}

/* ---------------------------------------------------------------- route --- */

static double sigmoid(double v)
{
    return 1.0 / (1.0 + exp(-v));
}

/* l[t, e] = sum_i x[t, i] * Wg[e, i]   (fp64, i ascending; the (t, e) sums
 * are independent and may run on any thread). */
ORACLE_API void oracle_router_logits(const float *x, const float *wg, int T,
                                     int d, int E, double *logits)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int i = 0; i < d; i++)
                acc += (double)x[(int64_t)t * d + i] * (double)wg[(int64_t)e * d + i];
            logits[(int64_t)t * E + e] = acc;
        }
}

/* True when expert a must come before expert b in the top-k order. */
static int key_before(double ka, int a, double kb, int b)
{
    if (ka != kb)
        return ka > kb;
    return a < b;
}

/*
 * Route one token: scores s_e = sigmoid(l_e), keys s_e + bias_e, top-k by key
 * (descending, ties -> lower id), then weights.  Selection is done by k passes
 * that each pick the best expert not yet chosen.
 *
 * top_p < 1 prunes the selection (the lossy "top-p gating" of "Public Colibri
 * Observation and Revision Ledger", "Exact-Versus-Lossy Mode Table"; the
 * `--topp` setting of the summary page "Colibri is an open-source, lightweight
 * Mixture-of-Experts", "Configuration"): the k chosen experts, in selection
 * order, keep their shortest prefix of m >= 1 slots whose scores add up to at
 * least top_p times the scores of all k,
 *     m = min { m : s_1 + ... + s_m >= top_p * (s_1 + ... + s_k) },
 * and the other k - m slots become empty (id -1, weight 0).  Normalised
 * weights are then taken over the m kept slots.  top_p >= 1 keeps all k.
 */
static void route_token(const double *l, const float *bias, int E, int k,
                        int normalize, double route_scale, double top_p,
                        int32_t *idx, double *w, double *keys)
{
    double *key = keys;
    char *taken = calloc((size_t)E, 1);
    for (int e = 0; e < E; e++)
        key[e] = sigmoid(l[e]) + (bias ? (double)bias[e] : 0.0);
    for (int j = 0; j < k; j++) {
        int best = -1;
        for (int e = 0; e < E; e++) {
            if (taken[e])
                continue;
            if (best < 0 || key_before(key[e], e, key[best], best))
                best = e;
        }
        taken[best] = 1;
        idx[j] = best;
        w[j] = sigmoid(l[best]);
    }
    int m = k;
    if (top_p < 1.0) {
        double total = 0.0;
        for (int j = 0; j < k; j++)
            total += w[j];
        double cum = 0.0;
        for (m = 1; m <= k; m++) {
            cum += w[m - 1];
            if (cum >= top_p * total)
                break;
        }
        if (m > k)
            m = k;
        for (int j = m; j < k; j++) {
            idx[j] = -1;
            w[j] = 0.0;
        }
    }
    if (normalize) {
        double sum = 0.0;
        for (int j = 0; j < m; j++)
            sum += w[j];
        for (int j = 0; j < m; j++)
            w[j] = route_scale * w[j] / sum;
    }
    free(taken);
}

/*
 * Route T tokens.  Outputs: idx [T][k] int32, w [T][k] fp64, and optionally
 * logits [T][E] and keys [T][E] (fp64; either may be NULL).  top_p as in
 * route_token (1 = plain top-k).
 */
ORACLE_API void oracle_route_topp(const float *x, const float *wg, const float *bias,
                                  int T, int d, int E, int k, int normalize,
                                  double route_scale, double top_p, int32_t *idx,
                                  double *w, double *logits_out, double *keys_out)
{
    double *logits = logits_out ? logits_out : malloc(sizeof(double) * (size_t)T * E);
    oracle_router_logits(x, wg, T, d, E, logits);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        double *keys = keys_out ? keys_out + (int64_t)t * E : malloc(sizeof(double) * (size_t)E);
        route_token(logits + (int64_t)t * E, bias, E, k, normalize, route_scale, top_p,
                    idx + (int64_t)t * k, w + (int64_t)t * k, keys);
        if (!keys_out)
            free(keys);
    }
    if (!logits_out)
        free(logits);
}

ORACLE_API void oracle_route(const float *x, const float *wg, const float *bias,
                             int T, int d, int E, int k, int normalize,
                             double route_scale, int32_t *idx, double *w,
                             double *logits_out, double *keys_out)
{
    oracle_route_topp(x, wg, bias, T, d, E, k, normalize, route_scale, 1.0, idx, w,
                      logits_out, keys_out);
}

/* Same as oracle_route_topp, but from precomputed fp64 logits [T][E]. */
ORACLE_API void oracle_route_from_logits(const double *logits, const float *bias,
                                         int T, int E, int k, int normalize,
                                         double route_scale, double top_p, int32_t *idx,
                                         double *w, double *keys_out)
{
    for (int t = 0; t < T; t++) {
        double *keys = keys_out ? keys_out + (int64_t)t * E : malloc(sizeof(double) * (size_t)E);
        route_token(logits + (int64_t)t * E, bias, E, k, normalize, route_scale, top_p,
                    idx + (int64_t)t * k, w + (int64_t)t * k, keys);
        if (!keys_out)
            free(keys);
    }
}

/* ---------------------------------------------------------------- union --- */

/*
 * Batch union of the routed (token, slot) pairs p = t*k + j.  A slot holding
 * -1 is empty (pruned by top-p): it joins no group and gets perm[p] = -1.
 * Returns 0, or -1 when any other expert id is outside [0, E).
 */
ORACLE_API int oracle_union(const int32_t *idx, int T, int k, int E,
                            int32_t *counts, int32_t *offsets, int32_t *perm,
                            int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq)
{
    int64_t P = (int64_t)T * k;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t p = 0; p < P; p++) {
        if (idx[p] == -1)
            continue;
        if (idx[p] < 0 || idx[p] >= E)
            return -1;
        counts[idx[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    /* stable placement: walk pairs in ascending p, each takes the next free
     * position of its expert's range */
    int32_t *next = malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; e++)
        next[e] = offsets[e];
    for (int64_t p = 0; p < P; p++) {
        if (idx[p] == -1) {
            perm[p] = -1;
            continue;
        }
        int32_t pos = next[idx[p]]++;
        perm[p] = pos;
        sorted_pair[pos] = (int32_t)p;
    }
    free(next);
    int32_t n = 0;
    for (int e = 0; e < E; e++)
        if (counts[e] > 0)
            uniq[n++] = e;
    *n_uniq = n;
    return 0;
}

/* Learn: hits[e] += counts[e]. */
ORACLE_API void oracle_hits(const int32_t *counts, int E, uint64_t *hits)
{
    for (int e = 0; e < E; e++)
        hits[e] += (uint64_t)counts[e];
}

/* ------------------------------------------------------------------ FFN --- */

/*
 * One expert on one token.  q/s point at the expert block (gate | up | down
 * packed bytes, then gate | up | down scales).  y has d entries (fp64).
 *   g_r = sum_i deq(Wgate)[r, i] x_i,  u_r = sum_i deq(Wup)[r, i] x_i
 *   h_r = g_r * sigmoid(g_r) * u_r
 *   y_c = sum_r deq(Wdown)[c, r] h_r
 */
ORACLE_API void oracle_expert_ffn(const float *x, const uint8_t *q, const float *s,
                                  int d, int f, int G, double *y)
{
    const uint8_t *q_gate = q;
    const uint8_t *q_up = q + (int64_t)f * d / 2;
    const uint8_t *q_down = q + 2 * (int64_t)f * d / 2;
    const float *s_gate = s;
    const float *s_up = s + (int64_t)f * d / G;
    const float *s_down = s + 2 * (int64_t)f * d / G;
    double *h = malloc(sizeof(double) * (size_t)f);
    /* Output rows are independent: they are split over the OpenMP threads when
     * this runs outside another parallel region (one token, as in decode).
     * Every row's sum keeps its order, so the bits do not depend on it. */
#pragma omp parallel for schedule(static)
    for (int r = 0; r < f; r++) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; i++) {
            g += deq(q_gate, s_gate, d, G, r, i) * (double)x[i];
            u += deq(q_up, s_up, d, G, r, i) * (double)x[i];
        }
        h[r] = g * sigmoid(g) * u;
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; c++) {
        double acc = 0.0;
        for (int r = 0; r < f; r++)
            acc += deq(q_down, s_down, f, G, c, r) * h[r];
        y[c] = acc;
    }
    free(h);
}

/* Threads of the OpenMP runtime (1 without OpenMP). */
static int max_threads(void);

/* The same FFN for a list of tokens (independent).  With at least as many
 * tokens as threads, OpenMP splits the tokens; with fewer, the rows inside
 * each token's FFN are split instead. */
ORACLE_API void oracle_expert_ffn_tokens(const float *x, const int32_t *tokens,
                                         int n, const uint8_t *q, const float *s,
                                         int d, int f, int G, double *y)
{
#pragma omp parallel for schedule(dynamic, 1) if (n >= max_threads())
    for (int i = 0; i < n; i++)
        oracle_expert_ffn(x + (int64_t)tokens[i] * d, q, s, d, f, G,
                          y + (int64_t)i * d);
}

/* --------------------------------------------------------------- layer ---- */

typedef struct {
    const float *x;        /* [T][d] */
    const float *wg;       /* [E][d] */
    const float *bias;     /* [E] or NULL */
    const uint8_t *q_base; /* E expert blocks, expert e at e * expert_q_bytes */
    const float *s_base;   /* E scale blocks, expert e at e * expert_s_count */
    const uint8_t *shared_q;
    const float *shared_s;
    const float *res;      /* [T][d] or NULL */
    int T, d, f, E, k, G, normalize;
    double route_scale;
    double top_p;          /* 1 = plain top-k; < 1 prunes as in route_token */
} oracle_layer;

/*
 * Dense masked evaluation for the tokens listed in `tokens` (n of them; pass
 * all 0..T-1 for the whole layer).  For each listed token t:
 *   out[t] = res[t] + shared(x_t) + sum_{j<k} w_tj FFN_{e_tj}(x_t)
 * Experts outside the top-k have mask 0 and contribute nothing, so they are
 * not evaluated.  idx/w/out are indexed by list position i (idx [n][k],
 * w [n][k], out [n][d]).
 */
ORACLE_API void oracle_moe_layer_tokens(const oracle_layer *L, const int32_t *tokens,
                                        int n, int32_t *idx, double *w, double *out)
{
    const int d = L->d, E = L->E, k = L->k;
    const int64_t qb = oracle_expert_q_bytes(d, L->f);
    const int64_t sc = oracle_expert_s_count(d, L->f, L->G);
#pragma omp parallel for schedule(dynamic, 1) if (n >= max_threads())
    for (int i = 0; i < n; i++) {
        int t = tokens[i];
        const float *xt = L->x + (int64_t)t * d;
        double *l = malloc(sizeof(double) * (size_t)E);
        double *keys = malloc(sizeof(double) * (size_t)E);
        double *y = malloc(sizeof(double) * (size_t)d);
        double *o = out + (int64_t)i * d;
        oracle_router_logits(xt, L->wg, 1, d, E, l);
        route_token(l, L->bias, E, k, L->normalize, L->route_scale, L->top_p,
                    idx + (int64_t)i * k, w + (int64_t)i * k, keys);
        oracle_expert_ffn(xt, L->shared_q, L->shared_s, d, L->f, L->G, y);
        for (int c = 0; c < d; c++)
            o[c] = (L->res ? (double)L->res[(int64_t)t * d + c] : 0.0) + y[c];
        for (int j = 0; j < k; j++) {
            int e = idx[(int64_t)i * k + j];
            double wj = w[(int64_t)i * k + j];
            if (e < 0)
                continue;   /* slot emptied by top-p */
            oracle_expert_ffn(xt, L->q_base + e * qb, L->s_base + e * sc, d, L->f,
                              L->G, y);
            for (int c = 0; c < d; c++)
                o[c] += wj * y[c];
        }
        free(l);
        free(keys);
        free(y);
    }
}

/*
 * Union-path evaluation of the whole layer (all T tokens): route every token,
 * form the batch union, evaluate each unique expert once over its grouped
 * pairs (y_pair in union order), evaluate the shared expert per token, then
 * combine per token in slot order through perm.  The per-(token, expert) FFN
 * and the combine order are those of the dense path, so both paths give the
 * same fp64 bits.  Also returns the union arrays.
 */
ORACLE_API int oracle_moe_layer_union(const oracle_layer *L, int32_t *idx, double *w,
                                      int32_t *counts, int32_t *offsets,
                                      int32_t *perm, int32_t *sorted_pair,
                                      int32_t *uniq, int32_t *n_uniq, double *out)
{
    const int T = L->T, d = L->d, E = L->E, k = L->k;
    const int64_t qb = oracle_expert_q_bytes(d, L->f);
    const int64_t sc = oracle_expert_s_count(d, L->f, L->G);
    oracle_route_topp(L->x, L->wg, L->bias, T, d, E, k, L->normalize, L->route_scale,
                      L->top_p, idx, w, NULL, NULL);
    if (oracle_union(idx, T, k, E, counts, offsets, perm, sorted_pair, uniq, n_uniq))
        return -1;
    int64_t P = (int64_t)T * k;
    double *y_pair = malloc(sizeof(double) * (size_t)(P * d));
    double *y_shared = malloc(sizeof(double) * (size_t)T * d);
    for (int u = 0; u < *n_uniq; u++) {
        int e = uniq[u];
        int n = counts[e];
        int32_t *tok = malloc(sizeof(int32_t) * (size_t)n);
        for (int i = 0; i < n; i++)
            tok[i] = sorted_pair[offsets[e] + i] / k;
        oracle_expert_ffn_tokens(L->x, tok, n, L->q_base + e * qb, L->s_base + e * sc,
                                 d, L->f, L->G, y_pair + (int64_t)offsets[e] * d);
        free(tok);
    }
    int32_t *all = malloc(sizeof(int32_t) * (size_t)T);
    for (int t = 0; t < T; t++)
        all[t] = t;
    oracle_expert_ffn_tokens(L->x, all, T, L->shared_q, L->shared_s, d, L->f, L->G,
                             y_shared);
    free(all);
    for (int t = 0; t < T; t++)
        for (int c = 0; c < d; c++) {
            double o = (L->res ? (double)L->res[(int64_t)t * d + c] : 0.0) +
                       y_shared[(int64_t)t * d + c];
            for (int j = 0; j < k; j++) {
                int32_t pos = perm[(int64_t)t * k + j];
                if (pos < 0)
                    continue;   /* slot emptied by top-p */
                o += w[(int64_t)t * k + j] * y_pair[(int64_t)pos * d + c];
            }
            out[(int64_t)t * d + c] = o;
        }
    free(y_pair);
    free(y_shared);
    return 0;
}

/* ------------------------------------------------------- layer stack ---- */

/* RMS normalisation of each row before a stacked MoE layer:
 *   n[t][i] = x[t][i] / sqrt( (1/d) sum_i x[t][i]^2 + eps ),  unit weight.
 * [arch] keeps the norms of the dense part in fp32; a stack of MoE layers with
 * nothing between them is not defined numerically (the SwiGLU is quadratic in
 * x, so activations overflow fp32 within four layers at the stated weight
 * distribution).  Reading: each stacked layer sees the RMS-normalised residual
 * stream, out_l = x_l + MoE(norm(x_l)), the pre-norm placement of the model
 * family.  Returns fp64 rows; the layer input is their fp32 rounding. */
ORACLE_API void oracle_rms_norm(const float *x, int T, int d, double eps, double *out)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        const float *xr = x + (int64_t)t * d;
        double ss = 0.0;
        for (int i = 0; i < d; i++)
            ss += (double)xr[i] * (double)xr[i];
        const double r = 1.0 / sqrt(ss / d + eps);
        for (int i = 0; i < d; i++)
            out[(int64_t)t * d + i] = (double)xr[i] * r;
    }
}

/* Thread count the OpenMP runtime will use (1 without OpenMP), and a setter
 * for it (tests check that results do not depend on it). */
#ifdef _OPENMP
#include <omp.h>
static int max_threads(void) { return omp_get_max_threads(); }
ORACLE_API void oracle_set_threads(int n) { if (n > 0) omp_set_num_threads(n); }
#else
static int max_threads(void) { return 1; }
ORACLE_API void oracle_set_threads(int n) { (void)n; }
#endif
ORACLE_API int oracle_threads(void) { return max_threads(); }
