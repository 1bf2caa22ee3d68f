/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously-correct CPU definition of the Mixtral sparse
 * mixture-of-experts feed-forward layer.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg may build, load or call this file.  It
 * shares no code, header, table or helper with the CUDA library; the two see
 * the same seeded inputs and nothing else.
 *
 * Every floating-point accumulation is done in double precision, term by term,
 * in index order, with no blocking or reordering.  OpenMP only spreads whole,
 * independent tokens over host threads (a token's result never depends on
 * another token: "Mixtral > Architecture Overview", paragraph on sparse
 * feed-forward computation).
 *
 * What each function follows:
 *   - router: a linear layer x . W_g giving one score per expert, the two
 *     largest kept, the rest set to -inf, and a softmax over what survives
 *     ("Mixtral of Experts" (azimuth.plus), router paragraph; "Mixtral of
 *     Experts" (tellworld.net), "How Mixtral 8x7B is built": two experts per
 *     token).
 *   - expert: a SwiGLU feed-forward network with its own weights
 *     ("Mixtral of Experts" (azimuth.plus), expert paragraph), made of gate,
 *     up and down projections 4096 -> 14336 -> 4096 ("Mixtral > Architecture
 *     Overview", parameter-count paragraph).
 *   - combine: the selected experts' outputs summed, weighted by the gates
 *     ("Mixtral & Sparse MoE (2024) > The Solution", routing paragraph).
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   - ties between equal scores go to the lower expert index;
 *   - SwiGLU uses beta = 1, i.e. silu(u) = u / (1 + exp(-u));
 *   - W1 is the gate projection, W3 the up projection, W2 the down projection;
 *   - the router has no bias; the optional per-expert bias is a benchmark
 *     construct added to the logits before selection;
 *   - router logits are stored as fp32 (one rounding of the exact sum);
 *   - the layer output is rounded once, to nearest-even, after the weighted sum;
 *   - RMSNorm (for the stacked-layer harness) uses gain 1;
 *   - variants: gating 1 = softmax over all experts then top-k without
 *     renormalising; a per-expert capacity keeps each expert's first
 *     `capacity` selections in token order, and a dropped slot's gate mass is
 *     either lost or spread proportionally over the token's kept slots.
 *
 * Layouts (row-major, the same as the library's):
 *   x    [T][d]        W_g  [E][d]
 *   W1[e], W3[e]  [ffn][d]   (row c holds the input weights of feature c)
 *   W2[e]         [d][ffn]   (row n holds the input weights of output n)
 *   out  [T][d]
 * Element type: 0 = fp32, 1 = bf16 (raw 16-bit patterns).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_NO_MEM = -2, ORACLE_NONFINITE = -3 };

/* ---- element access ---------------------------------------------------- */

/* bf16 is the top half of an IEEE binary32 pattern. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double elem(const void *p, size_t i, int dt)
{
    if (dt == ORACLE_F32)
        return (double)((const float *)p)[i];
    return bf16_bits_to_double(((const uint16_t *)p)[i]);
}

/* Nearest bf16 to v, ties to the even pattern; one rounding straight from
 * double.  Three neighbouring candidates around the float truncation are
 * compared by exact distance in double. */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    float f = (float)v;
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    uint32_t sign = b & 0x80000000u;
    double av = fabs(v);
    /* largest finite bf16 plus half an ulp: at or above it, nearest-even
     * rounding gives infinity */
    if (av >= 3.3961775292304e38)
        return (uint16_t)((sign | 0x7F800000u) >> 16);
    uint32_t trunc = (b & 0x7FFFFFFFu) & 0xFFFF0000u;
    uint32_t best = trunc;
    double bestd = INFINITY;
    for (int step = -1; step <= 1; ++step) {
        int64_t m = (int64_t)trunc + (int64_t)step * 0x10000;
        if (m < 0 || m > 0x7F7F0000)
            continue;
        uint32_t cb = (uint32_t)m;
        float c;
        memcpy(&c, &cb, sizeof c);
        double dist = fabs((double)c - av);
        if (dist < bestd || (dist == bestd && ((cb >> 16) & 1u) == 0)) {
            bestd = dist;
            best = cb;
        }
    }
    return (uint16_t)((sign | best) >> 16);
}

double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }

static void store_elem(void *p, size_t i, int dt, double v)
{
    if (dt == ORACLE_F32)
        ((float *)p)[i] = (float)v; /* C conversion: round to nearest even */
    else
        ((uint16_t *)p)[i] = oracle_double_to_bf16(v);
}

/* ---- router --------------------------------------------------------------- */

/* Logit of expert e for one token: the exact dot product x . W_g[e], plus the
 * optional bias, stored as fp32. */
static float router_logit(const void *x_row_base, size_t x_off, const void *Wg,
                          const float *bias, int d, int e, int dt)
{
    double s = 0.0;
    for (int i = 0; i < d; ++i)
        s += elem(x_row_base, x_off + (size_t)i, dt) * elem(Wg, (size_t)e * d + i, dt);
    if (bias)
        s += (double)bias[e];
    return (float)s;
}

/* Keep the k largest logits: pick the largest unchosen one k times; on equal
 * values the lower index is picked first.  Slot 0 holds the largest. */
static void select_top_k(const float *l, int E, int k, int *chosen)
{
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int q = 0; q < j; ++q)
                if (chosen[q] == e)
                    taken = 1;
            if (taken)
                continue;
            if (best < 0 || l[e] > l[best])
                best = e;
        }
        chosen[j] = best;
    }
}

/* Gating modes.
 *   0: keep the top k scores, set the others to -inf, softmax over what
 *      survives ("Mixtral of Experts" (azimuth.plus), router paragraph);
 *   1: softmax over all E scores, then keep the top k, without renormalising
 *      the kept probabilities (a reading of "Mixtral & Sparse MoE (2024) > The
 *      Solution", routing paragraph: scores normalised by a softmax, top-2
 *      selected, outputs combined by their routing scores).
 * The largest logit (chosen[0]) is subtracted before exponentiating. */
static void gates_of(const float *l, const int *chosen, int E, int k, int gating, double *g)
{
    double l0 = (double)l[chosen[0]];
    if (gating == 0) {
        double z = 0.0;
        for (int j = 0; j < k; ++j)
            z += exp((double)l[chosen[j]] - l0);
        for (int j = 0; j < k; ++j)
            g[j] = exp((double)l[chosen[j]] - l0) / z;
    } else {
        double zall = 0.0;
        for (int e = 0; e < E; ++e)
            zall += exp((double)l[e] - l0);
        for (int j = 0; j < k; ++j)
            g[j] = exp((double)l[chosen[j]] - l0) / zall;
    }
}

static int all_finite_f32(const float *p, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        if (!isfinite(p[i]))
            return 0;
    return 1;
}

/* Capacity ("Mixtral & Sparse MoE (2024) > The Solution", load-balancing
 * paragraph: a limit on how many tokens each expert takes).  Reading: an
 * expert keeps its first `capacity` (token, slot) selections in token order
 * and drops the rest; capacity <= 0 keeps everything. */
static void keep_flags(const int *idx, int T, int E, int k, int capacity, unsigned char *kept)
{
    int *taken = (int *)calloc((size_t)E, sizeof(int));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[(size_t)t * k + j];
            kept[(size_t)t * k + j] = (unsigned char)(capacity <= 0 || taken[e] < capacity);
            taken[e] += 1;
        }
    free(taken);
}

/* Gate actually applied to each slot.  A dropped slot contributes nothing.
 * drop_renorm = 0: its gate mass is lost; 1: the token's kept gates are
 * scaled so they sum to the token's total gate mass (all slots dropped:
 * every gate is 0). */
static void applied_gates(const double *g0, const unsigned char *kept, int k, int drop_renorm,
                          double *g)
{
    double total = 0.0, kept_total = 0.0;
    for (int j = 0; j < k; ++j) {
        total += g0[j];
        if (kept[j])
            kept_total += g0[j];
    }
    for (int j = 0; j < k; ++j) {
        if (!kept[j])
            g[j] = 0.0;
        else if (drop_renorm)
            g[j] = kept_total > 0.0 ? g0[j] * total / kept_total : 0.0;
        else
            g[j] = g0[j];
    }
}

/* ---- whole layer ------------------------------------------------------- */

/*
 * out[t] = sum over kept slots j of g[t][j] * W2[e_j] ( silu(W1[e_j] x_t) * (W3[e_j] x_t) )
 * with e_j the router's selection for token t and g the applied gates.
 *   gating: 0 or 1 (see gates_of); capacity: rows kept per expert (<= 0: all);
 *   drop_renorm: policy for dropped slots (see applied_gates).
 * Optional outputs (pass NULL to skip): logits [T][E] fp32, idx [T][k],
 * gates [T][k] in double (before any drop), and out_exact [T][d]: the
 * weighted sum in double before the one rounding to the element type.
 */
int oracle_moe_forward_ex(const void *x, const void *Wg, const float *bias,
                          const void *const *W1, const void *const *W3,
                          const void *const *W2, int T, int d, int ffn, int E, int k,
                          int dt, int gating, int capacity, int drop_renorm, void *out,
                          float *logits_out, int *idx_out, double *gates_out,
                          double *out_exact, int nthreads)
{
    if (T < 0 || d < 1 || ffn < 1 || E < 1 || k < 1 || k > E ||
        (dt != ORACLE_F32 && dt != ORACLE_BF16) || (gating != 0 && gating != 1))
        return ORACLE_BAD_ARG;
    if (T == 0)
        return ORACLE_OK;
    if (!x || !Wg || !W1 || !W3 || !W2 || !out)
        return ORACLE_BAD_ARG;
    for (int e = 0; e < E; ++e)
        if (!W1[e] || !W3[e] || !W2[e])
            return ORACLE_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    float *L = (float *)malloc(sizeof(float) * (size_t)T * E);
    int *IDX = (int *)malloc(sizeof(int) * (size_t)T * k);
    double *G = (double *)malloc(sizeof(double) * (size_t)T * k);
    unsigned char *KEPT = (unsigned char *)malloc((size_t)T * k);
    if (!L || !IDX || !G || !KEPT) {
        free(L);
        free(IDX);
        free(G);
        free(KEPT);
        return ORACLE_NO_MEM;
    }
    int status = ORACLE_OK;
    /* router, per token */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        float *l = L + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            l[e] = router_logit(x, (size_t)t * d, Wg, bias, d, e, dt);
        if (!all_finite_f32(l, (size_t)E)) {
#pragma omp atomic write
            status = ORACLE_NONFINITE;
        }
        select_top_k(l, E, k, IDX + (size_t)t * k);
        gates_of(l, IDX + (size_t)t * k, E, k, gating, G + (size_t)t * k);
    }
    /* capacity: which selections each expert keeps, in token order */
    keep_flags(IDX, T, E, k, capacity, KEPT);
    /* experts and the weighted sum, per token */
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        double *g = (double *)malloc(sizeof(double) * (size_t)k);
        double *h = (double *)malloc(sizeof(double) * (size_t)ffn);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        if (!g || !h || !acc) {
#pragma omp atomic write
            status = ORACLE_NO_MEM;
        } else {
            size_t xo = (size_t)t * d;
            const int *chosen = IDX + (size_t)t * k;
            applied_gates(G + (size_t)t * k, KEPT + (size_t)t * k, k, drop_renorm, g);
            for (int n = 0; n < d; ++n)
                acc[n] = 0.0;
            for (int j = 0; j < k; ++j) {
                if (!KEPT[(size_t)t * k + j])
                    continue;
                int e = chosen[j];
                /* gate and up projections, then the SwiGLU product */
                for (int c = 0; c < ffn; ++c) {
                    double u = 0.0, v = 0.0;
                    size_t wo = (size_t)c * d;
                    for (int i = 0; i < d; ++i) {
                        double xi = elem(x, xo + (size_t)i, dt);
                        u += xi * elem(W1[e], wo + (size_t)i, dt);
                        v += xi * elem(W3[e], wo + (size_t)i, dt);
                    }
                    h[c] = u / (1.0 + exp(-u)) * v;
                }
                /* down projection, weighted by this expert's gate */
                for (int n = 0; n < d; ++n) {
                    double y = 0.0;
                    size_t wo = (size_t)n * ffn;
                    for (int c = 0; c < ffn; ++c)
                        y += elem(W2[e], wo + (size_t)c, dt) * h[c];
                    acc[n] += g[j] * y;
                }
            }
            for (int n = 0; n < d; ++n)
                store_elem(out, xo + (size_t)n, dt, acc[n]);
            if (out_exact)
                for (int n = 0; n < d; ++n)
                    out_exact[xo + (size_t)n] = acc[n];
        }
        free(g);
        free(h);
        free(acc);
    }
    if (logits_out)
        memcpy(logits_out, L, sizeof(float) * (size_t)T * E);
    if (idx_out)
        memcpy(idx_out, IDX, sizeof(int) * (size_t)T * k);
    if (gates_out)
        memcpy(gates_out, G, sizeof(double) * (size_t)T * k);
    free(L);
    free(IDX);
    free(G);
    free(KEPT);
    return status;
}

/* The layer as the azimuth.plus router paragraph states it: gating 0, no
 * capacity limit. */
int oracle_moe_forward(const void *x, const void *Wg, const float *bias,
                       const void *const *W1, const void *const *W3,
                       const void *const *W2, int T, int d, int ffn, int E, int k,
                       int dt, void *out, float *logits_out, int *idx_out,
                       double *gates_out, double *out_exact, int nthreads)
{
    return oracle_moe_forward_ex(x, Wg, bias, W1, W3, W2, T, d, ffn, E, k, dt, 0, 0, 0, out,
                                 logits_out, idx_out, gates_out, out_exact, nthreads);
}

/* Router alone: logits (fp32), selection and gates, for every token. */
int oracle_router(const void *x, const void *Wg, const float *bias, int T, int d,
                  int E, int k, int dt, int gating, float *logits_out, int *idx_out,
                  double *gates_out)
{
    if (T < 0 || d < 1 || E < 1 || k < 1 || k > E || !logits_out || !idx_out || !gates_out ||
        (gating != 0 && gating != 1))
        return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        float *l = logits_out + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            l[e] = router_logit(x, (size_t)t * d, Wg, bias, d, e, dt);
        if (!all_finite_f32(l, (size_t)E)) {
#pragma omp atomic write
            status = ORACLE_NONFINITE;
        }
        select_top_k(l, E, k, idx_out + (size_t)t * k);
        gates_of(l, idx_out + (size_t)t * k, E, k, gating, gates_out + (size_t)t * k);
    }
    return status;
}

/*
 * Grouping tokens by expert, from given fp32 logits.  Selection and gates as
 * in the router; capacity as in keep_flags; then, over kept selections only,
 *   counts[e]  = number of (token, slot) pairs expert e keeps,
 *   offsets    = exclusive prefix sum of counts, offsets[E] = sum of counts,
 *   rows ordered by (expert, token) ascending: row r holds perm[r] = t*k + j,
 *   inv[t*k + j] = r, or -1 for a dropped selection.
 */
int oracle_route(const float *logits, int T, int E, int k, int gating, int capacity,
                 int *idx_out, double *gates_out, int *counts, int *offsets, int *perm,
                 int *inv)
{
    if (T < 0 || E < 1 || k < 1 || k > E || !idx_out || !gates_out || !counts ||
        !offsets || !perm || !inv || (gating != 0 && gating != 1))
        return ORACLE_BAD_ARG;
    if (!all_finite_f32(logits, (size_t)T * E))
        return ORACLE_NONFINITE;
    for (int t = 0; t < T; ++t) {
        select_top_k(logits + (size_t)t * E, E, k, idx_out + (size_t)t * k);
        gates_of(logits + (size_t)t * E, idx_out + (size_t)t * k, E, k, gating,
                 gates_out + (size_t)t * k);
    }
    unsigned char *kept = (unsigned char *)malloc((size_t)T * k + 1);
    if (!kept)
        return ORACLE_NO_MEM;
    keep_flags(idx_out, T, E, k, capacity, kept);
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (size_t s = 0; s < (size_t)T * k; ++s)
        if (kept[s])
            counts[idx_out[s]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int r = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (idx_out[(size_t)t * k + j] == e) {
                    if (!kept[(size_t)t * k + j]) {
                        inv[(size_t)t * k + j] = -1;
                        continue;
                    }
                    perm[r] = t * k + j;
                    inv[(size_t)t * k + j] = r;
                    ++r;
                }
    free(kept);
    return ORACLE_OK;
}

/* RMSNorm with gain 1: y = x / sqrt(mean(x^2) + eps), rounded to the element
 * type.  Used between stacked layers (a Mistral decoder block normalises the
 * input of its feed-forward sub-block). */
int oracle_rmsnorm(const void *x, int T, int d, double eps, int dt, void *y)
{
    if (T < 0 || d < 1 || !x || !y)
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        size_t o = (size_t)t * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) {
            double v = elem(x, o + (size_t)i, dt);
            ss += v * v;
        }
        double scale = 1.0 / sqrt(ss / d + eps);
        for (int i = 0; i < d; ++i)
            store_elem(y, o + (size_t)i, dt, elem(x, o + (size_t)i, dt) * scale);
    }
    return ORACLE_OK;
}

/* Residual update: z = a + b, rounded once to the element type. */
int oracle_add(const void *a, const void *b, size_t n, int dt, void *z)
{
    if (!a || !b || !z)
        return ORACLE_BAD_ARG;
    for (size_t i = 0; i < n; ++i)
        store_elem(z, i, dt, elem(a, i, dt) + elem(b, i, dt));
    return ORACLE_OK;
}

/* ---- backward (training) ------------------------------------------------ */

/* Logistic function and the derivative of silu(u) = u s(u):
 * silu'(u) = s(u) + u s(u) (1 - s(u)). */
static double logistic(double u) { return 1.0 / (1.0 + exp(-u)); }

/*
 * Gradients of L = sum_t <dout[t], out[t]> (dout: the upstream gradient of the
 * layer output) for the layer with gating 0 and no capacity limit, by the
 * chain rule through the forward's steps, in double, term by term.  Which
 * experts a token picks is piecewise constant in the inputs, so no gradient
 * flows through the selection; the fp32 rounding of the logits is taken as
 * the identity.  For token t and each slot j (expert e = e_j, gate g_j):
 *   u = W1[e] x,  v = W3[e] x,  h = silu(u) * v,  y_j = W2[e] h      (forward)
 *   dy_j = g_j dout[t]                                (weighted sum)
 *   dg_j = <dout[t], y_j>
 *   dh   = W2[e]^T dy_j,              dW2[e] += dy_j h^T
 *   du   = dh * v * silu'(u),  dv = dh * silu(u)      (SwiGLU product)
 *   dW1[e] += du x^T,  dW3[e] += dv x^T,  dx[t] += W1[e]^T du + W3[e]^T dv
 *   dl_j = g_j (dg_j - sum_m g_m dg_m)                (softmax over the kept)
 *   dW_g[e_j] += dl_j x,  dx[t] += sum_j dl_j W_g[e_j]
 * Outputs (double, any may be NULL): dx [T][d], dWg [E][d], and per expert
 * dW1[e], dW3[e] rows [c0, c1) of [ffn][d] (stored [c1-c0][d]) and dW2[e]
 * rows [n0, n1) of [d][ffn] (stored [n1-n0][ffn]).  Every weight-gradient
 * element sums its terms in token order, then slot order.
 */
int oracle_moe_backward(const void *x, const void *Wg, const float *bias,
                        const void *const *W1, const void *const *W3, const void *const *W2,
                        int T, int d, int ffn, int E, int k, int dt, const void *dout,
                        double *dx, double *dWg, double *const *dW1, double *const *dW3,
                        double *const *dW2, int c0, int c1, int n0, int n1, int nthreads)
{
    if (T < 0 || d < 1 || ffn < 1 || E < 1 || k < 1 || k > E ||
        (dt != ORACLE_F32 && dt != ORACLE_BF16) || c0 < 0 || c1 > ffn || c0 > c1 || n0 < 0 ||
        n1 > d || n0 > n1)
        return ORACLE_BAD_ARG;
    if (T == 0)
        return ORACLE_OK;
    if (!x || !Wg || !W1 || !W3 || !W2 || !dout)
        return ORACLE_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const size_t S = (size_t)T * k; /* (token, slot) pairs */
    int *IDX = (int *)malloc(sizeof(int) * S);
    double *G = (double *)malloc(sizeof(double) * S);
    double *DL = (double *)malloc(sizeof(double) * S);
    double *H = (double *)malloc(sizeof(double) * S * ffn);
    double *DU = (double *)malloc(sizeof(double) * S * ffn);
    double *DV = (double *)malloc(sizeof(double) * S * ffn);
    double *DY = (double *)malloc(sizeof(double) * S * d);
    if (!IDX || !G || !DL || !H || !DU || !DV || !DY) {
        free(IDX); free(G); free(DL); free(H); free(DU); free(DV); free(DY);
        return ORACLE_NO_MEM;
    }
    int status = ORACLE_OK;
    /* phase 1, per token: forward again, then the backward down to the
     * per-slot vectors and the token's input gradient */
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        float *l = (float *)malloc(sizeof(float) * (size_t)E);
        double *u = (double *)malloc(sizeof(double) * (size_t)ffn);
        double *v = (double *)malloc(sizeof(double) * (size_t)ffn);
        double *dg = (double *)malloc(sizeof(double) * (size_t)k);
        if (!l || !u || !v || !dg) {
#pragma omp atomic write
            status = ORACLE_NO_MEM;
            free(l); free(u); free(v); free(dg);
            continue;
        }
        const size_t xo = (size_t)t * d;
        for (int e = 0; e < E; ++e)
            l[e] = router_logit(x, xo, Wg, bias, d, e, dt);
        if (!all_finite_f32(l, (size_t)E)) {
#pragma omp atomic write
            status = ORACLE_NONFINITE;
        }
        int *chosen = IDX + (size_t)t * k;
        double *g = G + (size_t)t * k;
        select_top_k(l, E, k, chosen);
        gates_of(l, chosen, E, k, 0, g);
        for (int i = 0; i < d; ++i)
            if (dx)
                dx[xo + (size_t)i] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int e = chosen[j];
            const size_t sj = (size_t)t * k + j;
            double *h = H + sj * ffn, *du = DU + sj * ffn, *dv = DV + sj * ffn;
            double *dy = DY + sj * d;
            for (int c = 0; c < ffn; ++c) {
                double uu = 0.0, vv = 0.0;
                for (int i = 0; i < d; ++i) {
                    double xi = elem(x, xo + (size_t)i, dt);
                    uu += xi * elem(W1[e], (size_t)c * d + i, dt);
                    vv += xi * elem(W3[e], (size_t)c * d + i, dt);
                }
                u[c] = uu;
                v[c] = vv;
                h[c] = uu * logistic(uu) * vv;
            }
            /* y_j . dout and dy_j */
            double dgj = 0.0;
            for (int n = 0; n < d; ++n) {
                double y = 0.0;
                for (int c = 0; c < ffn; ++c)
                    y += elem(W2[e], (size_t)n * ffn + c, dt) * h[c];
                double o = elem(dout, xo + (size_t)n, dt);
                dgj += o * y;
                dy[n] = g[j] * o;
            }
            dg[j] = dgj;
            /* dh = W2^T dy, then through the SwiGLU product */
            for (int c = 0; c < ffn; ++c) {
                double dh = 0.0;
                for (int n = 0; n < d; ++n)
                    dh += elem(W2[e], (size_t)n * ffn + c, dt) * dy[n];
                double s = logistic(u[c]);
                du[c] = dh * v[c] * (s + u[c] * s * (1.0 - s));
                dv[c] = dh * u[c] * s;
            }
            if (dx)
                for (int i = 0; i < d; ++i) {
                    double acc = 0.0;
                    for (int c = 0; c < ffn; ++c)
                        acc += elem(W1[e], (size_t)c * d + i, dt) * du[c] +
                               elem(W3[e], (size_t)c * d + i, dt) * dv[c];
                    dx[xo + (size_t)i] += acc;
                }
        }
        /* softmax over the kept logits */
        double gdg = 0.0;
        for (int j = 0; j < k; ++j)
            gdg += g[j] * dg[j];
        for (int j = 0; j < k; ++j)
            DL[(size_t)t * k + j] = g[j] * (dg[j] - gdg);
        if (dx)
            for (int j = 0; j < k; ++j)
                for (int i = 0; i < d; ++i)
                    dx[xo + (size_t)i] +=
                        DL[(size_t)t * k + j] * elem(Wg, (size_t)chosen[j] * d + i, dt);
        free(l); free(u); free(v); free(dg);
    }
    /* phase 2, per weight-gradient row: sums over tokens in token order */
    if (dWg) {
#pragma omp parallel for schedule(static)
        for (int e = 0; e < E; ++e)
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (size_t s = 0; s < S; ++s)
                    if (IDX[s] == e)
                        acc += DL[s] * elem(x, (s / (size_t)k) * d + (size_t)i, dt);
                dWg[(size_t)e * d + i] = acc;
            }
    }
    if (dW1 || dW3) {
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
        for (int e = 0; e < E; ++e)
            for (int c = c0; c < c1; ++c)
                for (int i = 0; i < d; ++i) {
                    double a1 = 0.0, a3 = 0.0;
                    for (size_t s = 0; s < S; ++s) {
                        if (IDX[s] != e)
                            continue;
                        double xi = elem(x, (s / (size_t)k) * d + (size_t)i, dt);
                        a1 += DU[s * ffn + c] * xi;
                        a3 += DV[s * ffn + c] * xi;
                    }
                    if (dW1 && dW1[e])
                        dW1[e][(size_t)(c - c0) * d + i] = a1;
                    if (dW3 && dW3[e])
                        dW3[e][(size_t)(c - c0) * d + i] = a3;
                }
    }
    if (dW2) {
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
        for (int e = 0; e < E; ++e)
            for (int n = n0; n < n1; ++n)
                for (int c = 0; c < ffn; ++c) {
                    double a = 0.0;
                    for (size_t s = 0; s < S; ++s)
                        if (IDX[s] == e)
                            a += DY[s * d + n] * H[s * ffn + c];
                    if (dW2[e])
                        dW2[e][(size_t)(n - n0) * ffn + c] = a;
                }
    }
    free(IDX); free(G); free(DL); free(H); free(DU); free(DV); free(DY);
    return status;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
