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
 *   - RMSNorm (for the stacked-layer harness) uses gain 1.
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

/* Softmax over the kept logits only (every other score is -inf, so it
 * contributes exp(-inf) = 0).  The largest kept logit is subtracted first. */
static void gates_of(const float *l, const int *chosen, int k, double *g)
{
    double l0 = (double)l[chosen[0]];
    double z = 0.0;
    for (int j = 0; j < k; ++j)
        z += exp((double)l[chosen[j]] - l0);
    for (int j = 0; j < k; ++j)
        g[j] = exp((double)l[chosen[j]] - l0) / z;
}

static int all_finite_f32(const float *p, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        if (!isfinite(p[i]))
            return 0;
    return 1;
}

/* ---- whole layer ------------------------------------------------------- */

/*
 * out[t] = sum_j g[t][j] * W2[e_j] ( silu(W1[e_j] x_t) * (W3[e_j] x_t) )
 * with e_j and g the router's selection and gates for token t.
 * Optional outputs (pass NULL to skip): logits [T][E] fp32, idx [T][k],
 * gates [T][k] in double, and out_exact [T][d]: the weighted sum in double
 * before the one rounding to the element type.
 */
int oracle_moe_forward(const void *x, const void *Wg, const float *bias,
                       const void *const *W1, const void *const *W3,
                       const void *const *W2, int T, int d, int ffn, int E, int k,
                       int dt, void *out, float *logits_out, int *idx_out,
                       double *gates_out, double *out_exact, int nthreads)
{
    if (T < 0 || d < 1 || ffn < 1 || E < 1 || k < 1 || k > E ||
        (dt != ORACLE_F32 && dt != ORACLE_BF16))
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
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        float *l = (float *)malloc(sizeof(float) * (size_t)E);
        int *chosen = (int *)malloc(sizeof(int) * (size_t)k);
        double *g = (double *)malloc(sizeof(double) * (size_t)k);
        double *h = (double *)malloc(sizeof(double) * (size_t)ffn);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        if (!l || !chosen || !g || !h || !acc) {
#pragma omp atomic write
            status = ORACLE_NO_MEM;
        } else {
            size_t xo = (size_t)t * d;
            for (int e = 0; e < E; ++e)
                l[e] = router_logit(x, xo, Wg, bias, d, e, dt);
            if (!all_finite_f32(l, (size_t)E)) {
#pragma omp atomic write
                status = ORACLE_NONFINITE;
            }
            select_top_k(l, E, k, chosen);
            gates_of(l, chosen, k, g);
            for (int n = 0; n < d; ++n)
                acc[n] = 0.0;
            for (int j = 0; j < k; ++j) {
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
            if (logits_out)
                for (int e = 0; e < E; ++e)
                    logits_out[(size_t)t * E + e] = l[e];
            for (int j = 0; j < k; ++j) {
                if (idx_out)
                    idx_out[(size_t)t * k + j] = chosen[j];
                if (gates_out)
                    gates_out[(size_t)t * k + j] = g[j];
            }
        }
        free(l);
        free(chosen);
        free(g);
        free(h);
        free(acc);
    }
    return status;
}

/* Router alone: logits (fp32), selection and gates, for every token. */
int oracle_router(const void *x, const void *Wg, const float *bias, int T, int d,
                  int E, int k, int dt, float *logits_out, int *idx_out,
                  double *gates_out)
{
    if (T < 0 || d < 1 || E < 1 || k < 1 || k > E || !logits_out || !idx_out || !gates_out)
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
        gates_of(l, idx_out + (size_t)t * k, k, gates_out + (size_t)t * k);
    }
    return status;
}

/*
 * Grouping tokens by expert, from given fp32 logits.  Selection and gates as
 * in the router; then
 *   counts[e]  = number of (token, slot) pairs routed to e,
 *   offsets    = exclusive prefix sum of counts, offsets[E] = T*k,
 *   rows ordered by (expert, token) ascending: row r holds perm[r] = t*k + j,
 *   inv[t*k + j] = r.
 */
int oracle_route(const float *logits, int T, int E, int k, int *idx_out,
                 double *gates_out, int *counts, int *offsets, int *perm, int *inv)
{
    if (T < 0 || E < 1 || k < 1 || k > E || !idx_out || !gates_out || !counts ||
        !offsets || !perm || !inv)
        return ORACLE_BAD_ARG;
    if (!all_finite_f32(logits, (size_t)T * E))
        return ORACLE_NONFINITE;
    for (int t = 0; t < T; ++t) {
        select_top_k(logits + (size_t)t * E, E, k, idx_out + (size_t)t * k);
        gates_of(logits + (size_t)t * E, idx_out + (size_t)t * k, k,
                 gates_out + (size_t)t * k);
    }
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (size_t s = 0; s < (size_t)T * k; ++s)
        counts[idx_out[s]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int r = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (idx_out[(size_t)t * k + j] == e) {
                    perm[r] = t * k + j;
                    inv[(size_t)t * k + j] = r;
                    ++r;
                }
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

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
