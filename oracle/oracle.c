/*
 * oracle.c - plain, slow, sequential CPU oracle for batched draft
 * verification by lossless rejection sampling, and for D-cut's batch-level
 * allocation of verification depth.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this library.  The product path (the
 * CUDA kernels behind include/specverify.h) shares no code, header, table or
 * helper with it, and never calls it.
 *
 * Everything is computed in fp64 from the exact input values (bf16 -> fp32 is
 * exact; fp32 -> fp64 is exact), one request and one vocabulary entry at a
 * time, in the order the definitions state.  No blocking, fusion or
 * reordering.
 *
 * Sources:
 *  - What the path computes: "Tencent Hunyuan Turns Speculative Decoding Into
 *    a Full Open-Source Stack", section "What problem does it solve": the
 *    target checks the whole drafted block in one forward pass by rejection
 *    sampling and commits the accepted prefix plus one bonus token.
 *  - Accepted length = drafted tokens approved before the first mismatch:
 *    "Tencent rilascia AngelSpec in open source ...", section "Come AngelSpec
 *    rende DFly piu selettivo".
 *  - Losslessness (output law = target law): "Tencent ... AngelSpec ...",
 *    section "Qu'est-ce que le speculative decoding"; and the Italian page,
 *    section "Cosa non dimostrano i numeri di AngelSpec" (a correct
 *    accept/reject algorithm is required).
 *  - Greedy operation at T = 0: the French/Russian page's bullet list (rates
 *    quoted at T = 0).
 *  - The pages never write the accept/reject formulas down.  They are the
 *    standard ones: accept drafted x with probability min(1, p(x)/q(x));
 *    after a rejection sample from norm(max(0, p - q)); when every draft is
 *    accepted sample one more token from the next target distribution.
 *    Leviathan, Kalman & Matias 2023, "Fast Inference from Transformers via
 *    Speculative Decoding", section "Speculative Sampling"; Chen et al. 2023,
 *    "Accelerating Large Language Model Decoding with Speculative Sampling",
 *    "modified rejection sampling".
 *  - D-cut: the Italian page, section "Come AngelSpec rende DFly piu
 *    selettivo" (verification capacity as a batch-level shared resource; the
 *    expected value of keeping more positions weighed against cost; more
 *    depth to high-confidence prefixes) and the English page 5, "What problem
 *    does it solve", inference layer (depth per request from prefix
 *    confidence under load).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  accept iff u < p/q strictly (u in [0,1)); q(x) = 0 accepts iff p(x) > 0;
 *  an all-zero residual falls back to p; inverse CDF = smallest v with
 *  C(v) > u*S, falling back to the last v with w(v) > 0; greedy ties go to the
 *  lowest index; the temperature divides the logits of both target and draft
 *  rows; D-cut keeps the globally best `budget` prefix products P >= min_gain,
 *  ties broken by (request, depth) ascending.
 *
 * Parity pins: tests/test_oracle_pins.py checks every function here against
 * closed forms, library routines, brute force and chi-square losslessness.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_INVALID_ARG (-1)
#define ORC_ERR_NONFINITE (-4)

#define ORC_F32 0
#define ORC_BF16 1

/* Largest number of drafted tokens one request may verify. */
#define ORC_MAX_DRAFT 32

/* ------------------------------------------------------------------------ */
/* input access                                                              */
/* ------------------------------------------------------------------------ */

/* Exact value of one logit.  bf16 is the upper half of an IEEE fp32 word. */
static double logit_at(const void *base, int dtype, int64_t row, int64_t V, int64_t v)
{
    int64_t idx = row * V + v;
    if (dtype == ORC_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* NaN and +inf are errors; -inf (a masked vocabulary entry) is allowed. */
static int bad_value(double x)
{
    return isnan(x) || (isinf(x) && x > 0);
}

/* ------------------------------------------------------------------------ */
/* softmax with temperature                                                  */
/* ------------------------------------------------------------------------ */

/*
 * m = max_v l_v and s = sum_v exp((l_v - m) / T) over one row.
 * p(v) = exp((l_v - m) / T) / s is the temperature softmax.
 */
int oracle_softmax_stats(const void *logits, int dtype, int64_t row, int64_t V, double T,
                         double *m_out, double *s_out)
{
    if (V <= 0 || !(T > 0))
        return ORC_ERR_INVALID_ARG;
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, row, V, v);
        if (bad_value(l))
            return ORC_ERR_NONFINITE;
        if (l > m)
            m = l;
    }
    if (isinf(m))
        return ORC_ERR_NONFINITE; /* every entry masked */
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, row, V, v);
        s += exp((l - m) / T);
    }
    *m_out = m;
    *s_out = s;
    return ORC_OK;
}

/* p(v) for every v of one row. */
int oracle_softmax_row(const void *logits, int dtype, int64_t row, int64_t V, double T,
                       double *p_out)
{
    double m, s;
    int st = oracle_softmax_stats(logits, dtype, row, V, T, &m, &s);
    if (st != ORC_OK)
        return st;
    for (int64_t v = 0; v < V; ++v)
        p_out[v] = exp((logit_at(logits, dtype, row, V, v) - m) / T) / s;
    return ORC_OK;
}

/* p(x) for one entry x of one row. */
static int softmax_at(const void *logits, int dtype, int64_t row, int64_t V, double T,
                      int64_t x, double *p_out)
{
    double m, s;
    int st = oracle_softmax_stats(logits, dtype, row, V, T, &m, &s);
    if (st != ORC_OK)
        return st;
    *p_out = exp((logit_at(logits, dtype, row, V, x) - m) / T) / s;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* greedy argmax (T = 0)                                                     */
/* ------------------------------------------------------------------------ */

/* Lowest index attaining the row maximum. */
int oracle_argmax_row(const void *logits, int dtype, int64_t row, int64_t V, int32_t *idx_out)
{
    if (V <= 0)
        return ORC_ERR_INVALID_ARG;
    double best = -INFINITY;
    int64_t arg = -1;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, row, V, v);
        if (bad_value(l))
            return ORC_ERR_NONFINITE;
        if (l > best) { /* strict: an equal later value never replaces */
            best = l;
            arg = v;
        }
    }
    if (arg < 0)
        return ORC_ERR_NONFINITE; /* every entry masked */
    *idx_out = (int32_t)arg;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* inverse CDF                                                               */
/* ------------------------------------------------------------------------ */

/*
 * Given non-negative weights w[0..V) with S = sum w > 0 and u in [0,1):
 * the smallest v with C(v) > u*S, C the running sum of w in index order.
 * If rounding leaves no such v, the last v with w(v) > 0.
 * Returns -1 when S == 0.
 */
int64_t oracle_inverse_cdf(const double *w, int64_t V, double u, double *uS_out,
                           double *S_out)
{
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v)
        S += w[v];
    if (uS_out)
        *uS_out = u * S;
    if (S_out)
        *S_out = S;
    if (!(S > 0))
        return -1;
    double target = u * S;
    double C = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        C += w[v];
        if (C > target)
            return v;
    }
    for (int64_t v = V - 1; v >= 0; --v)
        if (w[v] > 0)
            return v;
    return -1;
}

/* ------------------------------------------------------------------------ */
/* verification                                                              */
/* ------------------------------------------------------------------------ */

static int64_t draft_index(const int32_t *cu, int32_t i, int32_t j, int32_t draft_stride)
{
    return draft_stride > 0 ? (int64_t)i * draft_stride + j : (int64_t)cu[i] + j;
}

static int64_t target_row(const int32_t *cu, int32_t i, int32_t j)
{
    return (int64_t)cu[i] + i + j;
}

/* cu[0] = 0, non-decreasing, every depth at most ORC_MAX_DRAFT (and at most
 * draft_stride when the draft side is padded). */
static int check_offsets(const int32_t *cu, int32_t B, int32_t draft_stride)
{
    if (cu[0] != 0)
        return ORC_ERR_INVALID_ARG;
    for (int32_t i = 0; i < B; ++i) {
        int32_t k = cu[i + 1] - cu[i];
        if (k < 0 || k > ORC_MAX_DRAFT || (draft_stride > 0 && k > draft_stride))
            return ORC_ERR_INVALID_ARG;
    }
    return ORC_OK;
}

static void poison_request(const int32_t *cu, int32_t i, int32_t *out_tokens,
                           int32_t *out_accept_len)
{
    int32_t k = cu[i + 1] - cu[i];
    for (int32_t j = 0; j <= k; ++j)
        out_tokens[target_row(cu, i, j)] = -1;
    out_accept_len[i] = -1;
}

/* Emitted row for request i: the accepted prefix x_0..x_{a-1}, then y at
 * position a, then -1 up to the bonus position. */
static void emit(const int32_t *cu, int32_t i, int32_t draft_stride, const int32_t *tokens,
                 int32_t a, int32_t y, int32_t *out_tokens, int32_t *out_accept_len)
{
    int32_t k = cu[i + 1] - cu[i];
    for (int32_t j = 0; j <= k; ++j) {
        int32_t t = -1;
        if (j < a)
            t = tokens[draft_index(cu, i, j, draft_stride)];
        else if (j == a)
            t = y;
        out_tokens[target_row(cu, i, j)] = t;
    }
    out_accept_len[i] = a;
}

/*
 * Greedy verification (T = 0).  Target row j's choice g_j is its argmax.
 * Every row of a request is read, so a non-finite value in any of them is an
 * error even past the first mismatch.
 * Draft j is accepted iff x_j == g_j; a = first mismatch (or K).  Emitted:
 * x_0..x_{a-1}, then g_a (the bonus row's argmax when a = K).
 * Returns the first error met; a failing request gets -1 outputs.
 */
int oracle_verify_greedy(const void *target, int dtype, const int32_t *tokens,
                         const int32_t *cu, int32_t B, int64_t V, int32_t draft_stride,
                         int32_t *out_tokens, int32_t *out_accept_len)
{
    if (B < 0 || V <= 0 || V > INT32_MAX || draft_stride < 0 ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_ERR_INVALID_ARG;
    if (B == 0)
        return ORC_OK;
    int st = check_offsets(cu, B, draft_stride);
    if (st != ORC_OK)
        return st;
    int first_err = ORC_OK;
    for (int32_t i = 0; i < B; ++i) {
        int32_t k = cu[i + 1] - cu[i];
        int err = ORC_OK;
        for (int32_t j = 0; j < k && err == ORC_OK; ++j) {
            int32_t x = tokens[draft_index(cu, i, j, draft_stride)];
            if (x < 0 || x >= V)
                err = ORC_ERR_INVALID_ARG;
        }
        /* every row of the request is read: g_0..g_K first, then the match */
        int32_t g[ORC_MAX_DRAFT + 1] = {0};
        for (int32_t j = 0; j <= k && err == ORC_OK; ++j)
            err = oracle_argmax_row(target, dtype, target_row(cu, i, j), V, &g[j]);
        int32_t a = k, y = -1;
        if (err == ORC_OK) {
            a = 0;
            while (a < k && tokens[draft_index(cu, i, a, draft_stride)] == g[a])
                ++a;
            y = g[a];
        }
        if (err != ORC_OK) {
            poison_request(cu, i, out_tokens, out_accept_len);
            if (first_err == ORC_OK)
                first_err = err;
            continue;
        }
        emit(cu, i, draft_stride, tokens, a, y, out_tokens, out_accept_len);
    }
    return first_err;
}

/*
 * Weights of the final draw for one request.
 *  rejection at position a (draft_row >= 0): w(v) = max(0, p(v) - q(v)),
 *    p from target row a, q from draft row a; if every w(v) is 0 the residual
 *    is undefined and w = p instead (*fallback = 1);
 *  every draft accepted (draft_row < 0): w = p of the bonus row.
 */
int oracle_final_weights(const void *target, const void *draft, int dtype, int64_t V,
                         double T, int64_t trow, int64_t drow, double *w_out,
                         int32_t *fallback)
{
    int st = oracle_softmax_row(target, dtype, trow, V, T, w_out);
    if (st != ORC_OK)
        return st;
    if (fallback)
        *fallback = 0;
    if (drow < 0)
        return ORC_OK;
    double *q = (double *)malloc((size_t)V * sizeof(double));
    if (!q)
        return ORC_ERR_INVALID_ARG;
    st = oracle_softmax_row(draft, dtype, drow, V, T, q);
    if (st != ORC_OK) {
        free(q);
        return st;
    }
    int any = 0;
    for (int64_t v = 0; v < V; ++v) {
        double r = w_out[v] - q[v];
        if (r > 0)
            any = 1;
    }
    if (any) {
        for (int64_t v = 0; v < V; ++v) {
            double r = w_out[v] - q[v];
            w_out[v] = r > 0 ? r : 0.0;
        }
    } else if (fallback) {
        *fallback = 1; /* w keeps p */
    }
    free(q);
    return ORC_OK;
}

/*
 * Sampling verification (T > 0).  For drafted x_j (j < K):
 *   p_j = p_{target row j}(x_j), q_j = q_{draft row j}(x_j),
 *   accept_j iff u_j < p_j / q_j   (q_j = 0: accept iff p_j > 0).
 * a = first rejected position (K if none).  The final token y is the inverse
 * CDF of the weights from oracle_final_weights at u_final.  Emitted:
 * x_0..x_{a-1}, y.
 *
 * out_p/out_q (draft index, float) hold p_j and q_j for every j < K.
 * Optional diagnostics: out_ratio[draft index] = p_j/q_j (+inf when q_j = 0
 * and p_j > 0); out_final[4*i..] = {u*S, S, C(y-1), C(y)} of the final draw.
 * Every row of a request (including the bonus row after an early rejection)
 * is read: a non-finite value in any of them is an error.
 * T == 0 runs the greedy verification.  Returns the first error met.
 */
int oracle_verify_sample(const void *target, const void *draft, int dtype,
                         const int32_t *tokens, const int32_t *cu, int32_t B, int64_t V,
                         int32_t draft_stride, double T, const float *u_accept,
                         const float *u_final, int32_t *out_tokens,
                         int32_t *out_accept_len, float *out_p, float *out_q,
                         double *out_ratio, double *out_final)
{
    if (T == 0.0)
        return oracle_verify_greedy(target, dtype, tokens, cu, B, V, draft_stride,
                                    out_tokens, out_accept_len);
    if (!(T > 0) || isinf(T) || B < 0 || V <= 0 || V > INT32_MAX || draft_stride < 0 ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_ERR_INVALID_ARG;
    if (B == 0)
        return ORC_OK;
    int st = check_offsets(cu, B, draft_stride);
    if (st != ORC_OK)
        return st;
    double *w = (double *)malloc((size_t)V * sizeof(double));
    if (!w)
        return ORC_ERR_INVALID_ARG;
    int first_err = ORC_OK;
    for (int32_t i = 0; i < B; ++i) {
        int32_t k = cu[i + 1] - cu[i];
        int err = ORC_OK;
        int32_t a = k;
        for (int32_t j = 0; j < k && err == ORC_OK; ++j) {
            int64_t di = draft_index(cu, i, j, draft_stride);
            int32_t x = tokens[di];
            if (x < 0 || x >= V) {
                err = ORC_ERR_INVALID_ARG;
                break;
            }
            double p, q;
            err = softmax_at(target, dtype, target_row(cu, i, j), V, T, x, &p);
            if (err == ORC_OK)
                err = softmax_at(draft, dtype, di, V, T, x, &q);
            if (err != ORC_OK)
                break;
            double ratio;
            if (q > 0)
                ratio = p / q;
            else
                ratio = p > 0 ? INFINITY : 0.0;
            int accept = (double)u_accept[di] < ratio;
            if (out_p)
                out_p[di] = (float)p;
            if (out_q)
                out_q[di] = (float)q;
            if (out_ratio)
                out_ratio[di] = ratio;
            if (!accept && a == k)
                a = j;
        }
        if (err == ORC_OK) { /* the bonus row is read even when a < K */
            double mb, sb;
            err = oracle_softmax_stats(target, dtype, target_row(cu, i, k), V, T, &mb, &sb);
        }
        int32_t y = -1;
        if (err == ORC_OK) {
            int64_t drow = a < k ? draft_index(cu, i, a, draft_stride) : -1;
            err = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a), drow,
                                       w, NULL);
            if (err == ORC_OK) {
                double uS, S;
                int64_t v = oracle_inverse_cdf(w, V, (double)u_final[i], &uS, &S);
                if (v < 0)
                    err = ORC_ERR_NONFINITE;
                else {
                    y = (int32_t)v;
                    if (out_final) {
                        double C = 0.0;
                        for (int64_t t = 0; t < v; ++t)
                            C += w[t];
                        out_final[4 * (int64_t)i + 0] = uS;
                        out_final[4 * (int64_t)i + 1] = S;
                        out_final[4 * (int64_t)i + 2] = C;
                        out_final[4 * (int64_t)i + 3] = C + w[v];
                    }
                }
            }
        }
        if (err != ORC_OK) {
            poison_request(cu, i, out_tokens, out_accept_len);
            if (first_err == ORC_OK)
                first_err = err;
            continue;
        }
        emit(cu, i, draft_stride, tokens, a, y, out_tokens, out_accept_len);
    }
    free(w);
    return first_err;
}

/*
 * Running sum C of the final-draw weights of request i, given its accepted
 * length a (test helper: decides the inverse-CDF exemption at any index).
 */
int oracle_final_cdf(const void *target, const void *draft, int dtype, const int32_t *cu,
                     int32_t i, int64_t V, int32_t draft_stride, double T, int32_t a,
                     double *cdf_out)
{
    int32_t k = cu[i + 1] - cu[i];
    if (a < 0 || a > k || !(T > 0))
        return ORC_ERR_INVALID_ARG;
    int64_t drow = a < k ? draft_index(cu, i, a, draft_stride) : -1;
    int st = oracle_final_weights(target, draft, dtype, V, T, target_row(cu, i, a), drow,
                                  cdf_out, NULL);
    if (st != ORC_OK)
        return st;
    double C = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        C += cdf_out[v];
        cdf_out[v] = C;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* D-cut                                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    float P;   /* prefix product of confidences through depth d */
    int32_t i; /* request */
    int32_t d; /* depth, 1..kmax[i] */
} dcut_cand;

/* Order: larger P first; equal P -> lower request, then lower depth. */
static int dcut_cmp(const void *pa, const void *pb)
{
    const dcut_cand *a = (const dcut_cand *)pa, *b = (const dcut_cand *)pb;
    if (a->P > b->P)
        return -1;
    if (a->P < b->P)
        return 1;
    if (a->i != b->i)
        return a->i < b->i ? -1 : 1;
    if (a->d != b->d)
        return a->d < b->d ? -1 : 1;
    return 0;
}

/*
 * D-cut allocation in verify-token units.
 * conf[i*Kmax + j] in [0,1] is request i's confidence in its drafted token j
 * (j < kmax[i]).  P_{i,d} = prod_{j<d} conf[i][j], multiplied in fp32 left
 * to right (d = 1..kmax[i]).  Every (i, d) is a candidate; the first
 * min(budget, #{P >= min_gain}) candidates in dcut_cmp order are kept;
 * depth_i = number kept for request i (a prefix, since P does not grow with
 * d); cu = exclusive prefix sum of depths; expected_i = sum_{d<=depth_i}
 * P_{i,d} (expected accepted drafts when conf is the conditional acceptance
 * probability), summed in fp64.
 */
int oracle_dcut_allocate(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                         int32_t budget, float min_gain, int32_t *out_depth, int32_t *out_cu,
                         double *out_expected)
{
    if (B < 0 || Kmax < 0 || Kmax > ORC_MAX_DRAFT || budget < 0 || isnan(min_gain))
        return ORC_ERR_INVALID_ARG;
    int64_t n = 0;
    for (int32_t i = 0; i < B; ++i) {
        if (kmax[i] < 0 || kmax[i] > Kmax)
            return ORC_ERR_INVALID_ARG;
        for (int32_t j = 0; j < kmax[i]; ++j) {
            float c = conf[(int64_t)i * Kmax + j];
            if (!(c >= 0.0f && c <= 1.0f))
                return ORC_ERR_INVALID_ARG;
        }
        n += kmax[i];
    }
    dcut_cand *cand = (dcut_cand *)malloc((size_t)(n > 0 ? n : 1) * sizeof(dcut_cand));
    if (!cand)
        return ORC_ERR_INVALID_ARG;
    int64_t c = 0, eligible = 0;
    for (int32_t i = 0; i < B; ++i) {
        float P = 1.0f; /* fp32 product, one rounding per factor */
        for (int32_t d = 1; d <= kmax[i]; ++d) {
            P = P * conf[(int64_t)i * Kmax + (d - 1)];
            cand[c].P = P;
            cand[c].i = i;
            cand[c].d = d;
            if (P >= min_gain)
                ++eligible;
            ++c;
        }
    }
    qsort(cand, (size_t)n, sizeof(dcut_cand), dcut_cmp);
    int64_t keep = eligible < budget ? eligible : budget;
    for (int32_t i = 0; i < B; ++i)
        out_depth[i] = 0;
    for (int64_t t = 0; t < keep; ++t)
        out_depth[cand[t].i] += 1;
    out_cu[0] = 0;
    for (int32_t i = 0; i < B; ++i)
        out_cu[i + 1] = out_cu[i] + out_depth[i];
    if (out_expected) {
        for (int32_t i = 0; i < B; ++i) {
            double e = 0.0;
            float P = 1.0f;
            for (int32_t d = 1; d <= out_depth[i]; ++d) {
                P = P * conf[(int64_t)i * Kmax + (d - 1)];
                e += (double)P;
            }
            out_expected[i] = e;
        }
    }
    free(cand);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* D-cut, cost-unit variant                                                  */
/* ------------------------------------------------------------------------ */

/*
 * The deep-dive page ("Tencent AngelSpec Speculative Decoding Framework Deep
 * Dive ...", its D-cut scheduler) budgets verification in profiled
 * latency-cost units instead of tokens.  What it computes:
 *  - cost(d): the latency of verifying depth d, given by the profiled table
 *    {1: 1.0, 2: 1.2, 4: 1.5, 8: 2.0, 16: 3.0}: the piecewise-linear
 *    function through those points, constant beyond both ends;
 *  - per request: the depth d in 1..kmax maximising
 *    benefit(d) = (conf_0 * ... * conf_{d-1}) * d / cost(d)
 *    (the first such d when several tie);
 *  - requests in decreasing order of that benefit (equal benefits keep
 *    request order), each admitted when the running cost total plus its own
 *    cost stays within max_cost; a request that does not fit is skipped and
 *    later ones are still tried.
 * Readings: all of it in fp64 (the page computes in Python floats), products
 * left to right; a request with kmax = 0 is no candidate; a request not admitted
 * verifies depth 0 (its bonus row only).
 */
/* The profiled latency table: cost at depths 1, 2, 4, 8 and 16. */
static const int32_t cost_at_depth[5] = {1, 2, 4, 8, 16};
static const double cost_value[5] = {1.0, 1.2, 1.5, 2.0, 3.0};

/*
 * cost(d) for d = 0..ORC_MAX_DRAFT, by definition: the piecewise-linear
 * function through the five (depth, cost) points, constant beyond the first
 * and the last point.  Filled segment by segment: between points a < b the
 * cost rises from cost(a) to cost(b) in proportion to (d - a) / (b - a).
 */
static void fill_cost_table(double table[ORC_MAX_DRAFT + 1])
{
    for (int32_t d = 0; d <= cost_at_depth[0]; ++d)
        table[d] = cost_value[0];
    for (int seg = 0; seg + 1 < 5; ++seg) {
        const int32_t a = cost_at_depth[seg], b = cost_at_depth[seg + 1];
        const double rise = cost_value[seg + 1] - cost_value[seg];
        for (int32_t d = a + 1; d <= b; ++d) {
            const double frac = (double)(d - a) / (double)(b - a);
            table[d] = cost_value[seg] + rise * frac;
        }
    }
    for (int32_t d = cost_at_depth[4] + 1; d <= ORC_MAX_DRAFT; ++d)
        table[d] = cost_value[4];
}

double oracle_dcut_cost(int32_t d)
{
    double table[ORC_MAX_DRAFT + 1];
    fill_cost_table(table);
    if (d < 0)
        d = 0;
    if (d > ORC_MAX_DRAFT)
        d = ORC_MAX_DRAFT;
    return table[d];
}

typedef struct {
    double benefit;
    int32_t i;
    int32_t d;
} dcut_cost_cand;

static int dcut_cost_cmp(const void *pa, const void *pb)
{
    const dcut_cost_cand *a = (const dcut_cost_cand *)pa, *b = (const dcut_cost_cand *)pb;
    if (a->benefit > b->benefit)
        return -1;
    if (a->benefit < b->benefit)
        return 1;
    return a->i < b->i ? -1 : (a->i > b->i ? 1 : 0);
}

int oracle_dcut_schedule_cost(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                              double max_cost, int32_t *out_depth, int32_t *out_cu,
                              double *out_benefit)
{
    if (B < 0 || Kmax < 0 || Kmax > ORC_MAX_DRAFT || isnan(max_cost))
        return ORC_ERR_INVALID_ARG;
    for (int32_t i = 0; i < B; ++i) {
        if (kmax[i] < 0 || kmax[i] > Kmax)
            return ORC_ERR_INVALID_ARG;
        for (int32_t j = 0; j < kmax[i]; ++j) {
            float c = conf[(int64_t)i * Kmax + j];
            if (!(c >= 0.0f && c <= 1.0f))
                return ORC_ERR_INVALID_ARG;
        }
    }
    dcut_cost_cand *cand = (dcut_cost_cand *)malloc((size_t)(B > 0 ? B : 1) * sizeof *cand);
    if (!cand)
        return ORC_ERR_INVALID_ARG;
    int32_t n = 0;
    for (int32_t i = 0; i < B; ++i) {
        out_depth[i] = 0;
        if (out_benefit)
            out_benefit[i] = 0.0;
        if (kmax[i] == 0)
            continue;
        double P = 1.0, best = -1.0;
        int32_t best_d = 0;
        for (int32_t d = 1; d <= kmax[i]; ++d) {
            P = P * (double)conf[(int64_t)i * Kmax + (d - 1)];
            double b = P * (double)d / oracle_dcut_cost(d);
            if (b > best) { /* strict: the first maximising depth is kept */
                best = b;
                best_d = d;
            }
        }
        cand[n].benefit = best;
        cand[n].i = i;
        cand[n].d = best_d;
        ++n;
    }
    qsort(cand, (size_t)n, sizeof *cand, dcut_cost_cmp);
    double total = 0.0;
    for (int32_t t = 0; t < n; ++t) {
        double c = oracle_dcut_cost(cand[t].d);
        if (total + c <= max_cost) {
            total += c;
            out_depth[cand[t].i] = cand[t].d;
            if (out_benefit)
                out_benefit[cand[t].i] = cand[t].benefit;
        }
    }
    out_cu[0] = 0;
    for (int32_t i = 0; i < B; ++i)
        out_cu[i + 1] = out_cu[i] + out_depth[i];
    free(cand);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* prefix confidence of drafted tokens                                       */
/* ------------------------------------------------------------------------ */

/*
 * D-cut allocates depth from per-request prefix confidence ("Tencent Hunyuan
 * Turns Speculative Decoding Into a Full Open-Source Stack", "What problem
 * does it solve", inference layer).  Reading: the confidence of drafted
 * token x_{i,j} is the drafter's own probability of it, q_{i,j}(x_{i,j}) =
 * softmax(draft row (i, j) / T)(x_{i,j}); at T = 0 the drafter is greedy and
 * the confidence is 1 when x_{i,j} is the row's lowest-index maximum, else 0.
 * Rows are padded, row i*Kmax + j; entries j >= kmax[i] are 0.  A failing
 * row (NaN / +inf / all masked, or a token outside [0, V)) gets NaN and the
 * first error is returned.
 */
int oracle_draft_confidence(const void *draft, int dtype, const int32_t *tokens,
                            const int32_t *kmax, int32_t B, int32_t Kmax, int64_t V, double T,
                            float *out_conf)
{
    if (B < 0 || Kmax < 0 || Kmax > ORC_MAX_DRAFT || V <= 0 || !(T >= 0) || isinf(T) ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_ERR_INVALID_ARG;
    int first_err = ORC_OK;
    for (int32_t i = 0; i < B; ++i) {
        if (kmax[i] < 0 || kmax[i] > Kmax)
            return ORC_ERR_INVALID_ARG;
        for (int32_t j = 0; j < Kmax; ++j) {
            int64_t r = (int64_t)i * Kmax + j;
            if (j >= kmax[i]) {
                out_conf[r] = 0.0f;
                continue;
            }
            int32_t x = tokens[r];
            int err = ORC_OK;
            double c = 0.0;
            if (x < 0 || x >= V) {
                err = ORC_ERR_INVALID_ARG;
            } else if (T == 0.0) {
                int32_t g;
                err = oracle_argmax_row(draft, dtype, r, V, &g);
                c = (err == ORC_OK && g == x) ? 1.0 : 0.0;
            } else {
                err = softmax_at(draft, dtype, r, V, T, x, &c);
            }
            if (err != ORC_OK) {
                out_conf[r] = NAN;
                if (first_err == ORC_OK)
                    first_err = err;
                continue;
            }
            out_conf[r] = (float)c;
        }
    }
    return first_err;
}

/* ------------------------------------------------------------------------ */
/* drafted tokens and acceptance statistics                                  */
/* ------------------------------------------------------------------------ */

/*
 * The step before verification: the drafter proposes its tokens
 * ("Tencent Hunyuan Turns Speculative Decoding Into a Full Open-Source
 * Stack", "What problem does it solve": a lightweight drafter proposes the
 * candidate sequence).  Reading: for a drafter that samples, x_{i,j} is the
 * inverse CDF of q_{i,j} = softmax(draft row (i, j) / T) at the uniform
 * u[i*Kmax + j] (smallest v with C(v) > u * S, as for the final draw);
 * greedy (T = 0) takes the lowest-index maximum.  out_conf = q(x) (1 at
 * T = 0).  Rows j >= kmax[i] give token -1 and conf 0; a failing row gives
 * -1 and NaN and the first error is returned.
 */
int oracle_draft_sample(const void *draft, int dtype, const int32_t *kmax, int32_t B,
                        int32_t Kmax, int64_t V, double T, const float *u, int32_t *out_tokens,
                        float *out_conf)
{
    if (B < 0 || Kmax < 0 || Kmax > ORC_MAX_DRAFT || V <= 0 || V > INT32_MAX || !(T >= 0) ||
        isinf(T) || (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_ERR_INVALID_ARG;
    double *w = (double *)malloc((size_t)V * sizeof(double));
    if (!w)
        return ORC_ERR_INVALID_ARG;
    int first_err = ORC_OK;
    for (int32_t i = 0; i < B; ++i) {
        if (kmax[i] < 0 || kmax[i] > Kmax) {
            free(w);
            return ORC_ERR_INVALID_ARG;
        }
        for (int32_t j = 0; j < Kmax; ++j) {
            int64_t r = (int64_t)i * Kmax + j;
            out_tokens[r] = -1;
            out_conf[r] = 0.0f;
            if (j >= kmax[i])
                continue;
            int err;
            if (T == 0.0) {
                int32_t g;
                err = oracle_argmax_row(draft, dtype, r, V, &g);
                if (err == ORC_OK) {
                    out_tokens[r] = g;
                    out_conf[r] = 1.0f;
                }
            } else {
                err = oracle_softmax_row(draft, dtype, r, V, T, w);
                if (err == ORC_OK) {
                    int64_t x = oracle_inverse_cdf(w, V, (double)u[r], NULL, NULL);
                    if (x < 0) {
                        err = ORC_ERR_NONFINITE;
                    } else {
                        out_tokens[r] = (int32_t)x;
                        out_conf[r] = (float)w[x];
                    }
                }
            }
            if (err != ORC_OK) {
                out_conf[r] = NAN;
                if (first_err == ORC_OK)
                    first_err = err;
            }
        }
    }
    free(w);
    return first_err;
}

/*
 * The statistics the pages report for a drafter (mean accepted length;
 * per-position acceptance: the French/Russian page's numbers at T = 0 and by
 * position; the online evaluation reads both from the serving engine,
 * "Tencent Hunyuan Turns Speculative Decoding ...", "Five angles worth a
 * closer look", item 4), from one verification call's outputs:
 *   reached[j]  = #{ i : K_i > j and a_i >= j }   (position j was tested)
 *   accepted[j] = #{ i : a_i > j }                 (and accepted)
 *   mean accepted length = sum a_i / #requests
 * over requests whose a_i >= 0 (poisoned requests are left out), j < Kmax.
 */
int oracle_acceptance_stats(const int32_t *accept_len, const int32_t *cu, int32_t B,
                            int32_t Kmax, int32_t *out_reached, int32_t *out_accepted,
                            double *out_mean)
{
    if (B < 0 || Kmax < 0 || Kmax > ORC_MAX_DRAFT)
        return ORC_ERR_INVALID_ARG;
    for (int32_t j = 0; j < Kmax; ++j)
        out_reached[j] = out_accepted[j] = 0;
    int64_t total = 0, n = 0;
    for (int32_t i = 0; i < B; ++i) {
        int32_t a = accept_len[i], k = cu[i + 1] - cu[i];
        if (a < 0)
            continue;
        if (a > k || k > Kmax)
            return ORC_ERR_INVALID_ARG;
        total += a;
        ++n;
        for (int32_t j = 0; j < k; ++j) {
            if (a >= j)
                out_reached[j] += 1;
            if (a > j)
                out_accepted[j] += 1;
        }
    }
    *out_mean = n > 0 ? (double)total / (double)n : 0.0;
    return ORC_OK;
}
