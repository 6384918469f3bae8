/*
 * spec_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, fp64 CPU statement of the target-side verify step of speculative decoding.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg load this file's
 * library; the CUDA product path never calls it and shares no code, header or table with it.
 *
 * Every function follows the page that defines the operation (page title + section):
 *   [M7.1]  "M7.1 - Speculative Decoding: Draft, Verify, Accept, Reject"
 *           (transformer-system.numinens.com), sections 0x03, 0x03B-0x03D, 0x03F-0x03H, 0x04, 0x04J.
 *   [M16]   "Module 16" speculative-decoding lesson (learnllm.pages.dev), "The Math: Speculative
 *           Sampling", "The Candidate Tree", "Verify the Tree -- and Why It's Exact".
 *   [M7.7]  "M7.7 - Draft Sources, Dependent Heads, Hardware-Aware Trees", section 0x07E
 *           (candidate row / predictor row convention), 0x08B (re-testing k candidates against the
 *           same target is wrong), 0x09A (stochastic residual update over a node's children).
 *   [TRLM]  "Exact speculative and assisted decoding for TinyRustLM" (mikekappel.com),
 *           "Normative stochastic pseudocode", "Normative edge-case behavior".
 *   [SMC]   the same Module 16 lesson, "SMC Speculative Decoding: Resample, Don't Reject":
 *           "The Math: Reweight, Don't Reject" (block weight, ESS, Algorithm 1), "Two Exact Anchors".
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - accept iff u < a with u in [0,1)                            ([M16] accept rule)
 *   - one uniform draws a categorical by inverse CDF in ascending token order on the
 *     unnormalised mass: the smallest v with u*Z < C(v); if rounding runs off the end,
 *     the largest v with positive mass
 *   - uniform slot gamma feeds the correction draw, slot gamma+1 the bonus draw
 *   - top-k keeps every token whose stored logit is >= the k-th largest stored logit
 *     (counted with multiplicity), applied to target and draft rows alike, before temperature
 *   - a request whose rows hold NaN or +inf, or a row with no finite-or-minus-inf mass, is
 *     reported as non-finite; a draft token outside [0,V) or with q(x) = 0 is a bad token;
 *     uniforms outside [0,1) are a bad uniform; such requests emit nothing (-1).
 *   - tree argmax ties go to the lowest token index; the deepest valid node wins, ties to the
 *     lowest node index.
 *   - top-p keeps whole groups of equal stored logit in descending order until the kept mass (after
 *     temperature) first reaches top_p, ties with the last group kept included
 *   - typical acceptance (tree): a node passes when p(x) > min(eps, delta exp(-H)) strictly, H the
 *     natural-log entropy of its predictor row after temperature; the token after the accepted
 *     path is drawn from p of the accepted node's own row with the request's one uniform
 *   - SMC-SD round: uniform slot 0 draws the extension token from row K, slot 1 the particle's
 *     ancestor; ancestors are drawn by inverse CDF over the group's normalised weights in particle
 *     order; a particle with a bad status leaves its group's ESS and resampling undefined (NaN, -1)
 *   - stochastic tree: a node's children are tested in ascending node index; node i's accept test
 *     uses uniform slot i and the one final draw (correction or bonus) uses slot N; only the rows
 *     the walk visits are read, so a bad value in a row it never reaches goes unseen.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };
enum {
    OR_ROW_OK = 0,
    OR_ROW_NONFINITE = 1,
    OR_ROW_DEGENERATE = 2,
    OR_ROW_BAD_TOKEN = 3,
    OR_ROW_BAD_PARENT = 5,
    OR_ROW_OVERFLOW = 6,
    OR_ROW_BAD_UNIFORM = 7,
    OR_ROW_BAD_QROW = 8
};

/* ---------------------------------------------------------------- element access */

static double load_logit(const void* base, int dtype, size_t i)
{
    if (dtype == OR_F64) return ((const double*)base)[i];
    if (dtype == OR_F32) return (double)((const float*)base)[i];
    /* bf16: the stored 16 bits are the high half of an IEEE binary32 */
    uint16_t h = ((const uint16_t*)base)[i];
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- top-k threshold */

static int cmp_desc(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

/* k-th largest of x[0..n) counted with multiplicity: sort a copy in descending order. */
double oracle_kth_largest(const double* x, int n, int k)
{
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    memcpy(s, x, sizeof(double) * (size_t)n);
    qsort(s, (size_t)n, sizeof(double), cmp_desc);
    double t = s[k - 1];
    free(s);
    return t;
}

/* ---------------------------------------------------------------- processors + softmax */

/* Grammar mask bit of token v: bit (v mod 32) of 32-bit word v / 32 of the row's words. */
static int token_allowed(const uint32_t* allowed, int v)
{
    return (int)((allowed[v / 32] >> (v % 32)) & 1u);
}

/*
 * One probability row after the declared processors ([M7.1] 0x02A: p_i = Pi_T(logits)):
 *   optional grammar mask, optional top-k on the stored logits, then z = logit / T, then max-shift
 *   softmax ([M7.1] 0x04J backend 1).  Returns a row status; fills p[0..V) and *lse (natural log
 *   of the normaliser of z over the kept tokens) and *thr (the top-k threshold, -inf without
 *   top-k).
 *
 * The grammar mask ([TRLM] "Grammar and deterministic opportunities") replaces q by
 *   q_G(x) = q(x) 1[x in A_G] / sum_v q(v) 1[v in A_G]:
 * `allowed` (NULL = every token) holds one bit per token of the valid set A_G.  A token outside
 * A_G is removed before anything else reads the row: its stored logit becomes -inf, so a NaN or
 * +inf there is never seen.  The normalisation over A_G is then the softmax's own.
 */
int oracle_row_probs_masked(const void* base, int dtype, size_t off, int V, double T, int top_k,
                            const uint32_t* allowed, double* p, double* lse, double* thr)
{
    if (V < 1) return OR_ROW_NONFINITE;
    double* x = (double*)malloc(sizeof(double) * (size_t)V);
    int v;
    for (v = 0; v < V; ++v) {
        x[v] = (allowed && !token_allowed(allowed, v)) ? -INFINITY
                                                       : load_logit(base, dtype, off + (size_t)v);
        if (isnan(x[v]) || (isinf(x[v]) && x[v] > 0)) { free(x); return OR_ROW_NONFINITE; }
    }
    double t = -INFINITY;
    if (top_k > 0 && top_k < V) t = oracle_kth_largest(x, V, top_k);
    *thr = t;

    /* z over the kept set; -inf elsewhere */
    double m = -INFINITY;
    for (v = 0; v < V; ++v) {
        double z = (x[v] >= t) ? x[v] / T : -INFINITY;
        x[v] = z;
        if (z > m) m = z;
    }
    if (m == -INFINITY) { free(x); return OR_ROW_NONFINITE; } /* no valid token */
    double S = 0.0;
    for (v = 0; v < V; ++v) {
        double e = (x[v] == -INFINITY) ? 0.0 : exp(x[v] - m);
        p[v] = e;
        S += e;
    }
    for (v = 0; v < V; ++v) p[v] /= S;
    *lse = m + log(S);
    free(x);
    return OR_ROW_OK;
}

/* The same row without a grammar mask. */
int oracle_row_probs(const void* base, int dtype, size_t off, int V, double T, int top_k,
                     double* p, double* lse, double* thr)
{
    return oracle_row_probs_masked(base, dtype, off, V, T, top_k, NULL, p, lse, thr);
}

/* (stored logit, probability) pairs, ordered by descending logit */
typedef struct {
    double x, p;
} xp_pair;

static int cmp_pair_desc(const void* a, const void* b)
{
    double x = ((const xp_pair*)a)->x, y = ((const xp_pair*)b)->x;
    return (x < y) - (x > y);
}

/*
 * One probability row after temperature and a top-p (nucleus) processor: with p = softmax(x / T),
 * keep the tokens of largest probability, whole groups of equal stored logit at a time in
 * descending order, until the kept mass first reaches top_p; every token tied with the last group
 * kept stays in.  The kept set is {v : x_v >= g}, g that group's logit; p is then renormalised over
 * it.  top_p >= 1 keeps every token.  *thr receives g (-inf when all are kept) and *margin the
 * distance between top_p and the two cumulative masses around the chosen group (the decision's
 * rounding exposure).
 */
int oracle_row_probs_topp(const void* base, int dtype, size_t off, int V, double T, double top_p,
                          double* p, double* lse, double* thr, double* margin)
{
    double t = -INFINITY, mg = INFINITY;
    int st = oracle_row_probs(base, dtype, off, V, T, 0, p, lse, thr);
    if (st != OR_ROW_OK || !(top_p < 1.0)) {
        *thr = -INFINITY;
        *margin = mg;
        return st;
    }
    xp_pair* srt = (xp_pair*)malloc(sizeof(xp_pair) * (size_t)V);
    for (int v = 0; v < V; ++v) {
        srt[v].x = load_logit(base, dtype, off + (size_t)v);
        srt[v].p = p[v];
    }
    qsort(srt, (size_t)V, sizeof(xp_pair), cmp_pair_desc);
    double cum = 0.0;
    for (int i = 0; i < V;) {
        const double g = srt[i].x;
        const double before = cum;
        while (i < V && srt[i].x == g) cum += srt[i++].p; /* the whole group of equal logits */
        if (cum >= top_p) {
            t = g;
            mg = fmin(fabs(before - top_p), fabs(cum - top_p));
            break;
        }
    }
    free(srt);
    /* renormalise over the kept set {x >= t} */
    double m = -INFINITY, S = 0.0;
    for (int v = 0; v < V; ++v) {
        const double x = load_logit(base, dtype, off + (size_t)v);
        if (x >= t && x / T > m) m = x / T;
    }
    for (int v = 0; v < V; ++v) {
        const double x = load_logit(base, dtype, off + (size_t)v);
        p[v] = (x >= t && x > -INFINITY) ? exp(x / T - m) : 0.0;
        S += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= S;
    *lse = m + log(S);
    *thr = t;
    *margin = mg;
    return OR_ROW_OK;
}

/* Backend 2 of [M7.1] 0x04J: an online (m, l) merge over vocabulary blocks of width `block`.
 * Returns the log-normaliser of z[0..n). */
double oracle_lse_online(const double* z, int n, int block)
{
    double m = -INFINITY, l = 0.0;
    for (int s = 0; s < n; s += block) {
        int e = s + block < n ? s + block : n;
        double bm = -INFINITY, bl = 0.0;
        for (int v = s; v < e; ++v) if (z[v] > bm) bm = z[v];
        if (bm == -INFINITY) continue;
        for (int v = s; v < e; ++v) bl += exp(z[v] - bm);
        double nm = bm > m ? bm : m;
        l = l * exp(m - nm) + bl * exp(bm - nm);
        m = nm;
    }
    return m + log(l);
}

/* Backend 1 of [M7.1] 0x04J: conventional max-shift log-normaliser. */
double oracle_lse_maxshift(const double* z, int n)
{
    double m = -INFINITY, S = 0.0;
    for (int v = 0; v < n; ++v) if (z[v] > m) m = z[v];
    for (int v = 0; v < n; ++v) S += exp(z[v] - m);
    return m + log(S);
}

/* Acceptance rate alpha = sum_x min(p(x), q(x))  ([M7.1] 0x03B). */
double oracle_alpha(const double* p, const double* q, int V)
{
    double a = 0.0;
    for (int v = 0; v < V; ++v) a += p[v] < q[v] ? p[v] : q[v];
    return a;
}

/* Normalised positive residual [p - q]_+ / Z ([M7.1] 0x03C); returns Z. */
double oracle_residual(const double* p, const double* q, int V, double* out)
{
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        double r = p[v] - q[v];
        out[v] = r > 0.0 ? r : 0.0; /* clamp tiny negatives ([M7.1] 0x03D) */
        Z += out[v];
    }
    if (Z > 0.0)
        for (int v = 0; v < V; ++v) out[v] /= Z;
    return Z;
}

/*
 * Inverse-CDF draw from unnormalised mass r[0..V) with one uniform u: the smallest v with
 * u*Z < C(v), C the running sum in ascending index order.  Returns -1 when Z <= 0.  *lo and *hi
 * receive C(v-1)/Z and C(v)/Z of the chosen token (for boundary-distance reporting).
 */
int oracle_inverse_cdf(const double* r, int V, double u, double* lo, double* hi)
{
    double Z = 0.0;
    int v;
    for (v = 0; v < V; ++v) Z += r[v];
    if (!(Z > 0.0)) return -1;
    double t = u * Z, C = 0.0, Cprev = 0.0;
    for (v = 0; v < V; ++v) {
        Cprev = C;
        C += r[v];
        if (t < C) { *lo = Cprev / Z; *hi = C / Z; return v; }
    }
    for (v = V - 1; v >= 0; --v) /* rounding ran off the end */
        if (r[v] > 0.0) { *lo = 1.0; *hi = 1.0; return v; }
    return -1;
}

/* ---------------------------------------------------------------- the verify round */

/*
 * Exact speculative sampling verify for B independent requests ([M7.1] 0x04 loop body,
 * [TRLM] exact_speculative_round, [M16] accept rule + residual):
 *
 *   target  [B, gamma+1, V]  row i scores draft token i; row gamma scores the bonus position
 *   draft   [B, gamma,   V]  row i is the proposal row that sampled draft token i
 *   tokens  [B, gamma]
 *   uniforms[B, gamma+2]     slots 0..gamma-1 accept draws, slot gamma correction, gamma+1 bonus
 *
 * Outputs: accepted_len[B] (A, or -1), out_tokens[B, gamma+1] (accepted prefix, correction or
 * bonus, then -1), row_status[B], lse_p[B, gamma+1], lse_q[B, gamma], accept[B, gamma]
 * (a_i = min(1, p_i(x_i)/q_i(x_i)) at every position), margin[B] (smallest distance between a
 * used uniform and a decision boundary it was compared with: |u_i - a_i| for every reached
 * accept test and |u - C(v-1)/Z|, |u - C(v)/Z| for the drawn token; under top-p it also covers
 * every row's kept-set decision), set_margin[B] (top-p only: the smallest distance between top_p
 * and the cumulative masses around a row's last kept group, over the request's rows; +inf when no
 * kept set was chosen by mass).  Any output pointer except the first two may be NULL.
 */
static int spec_verify_impl(const void* target, const void* draft, int dtype, const int32_t* tokens,
                            const float* uniforms, int B, int gamma, int V, double T, int top_k,
                            const uint32_t* allowed, double top_p, int32_t* accepted_len,
                            int32_t* out_tokens, int32_t* row_status, double* lse_p,
                            double* lse_q, double* accept, double* margin, double* set_margin)
{
    if (B < 0 || gamma < 0 || V < 1 || !(T > 0.0)) return 1;
    const size_t W = (size_t)(V + 31) / 32; /* mask words per position */
    double* p = (double*)malloc(sizeof(double) * (size_t)(gamma + 1) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)(gamma > 0 ? gamma : 1) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int st = OR_ROW_OK;
        double thr, rmg = INFINITY, rm;
        for (int i = 0; i <= gamma; ++i) {
            double l = NAN;
            size_t off = ((size_t)b * (size_t)(gamma + 1) + (size_t)i) * (size_t)V;
            const uint32_t* m = allowed ? allowed + ((size_t)b * (size_t)(gamma + 1) + (size_t)i) * W : NULL;
            int s = top_p < 1.0
                        ? oracle_row_probs_topp(target, dtype, off, V, T, top_p, p + (size_t)i * V, &l, &thr, &rm)
                        : oracle_row_probs_masked(target, dtype, off, V, T, top_k, m, p + (size_t)i * V, &l, &thr);
            if (top_p < 1.0 && rm < rmg) rmg = rm;
            if (s != OR_ROW_OK) st = OR_ROW_NONFINITE;
            if (lse_p) lse_p[(size_t)b * (gamma + 1) + i] = l;
        }
        for (int i = 0; i < gamma; ++i) {
            double l = NAN;
            size_t off = ((size_t)b * (size_t)gamma + (size_t)i) * (size_t)V;
            /* the draft row of position i sampled under the same grammar state as target row i */
            const uint32_t* m = allowed ? allowed + ((size_t)b * (size_t)(gamma + 1) + (size_t)i) * W : NULL;
            int s = top_p < 1.0
                        ? oracle_row_probs_topp(draft, dtype, off, V, T, top_p, q + (size_t)i * V, &l, &thr, &rm)
                        : oracle_row_probs_masked(draft, dtype, off, V, T, top_k, m, q + (size_t)i * V, &l, &thr);
            if (top_p < 1.0 && rm < rmg) rmg = rm;
            if (s != OR_ROW_OK) st = OR_ROW_NONFINITE;
            if (lse_q) lse_q[(size_t)b * gamma + i] = l;
        }
        const int32_t* tok = tokens + (size_t)b * gamma;
        const float* u = uniforms + (size_t)b * (gamma + 2);
        if (st == OR_ROW_OK)
            for (int i = 0; i < gamma; ++i)
                if (tok[i] < 0 || tok[i] >= V) st = OR_ROW_BAD_TOKEN;
        double* a = (double*)malloc(sizeof(double) * (size_t)(gamma > 0 ? gamma : 1));
        for (int i = 0; i < gamma; ++i) a[i] = NAN;
        if (st == OR_ROW_OK) {
            for (int i = 0; i < gamma; ++i) {
                double pi = p[(size_t)i * V + tok[i]], qi = q[(size_t)i * V + tok[i]];
                if (qi == 0.0) { st = OR_ROW_BAD_TOKEN; break; } /* q never proposes x */
                double ratio = pi / qi;
                a[i] = ratio < 1.0 ? ratio : 1.0;
            }
        }
        if (st == OR_ROW_OK)
            for (int i = 0; i < gamma + 2; ++i)
                if (!(u[i] >= 0.0f && u[i] < 1.0f)) st = OR_ROW_BAD_UNIFORM;
        if (accept)
            for (int i = 0; i < gamma; ++i) accept[(size_t)b * gamma + i] = a[i];

        int32_t* out = out_tokens + (size_t)b * (gamma + 1);
        for (int i = 0; i <= gamma; ++i) out[i] = -1;
        double mg = rmg; /* top-p: how close a row's kept set came to changing */
        int A = -1;
        if (st == OR_ROW_OK) {
            /* first rejection ([M7.1] 0x03G) */
            A = gamma;
            for (int i = 0; i < gamma; ++i) {
                double d = fabs((double)u[i] - a[i]);
                if (d < mg) mg = d;
                if (!((double)u[i] < a[i])) { A = i; break; }
            }
            double uu;
            if (A < gamma) { /* correction from the positive residual ([M7.1] 0x03C) */
                for (int v = 0; v < V; ++v) {
                    double d = p[(size_t)A * V + v] - q[(size_t)A * V + v];
                    r[v] = d > 0.0 ? d : 0.0;
                }
                uu = (double)u[gamma];
            } else {       /* bonus from the target row after the full draft ([M7.1] 0x03H) */
                for (int v = 0; v < V; ++v) r[v] = p[(size_t)gamma * V + v];
                uu = (double)u[gamma + 1];
            }
            double lo = 0.0, hi = 0.0;
            int y = oracle_inverse_cdf(r, V, uu, &lo, &hi);
            if (y < 0) {
                st = OR_ROW_DEGENERATE;
                A = -1;
            } else {
                double d1 = fabs(uu - lo), d2 = fabs(uu - hi);
                if (d1 < mg) mg = d1;
                if (d2 < mg) mg = d2;
                for (int i = 0; i < A; ++i) out[i] = tok[i];
                out[A] = y;
            }
        }
        if (st != OR_ROW_OK) A = -1;
        accepted_len[b] = A;
        if (row_status) row_status[b] = st;
        if (margin) margin[b] = mg;
        if (set_margin) set_margin[b] = rmg;
        free(a);
    }
    free(p);
    free(q);
    free(r);
    return 0;
}

int oracle_spec_verify(const void* target, const void* draft, int dtype, const int32_t* tokens,
                       const float* uniforms, int B, int gamma, int V, double T, int top_k,
                       int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                       double* lse_p, double* lse_q, double* accept, double* margin)
{
    return spec_verify_impl(target, draft, dtype, tokens, uniforms, B, gamma, V, T, top_k, NULL,
                            2.0, accepted_len, out_tokens, row_status, lse_p, lse_q, accept, margin,
                            NULL);
}

/*
 * The verify round with a top-p (nucleus) processor on every target and draft row after temperature
 * (oracle_row_probs_topp; "Exact speculative and assisted decoding for TinyRustLM": top-p is one of
 * the declared processors both distributions pass through; M7.1 0x03D: truncation keeps exactness
 * when q is the truncated distribution that sampled the draft).  0 < top_p; top_p >= 1 is the plain
 * round.  margin[b] also covers each row's kept-set decision; set_margin[b] is that decision's part
 * alone (the normalisers and accept ratios depend on it, not on the uniforms).  Everything else as
 * oracle_spec_verify.
 */
int oracle_spec_verify_topp(const void* target, const void* draft, int dtype, const int32_t* tokens,
                            const float* uniforms, int B, int gamma, int V, double T, double top_p,
                            int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                            double* lse_p, double* lse_q, double* accept, double* margin,
                            double* set_margin)
{
    if (!(top_p > 0.0)) return 1;
    return spec_verify_impl(target, draft, dtype, tokens, uniforms, B, gamma, V, T, 0, NULL, top_p,
                            accepted_len, out_tokens, row_status, lse_p, lse_q, accept, margin,
                            set_margin);
}

/*
 * The verify round under a grammar mask ([TRLM] "Grammar and deterministic opportunities": exact
 * speculation is exact relative to q_G when baseline and speculative execution mask alike).
 *   allowed [B, gamma+1, ceil(V/32)] uint32: the valid-token set of position i, one bit per token
 *           (bit v mod 32 of word v / 32).  Position i masks target row i and draft row i (the
 *           draft sampled token i in the same grammar state); position gamma masks the bonus row.
 * Temperature only (no top-k); everything else as oracle_spec_verify.
 */
int oracle_spec_verify_masked(const void* target, const void* draft, int dtype,
                              const int32_t* tokens, const float* uniforms, int B, int gamma,
                              int V, double T, const uint32_t* allowed, int32_t* accepted_len,
                              int32_t* out_tokens, int32_t* row_status, double* lse_p,
                              double* lse_q, double* accept, double* margin)
{
    if (!allowed) return 1;
    return spec_verify_impl(target, draft, dtype, tokens, uniforms, B, gamma, V, T, 0, allowed, 2.0,
                            accepted_len, out_tokens, row_status, lse_p, lse_q, accept, margin, NULL);
}

/* ---------------------------------------------------------------- greedy tree verify */

/*
 * Medusa-style greedy tree verify ([M16] "Verify the Tree", [M7.7] 0x07E row convention):
 *   logits  [B, N+1, V]  row 0 = prefix frontier, row i+1 = produced at candidate node i
 *   parents [B, N]       parent node of node i, -1 for a depth-1 node, else in [0, i)
 *   tokens  [B, N]       candidate token of node i
 * Node i is valid when its token equals the argmax of its predictor row (frontier row for a
 * depth-1 node, row parent+1 otherwise) and its parent is valid.  The deepest valid node (lowest
 * index on ties) is accepted with its root path; the bonus is the argmax of that node's own row
 * (of the frontier row when no node is valid).
 * Outputs: accepted_len[B], out_tokens[B, max_out] (path tokens, bonus, then -1),
 * out_nodes[B, max_out-1] (node ids on the path, then -1; may be NULL), row_status[B],
 * amax[B, N+1] (argmax of each row; may be NULL).
 */
int oracle_tree_verify_greedy(const void* logits, int dtype, const int32_t* parents,
                              const int32_t* tokens, int B, int N, int V, int max_out,
                              int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                              int32_t* row_status, int32_t* amax_out)
{
    if (B < 0 || N < 0 || V < 1 || max_out < 1) return 1;
    int32_t* amax = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
    int32_t* valid = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int32_t* path = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
    for (int b = 0; b < B; ++b) {
        int st = OR_ROW_OK;
        for (int j = 0; j <= N; ++j) {
            size_t off = ((size_t)b * (size_t)(N + 1) + (size_t)j) * (size_t)V;
            double best = -INFINITY;
            int bi = -1;
            for (int v = 0; v < V; ++v) {
                double x = load_logit(logits, dtype, off + (size_t)v);
                if (isnan(x)) { st = OR_ROW_NONFINITE; continue; }
                if (bi < 0 ? x > -INFINITY : x > best) { best = x; bi = v; }
            }
            if (bi < 0) st = OR_ROW_NONFINITE; /* every entry -inf: no valid token */
            amax[j] = bi;
            if (amax_out) amax_out[(size_t)b * (N + 1) + j] = bi;
        }
        const int32_t* par = parents + (size_t)b * N;
        const int32_t* tok = tokens + (size_t)b * N;
        if (st == OR_ROW_OK)
            for (int i = 0; i < N; ++i) {
                if (par[i] < -1 || par[i] >= i) { st = OR_ROW_BAD_PARENT; break; }
                if (tok[i] < 0 || tok[i] >= V) st = OR_ROW_BAD_TOKEN;
            }
        int best = -1, bestd = 0;
        if (st == OR_ROW_OK) {
            for (int i = 0; i < N; ++i) {
                int pr = par[i];
                int row = pr < 0 ? 0 : pr + 1;
                valid[i] = (tok[i] == amax[row]) && (pr < 0 || valid[pr]);
                depth[i] = pr < 0 ? 1 : depth[pr] + 1;
                if (valid[i] && depth[i] > bestd) { bestd = depth[i]; best = i; }
            }
            if (bestd + 1 > max_out) st = OR_ROW_OVERFLOW;
        }
        int32_t* out = out_tokens + (size_t)b * max_out;
        int32_t* on = out_nodes ? out_nodes + (size_t)b * (max_out - 1) : NULL;
        for (int i = 0; i < max_out; ++i) out[i] = -1;
        if (on) for (int i = 0; i < max_out - 1; ++i) on[i] = -1;
        if (st == OR_ROW_OK) {
            int n = 0;
            for (int i = best; i >= 0; i = par[i]) path[n++] = i;
            for (int j = 0; j < n; ++j) {
                out[j] = tok[path[n - 1 - j]];
                if (on) on[j] = path[n - 1 - j];
            }
            out[n] = amax[best < 0 ? 0 : best + 1];
            accepted_len[b] = n;
        } else {
            accepted_len[b] = -1;
        }
        if (row_status) row_status[b] = st;
    }
    free(amax);
    free(valid);
    free(depth);
    free(path);
    return 0;
}

/* ---------------------------------------------------------------- typical-acceptance tree verify */

/*
 * Medusa-style tree verify with typical acceptance ([M16] "Verify the Tree": Medusa's sampling
 * mode swaps the greedy check for typical acceptance, accepting a token when the target's
 * probability clears min(eps, delta * exp(-H))):
 *   logits   [B, N+1, V]  row 0 = prefix frontier, row i+1 = produced at candidate node i
 *   parents  [B, N]       -1 for a depth-1 node, else in [0, i)
 *   tokens   [B, N]
 *   uniforms [B]          the final draw
 * Row j's distribution is p_j = softmax(logits[b][j] / T) and its entropy H_j = -sum p_j ln p_j.
 * Node i is typical when p_r(tok_i) > min(eps, delta * exp(-H_r)), r its predictor row (0 for a
 * depth-1 node, parent + 1 otherwise), and valid when it is typical and its parent is valid.  The
 * deepest valid node (lowest index on ties) is accepted with its root path.  The token after the
 * path is drawn from p of the accepted node's own row (the frontier row when no node is valid) by
 * inverse CDF with uniforms[b]: in sampling mode the next token comes from the target there.
 * Statuses: a row with NaN, +inf or no finite entry -> non-finite; then a bad parent, a token
 * outside [0, V), a uniform outside [0, 1); a path and final token longer than max_out -> overflow.
 * Outputs: accepted_len[B] (path length or -1), out_tokens[B, max_out] (path tokens, the drawn
 * token, then -1), out_nodes[B, max_out-1] (nullable), row_status[B], and, each nullable:
 * entropy[B, N+1] (H of every row), logp[B, N] (ln p_r(tok_i) of every node), margin[B] (the
 * smallest |ln p_r(tok_i) - ln threshold| over the nodes whose parent is valid, and |u - C| for the
 * two CDF boundaries of the drawn token).
 */
int oracle_tree_verify_typical(const void* logits, int dtype, const int32_t* parents,
                               const int32_t* tokens, const float* uniforms, int B, int N, int V,
                               double T, double eps, double delta, int max_out,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                               int32_t* row_status, double* entropy, double* logp, double* margin)
{
    if (B < 0 || N < 0 || V < 1 || max_out < 1 || !(T > 0.0) || !(eps >= 0.0) || !(delta >= 0.0) ||
        !isfinite(eps) || !isfinite(delta))
        return 1;
    const size_t R = (size_t)N + 1;
    double* p = (double*)malloc(sizeof(double) * R * (size_t)V);
    double* H = (double*)malloc(sizeof(double) * R);
    int32_t* valid = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int32_t* path = (int32_t*)malloc(sizeof(int32_t) * R);
    for (int b = 0; b < B; ++b) {
        int st = OR_ROW_OK;
        for (size_t j = 0; j < R; ++j) {
            double lse, thr;
            double* pj = p + j * (size_t)V;
            int s = oracle_row_probs(logits, dtype, ((size_t)b * R + j) * (size_t)V, V, T, 0, pj,
                                     &lse, &thr);
            H[j] = NAN;
            if (s != OR_ROW_OK) {
                st = OR_ROW_NONFINITE;
            } else {
                double h = 0.0;
                for (int v = 0; v < V; ++v)
                    if (pj[v] > 0.0) h -= pj[v] * log(pj[v]);
                H[j] = h;
            }
            if (entropy) entropy[(size_t)b * R + j] = H[j];
        }
        const int32_t* par = parents + (size_t)b * N;
        const int32_t* tok = tokens + (size_t)b * N;
        const double u = (double)uniforms[b];
        if (st == OR_ROW_OK)
            for (int i = 0; i < N; ++i) {
                if (par[i] < -1 || par[i] >= i) { st = OR_ROW_BAD_PARENT; break; }
                if (tok[i] < 0 || tok[i] >= V) st = OR_ROW_BAD_TOKEN;
            }
        if (st == OR_ROW_OK && !(u >= 0.0 && u < 1.0)) st = OR_ROW_BAD_UNIFORM;
        double mg = INFINITY;
        int best = -1, bestd = 0;
        for (int i = 0; i < N; ++i)
            if (logp) logp[(size_t)b * N + i] = NAN;
        if (st == OR_ROW_OK) {
            for (int i = 0; i < N; ++i) {
                const int pr = par[i];
                const int row = pr < 0 ? 0 : pr + 1;
                const double px = p[(size_t)row * V + tok[i]];
                const double thr = fmin(eps, delta * exp(-H[row]));
                const int typical = px > thr;
                if (logp) logp[(size_t)b * N + i] = log(px);
                if (pr < 0 || valid[pr]) { /* a test that decides the outcome */
                    double d = fabs(log(px) - log(thr));
                    if (d < mg) mg = d;
                }
                valid[i] = typical && (pr < 0 || valid[pr]);
                depth[i] = pr < 0 ? 1 : depth[pr] + 1;
                if (valid[i] && depth[i] > bestd) { bestd = depth[i]; best = i; }
            }
            if (bestd + 1 > max_out) st = OR_ROW_OVERFLOW;
        }
        int32_t* out = out_tokens + (size_t)b * max_out;
        int32_t* on = out_nodes ? out_nodes + (size_t)b * (max_out - 1) : NULL;
        for (int i = 0; i < max_out; ++i) out[i] = -1;
        if (on) for (int i = 0; i < max_out - 1; ++i) on[i] = -1;
        if (st == OR_ROW_OK) {
            const int row = best < 0 ? 0 : best + 1;
            double lo = 0.0, hi = 0.0;
            const int y = oracle_inverse_cdf(p + (size_t)row * V, V, u, &lo, &hi);
            double d1 = fabs(u - lo), d2 = fabs(u - hi);
            if (d1 < mg) mg = d1;
            if (d2 < mg) mg = d2;
            int n = 0;
            for (int i = best; i >= 0; i = par[i]) path[n++] = i;
            for (int j = 0; j < n; ++j) {
                out[j] = tok[path[n - 1 - j]];
                if (on) on[j] = path[n - 1 - j];
            }
            out[n] = y;
            accepted_len[b] = n;
        } else {
            accepted_len[b] = -1;
        }
        if (row_status) row_status[b] = st;
        if (margin) margin[b] = mg;
    }
    free(p);
    free(H);
    free(valid);
    free(depth);
    free(path);
    return 0;
}

/* ---------------------------------------------------------------- stochastic tree verify */

/*
 * Stochastic verification of a candidate tree by the residual update over children
 * ([M7.7] 0x09A; [M7.7] 0x07E row convention; [M16] accept rule and inverse-CDF draw):
 *   target   [B, N+1, V]  row 0 = prefix frontier, row i+1 = produced at node i
 *   draft    [B, Nq, V]   proposal rows; node i's token was drawn from row qrow[b,i]
 *   parents  [B, N]       -1 for a depth-1 node, else in [0, i)
 *   tokens   [B, N], qrow [B, N]
 *   uniforms [B, N+1]     slot i = the accept test of node i, slot N = the final draw
 * The walk starts at the frontier.  At the current node it sets r = p (the processed target row of
 * the node) and tests the children in ascending index: child s with token x is accepted when
 * u[s] < min(1, r(x)/q_s(x)); the walk then moves to s.  On rejection r becomes the normalised
 * positive part of r - q_s.  When every child is rejected the final token is drawn from r; when the
 * node has no children it is the bonus, drawn from p.  Either way the draw uses u[N].
 * Outputs: accepted_len[B] (path length, or -1), out_tokens[B, max_out] (path tokens, final token,
 * then -1), out_nodes[B, max_out-1] (path node ids, then -1; may be NULL), row_status[B], and, each
 * nullable: accept[B, N] (the ratio of every tested node, NaN for the rest), margin[B] (smallest
 * distance between a used uniform and a boundary it was compared with), draw_lo / draw_hi [B] (the
 * normalised CDF interval [C(y-1), C(y)) of the final token).
 */
int oracle_tree_verify_sample(const void* target, const void* draft, int dtype,
                              const int32_t* parents, const int32_t* tokens, const int32_t* qrow,
                              const float* uniforms, int B, int N, int Nq, int V, double T,
                              int max_out, int32_t* accepted_len, int32_t* out_tokens,
                              int32_t* out_nodes, int32_t* row_status, double* accept,
                              double* margin, double* draw_lo, double* draw_hi)
{
    if (B < 0 || N < 0 || Nq < 0 || V < 1 || !(T > 0.0) || max_out < 1) return 1;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    int32_t* path = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N + 1));
    for (int b = 0; b < B; ++b) {
        const int32_t* par = parents + (size_t)b * N;
        const int32_t* tok = tokens + (size_t)b * N;
        const int32_t* qr = qrow + (size_t)b * N;
        const float* u = uniforms + (size_t)b * (N + 1);
        int st = OR_ROW_OK;
        /* what the host-side description fixes, before any row is read */
        for (int i = 0; i < N && st == OR_ROW_OK; ++i)
            if (par[i] < -1 || par[i] >= i) st = OR_ROW_BAD_PARENT;
        for (int i = 0; i < N && st == OR_ROW_OK; ++i)
            if (qr[i] < 0 || qr[i] >= Nq) st = OR_ROW_BAD_QROW;
        for (int i = 0; i < N && st == OR_ROW_OK; ++i)
            if (tok[i] < 0 || tok[i] >= V) st = OR_ROW_BAD_TOKEN;
        for (int i = 0; i <= N && st == OR_ROW_OK; ++i)
            if (!(u[i] >= 0.0f && u[i] < 1.0f)) st = OR_ROW_BAD_UNIFORM;
        if (accept)
            for (int i = 0; i < N; ++i) accept[(size_t)b * N + i] = NAN;

        double mg = INFINITY, lo = NAN, hi = NAN;
        int n = 0, y = -1;
        int cur = -1; /* the frontier */
        while (st == OR_ROW_OK) {
            double l, thr;
            size_t off = ((size_t)b * (size_t)(N + 1) + (size_t)(cur + 1)) * (size_t)V;
            if (oracle_row_probs(target, dtype, off, V, T, 0, p, &l, &thr) != OR_ROW_OK) {
                st = OR_ROW_NONFINITE;
                break;
            }
            for (int v = 0; v < V; ++v) r[v] = p[v];
            int next = -1;
            for (int s = cur + 1; s < N && next < 0; ++s) {
                if (par[s] != cur) continue;
                size_t qoff = ((size_t)b * (size_t)Nq + (size_t)qr[s]) * (size_t)V;
                if (oracle_row_probs(draft, dtype, qoff, V, T, 0, q, &l, &thr) != OR_ROW_OK) {
                    st = OR_ROW_NONFINITE;
                    break;
                }
                int x = tok[s];
                if (q[x] == 0.0) { st = OR_ROW_BAD_TOKEN; break; } /* q never proposes x */
                double ratio = r[x] / q[x];
                double a = ratio < 1.0 ? ratio : 1.0;
                if (accept) accept[(size_t)b * N + s] = a;
                double d = fabs((double)u[s] - a);
                if (d < mg) mg = d;
                if ((double)u[s] < a) { next = s; break; }
                /* rejected: the remaining target mass is the positive residual ([M7.7] 0x09A) */
                double Z = oracle_residual(r, q, V, r);
                if (!(Z > 0.0)) { st = OR_ROW_DEGENERATE; break; }
            }
            if (st != OR_ROW_OK) break;
            if (next >= 0) {
                path[n++] = next;
                cur = next;
                if (n + 1 > max_out) { st = OR_ROW_OVERFLOW; break; }
                continue;
            }
            /* every child rejected (correction from r), or a leaf (bonus from p = r) */
            y = oracle_inverse_cdf(r, V, (double)u[N], &lo, &hi);
            if (y < 0) { st = OR_ROW_DEGENERATE; break; }
            double d1 = fabs((double)u[N] - lo), d2 = fabs((double)u[N] - hi);
            if (d1 < mg) mg = d1;
            if (d2 < mg) mg = d2;
            break;
        }

        int32_t* out = out_tokens + (size_t)b * max_out;
        int32_t* on = out_nodes ? out_nodes + (size_t)b * (max_out - 1) : NULL;
        for (int i = 0; i < max_out; ++i) out[i] = -1;
        if (on) for (int i = 0; i < max_out - 1; ++i) on[i] = -1;
        if (st == OR_ROW_OK) {
            for (int j = 0; j < n; ++j) {
                out[j] = tok[path[j]];
                if (on) on[j] = path[j];
            }
            out[n] = y;
            accepted_len[b] = n;
        } else {
            accepted_len[b] = -1;
            lo = hi = NAN;
        }
        if (row_status) row_status[b] = st;
        if (margin) margin[b] = mg;
        if (draw_lo) draw_lo[b] = lo;
        if (draw_hi) draw_hi[b] = hi;
    }
    free(p);
    free(q);
    free(r);
    free(path);
    return 0;
}

/* ---------------------------------------------------------------- SMC-SD verify round */

/*
 * Effective sample size of n weights given as logs ([SMC] "The Math"): (sum w)^2 / sum w^2, with the
 * weights scaled by their largest (the ratio does not change).  Returns NaN if a weight is NaN.
 */
double oracle_ess(const double* logw, int n)
{
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
        if (isnan(logw[i])) return NAN;
        if (logw[i] > m) m = logw[i];
    }
    if (m == -INFINITY) return NAN;
    double s1 = 0.0, s2 = 0.0;
    for (int i = 0; i < n; ++i) {
        double w = exp(logw[i] - m);
        s1 += w;
        s2 += w * w;
    }
    return s1 * s1 / s2;
}

/*
 * One SMC-SD round on the verify side for G groups of Np particles, B = G * Np requests, particle n
 * of group g at request g * Np + n ([SMC] Algorithm 1, steps 2-5):
 *   target [B, K+1, V], draft [B, K, V], tokens [B, K], logw_in [B] (natural-log weights before the
 *   round), uniforms [B, 2] (slot 0: the extension draw, slot 1: the ancestor draw), eta.
 * Per particle (processed rows as oracle_spec_verify, with temperature T and optional top-k):
 *   log W = sum_j log p_j(d_j) - log q_j(d_j)                   (step 3, in log space)
 *   x+ = inverse-CDF draw from p_K with slot 0                   (step 4)
 *   out_tokens = d_1 .. d_K, x+
 * Per group, when every particle is OK:
 *   logw_mid = logw_in + log W; ESS over logw_mid                (step 5)
 *   ESS < eta: ancestor of n = inverse-CDF draw over the normalised weights (particle order) with
 *              slot 1 of particle n; logw_out = log(1/Np); resampled = 1
 *   otherwise: ancestor of n = n; logw_out = logw_mid; resampled = 0
 * A group with a particle whose status is not OK: ess NaN, resampled -1, ancestors -1, logw_out NaN
 * (its OK particles still report their block ratio and tokens).
 * Outputs (out_tokens, row_status and logw_out required, the rest nullable): log_ratio [B], logw_out [B], ess [G],
 * resampled [G], ancestors [B], margin [B] (smallest distance of a used uniform to a boundary it was
 * compared with, over the extension and ancestor draws), ess_margin [G] (|ESS - eta| / eta).
 */
int oracle_smc_verify(const void* target, const void* draft, int dtype, const int32_t* tokens,
                      const double* logw_in, const float* uniforms, int G, int Np, int K, int V,
                      double T, int top_k, double eta, int32_t* out_tokens, int32_t* row_status,
                      double* log_ratio, double* logw_out, double* ess, int32_t* resampled,
                      int32_t* ancestors, double* margin, double* ess_margin)
{
    if (G < 0 || Np < 1 || K < 0 || V < 1 || !(T > 0.0) || !logw_out) return 1;
    const int B = G * Np;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* lw = (double*)malloc(sizeof(double) * (size_t)Np);
    double* w = (double*)malloc(sizeof(double) * (size_t)Np);
    for (int b = 0; b < B; ++b) {
        /* statuses in the order of the plain round (a non-finite row anywhere, then the tokens,
         * then the uniforms), the log ratios gathered on the way */
        int st = OR_ROW_OK, badtok = 0;
        double lr = 0.0, l, thr;
        const int32_t* tok = tokens + (size_t)b * (K > 0 ? K : 0);
        const float* u = uniforms + (size_t)b * 2;
        double mg = INFINITY;
        for (int j = 0; j < K; ++j) {
            size_t off_p = ((size_t)b * (size_t)(K + 1) + (size_t)j) * (size_t)V;
            size_t off_q = ((size_t)b * (size_t)K + (size_t)j) * (size_t)V;
            int sp = oracle_row_probs(target, dtype, off_p, V, T, top_k, p, &l, &thr);
            int sq = oracle_row_probs(draft, dtype, off_q, V, T, top_k, q, &l, &thr);
            if (sp != OR_ROW_OK || sq != OR_ROW_OK) { st = OR_ROW_NONFINITE; continue; }
            if (tok[j] < 0 || tok[j] >= V) { badtok = 1; continue; }
            if (q[tok[j]] == 0.0) { badtok = 1; continue; } /* q never proposes d_j */
            lr += log(p[tok[j]]) - log(q[tok[j]]);
        }
        size_t off_b = ((size_t)b * (size_t)(K + 1) + (size_t)K) * (size_t)V;
        if (oracle_row_probs(target, dtype, off_b, V, T, top_k, p, &l, &thr) != OR_ROW_OK)
            st = OR_ROW_NONFINITE; /* the row the extension token is drawn from */
        if (st == OR_ROW_OK && badtok) st = OR_ROW_BAD_TOKEN;
        if (st == OR_ROW_OK && !(u[0] >= 0.0f && u[0] < 1.0f && u[1] >= 0.0f && u[1] < 1.0f))
            st = OR_ROW_BAD_UNIFORM;
        int32_t* out = out_tokens + (size_t)b * (K + 1);
        for (int j = 0; j <= K; ++j) out[j] = -1;
        if (st == OR_ROW_OK) {
            double lo, hi;
            int y = oracle_inverse_cdf(p, V, (double)u[0], &lo, &hi);
            if (y < 0) {
                st = OR_ROW_DEGENERATE;
            } else {
                for (int j = 0; j < K; ++j) out[j] = tok[j];
                out[K] = y;
                mg = fmin(fabs((double)u[0] - lo), fabs((double)u[0] - hi));
            }
        }
        row_status[b] = st;
        if (log_ratio) log_ratio[b] = (st == OR_ROW_OK) ? lr : NAN;
        logw_out[b] = (st == OR_ROW_OK) ? logw_in[b] + lr : NAN;
        if (margin) margin[b] = mg;
    }
    /* groups: ESS and resampling (step 5) */
    for (int g = 0; g < G; ++g) {
        int ok = 1;
        for (int n = 0; n < Np; ++n) {
            const int b = g * Np + n;
            if (row_status[b] != OR_ROW_OK) ok = 0;
        }
        if (!ok) {
            if (ess) ess[g] = NAN;
            if (resampled) resampled[g] = -1;
            if (ess_margin) ess_margin[g] = INFINITY;
            for (int n = 0; n < Np; ++n) {
                if (ancestors) ancestors[g * Np + n] = -1;
                logw_out[g * Np + n] = NAN;
            }
            continue;
        }
        for (int n = 0; n < Np; ++n) lw[n] = logw_out[g * Np + n]; /* logw_in + log W */
        const double e = oracle_ess(lw, Np);
        if (ess) ess[g] = e;
        if (ess_margin) ess_margin[g] = fabs(e - eta) / eta;
        const int rs = e < eta;
        if (resampled) resampled[g] = rs;
        if (rs) {
            double m = -INFINITY;
            for (int n = 0; n < Np; ++n) if (lw[n] > m) m = lw[n];
            for (int n = 0; n < Np; ++n) w[n] = exp(lw[n] - m);
            for (int n = 0; n < Np; ++n) {
                const int b = g * Np + n;
                double lo, hi;
                const double un = (double)uniforms[(size_t)b * 2 + 1];
                const int a = oracle_inverse_cdf(w, Np, un, &lo, &hi);
                if (ancestors) ancestors[b] = a;
                if (margin) margin[b] = fmin(margin[b], fmin(fabs(un - lo), fabs(un - hi)));
            }
            for (int n = 0; n < Np; ++n) logw_out[g * Np + n] = -log((double)Np);
        } else {
            for (int n = 0; n < Np; ++n)
                if (ancestors) ancestors[g * Np + n] = n;
        }
    }
    free(p);
    free(q);
    free(lw);
    free(w);
    return 0;
}
