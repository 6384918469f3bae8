// sv_plan.cuh -- the per-request acceptance scan, run by one CTA once every logit row of the
// request has its normaliser.
//
// M7.1 section 0x03 / Module 16 "The Math: Speculative Sampling": draft token x_i is accepted when
// u_i < a_i = min(1, p_i(x_i) / q_i(x_i)); M7.1 section 0x03G: the round stops at the first
// rejection A; the correction row pair is (p_A, q_A), or the bonus row p_gamma when every draft
// token is accepted (M7.1 section 0x03H).  The ratio is formed in the log2 domain in fp64:
//   log2 p_i(x) = fma(x, c, -MC_i) - log2(S_i)      (same exponent as the row's own sum)
// so that MC's rounding cancels exactly.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr double LN2 = 0.69314718055994530942;

__device__ __forceinline__ RowStats ld_rowstats(const RowStats* p)
{
    RowStats r;
    r.M = __ldcg(&p->M);
    r.MC = __ldcg(&p->MC);
    r.S = __ldcg(&p->S);
    r.thr = __ldcg(&p->thr);
    r.status = __ldcg(&p->status);
    r.klist_n = __ldcg(&p->klist_n);
    r.dense = __ldcg(&p->dense);
    r.lse = __ldcg(&p->lse);
    r.invS = __ldcg(&p->invS);
    r.lx = __ldcg(&p->lx);
    return r;
}

__device__ __forceinline__ Plan ld_plan(const Plan* p)
{
    Plan r;
    r.status = __ldcg(&p->status);
    r.A = __ldcg(&p->A);
    r.rp = __ldcg(&p->rp);
    r.rq = __ldcg(&p->rq);
    r.MCp = __ldcg(&p->MCp);
    r.MCq = __ldcg(&p->MCq);
    r.invSp = __ldcg(&p->invSp);
    r.invSq = __ldcg(&p->invSq);
    r.thrp = __ldcg(&p->thrp);
    r.thrq = __ldcg(&p->thrq);
    r.u = __ldcg(&p->u);
    return r;
}

// log2 of the processed probability of stored logit x in a row described by rs.
__device__ __forceinline__ double row_log2prob(float x, const RowStats& rs, float c, bool topk)
{
    if (topk && !(x >= rs.thr)) return -INFINITY;
    return (double)fmaf(x, c, -rs.MC) - log2(rs.S);
}

// Natural-log normaliser of logits/T over the kept tokens.  S is relative to MC = fp32(M*c); the
// exact product M*c (fp64) recovers the normaliser relative to M/T.
__device__ __forceinline__ float row_lse(const RowStats& rs, float c, double T)
{
    if (rs.status != ROW_OK) return __int_as_float(0x7fc00000);
    double exact = (double)rs.M * (double)c;
    return (float)((double)rs.M / T + log(rs.S) - LN2 * (exact - (double)rs.MC));
}

// Computes the plan of request b.  Must be called by all 32 lanes of one warp; every lane gets the
// plan.  Writes the aux outputs (lse per row, accept ratio per position).  With PRE the rows' lse,
// 1/S and log2 p(x) of their scoring tokens come from RowStats (filled by whoever finished the
// rows) instead of being computed here.
template <int DT, bool PRE = false>
__device__ Plan compute_plan_warp(const SpecParams& P, int b, bool topk)
{
    const int g = P.gamma, R = P.R, lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;

    int bad = 0, tmo = 0;
    for (int r = lane; r < R; r += 32) {
        RowStats rs = ld_rowstats(P.rstats + (size_t)b * R + r);
        if (rs.status != ROW_OK) bad = 1;
        if (rs.status == ROW_TIMEOUT) tmo = 1;
        const float lse = PRE ? (rs.status == ROW_OK ? rs.lse : __int_as_float(0x7fc00000))
                              : row_lse(rs, P.c, P.T);
        if (r <= g) {
            if (P.aux_lse_p) P.aux_lse_p[(size_t)b * (g + 1) + r] = lse;
        } else if (P.aux_lse_q) {
            P.aux_lse_q[(size_t)b * g + (r - g - 1)] = lse;
        }
    }
    const int nonfinite = __any_sync(FULL, bad);
    const int timeout = __any_sync(FULL, tmo);

    // acceptance ratios at every position
    int badtok = 0;
    int rej_first = g;
    const float* u = P.uniforms + (size_t)b * (g + 2);
    for (int i = lane; i < g; i += 32) {
        const int x = P.tokens[(size_t)b * g + i];
        double a = __longlong_as_double(0x7ff8000000000000ll);
        double plp = 0.0, plq = 0.0;
        if constexpr (PRE) {
            plp = __ldcg(&P.rstats[(size_t)b * R + i].lx);
            plq = __ldcg(&P.rstats[(size_t)b * R + g + 1 + i].lx);
        }
        if (x < 0 || x >= P.V) {
            badtok = 1;
        } else if (!nonfinite) {
            double lp, lq;
            if constexpr (PRE) {
                lp = plp;
                lq = plq;
            } else {
                const RowStats rp = ld_rowstats(P.rstats + (size_t)b * R + i);
                const RowStats rq = ld_rowstats(P.rstats + (size_t)b * R + g + 1 + i);
                const float xp = load_logit(spec_row_ptr(P, b, i), DT, x);
                const float xq = load_logit(spec_row_ptr(P, b, g + 1 + i), DT, x);
                lp = row_log2prob(xp, rp, P.c, topk);
                lq = row_log2prob(xq, rq, P.c, topk);
            }
            if (lq == -INFINITY) {
                badtok = 1;  // q(x) = 0: the draft cannot have proposed x
            } else {
                a = (lp >= lq) ? 1.0 : exp2(lp - lq);
                if (!((double)u[i] < a) && i < rej_first) rej_first = i;
            }
        }
        if (P.aux_accept) P.aux_accept[(size_t)b * g + i] = (float)a;
    }
    badtok = __any_sync(FULL, badtok);
    int badu = 0;
    for (int i = lane; i < g + 2; i += 32) {
        const float v = u[i];
        if (!(v >= 0.0f && v < 1.0f)) badu = 1;
    }
    badu = __any_sync(FULL, badu);

    Plan pl;
    pl.status = timeout ? ROW_TIMEOUT : nonfinite ? ROW_NONFINITE : badtok ? ROW_BAD_TOKEN : badu ? ROW_BAD_UNIFORM : ROW_OK;
    pl.A = __reduce_min_sync(FULL, rej_first);
    pl.rp = (pl.A < g) ? pl.A : g;
    pl.rq = (pl.A < g) ? g + 1 + pl.A : -1;
    const RowStats sp = ld_rowstats(P.rstats + (size_t)b * R + pl.rp);
    pl.MCp = sp.MC;
    pl.invSp = PRE ? sp.invS : (float)(1.0 / sp.S);
    pl.thrp = sp.thr;
    if (pl.rq >= 0) {
        const RowStats sq = ld_rowstats(P.rstats + (size_t)b * R + pl.rq);
        pl.MCq = sq.MC;
        pl.invSq = PRE ? sq.invS : (float)(1.0 / sq.S);
        pl.thrq = sq.thr;
    } else {
        pl.MCq = 0.f;
        pl.invSq = 0.f;
        pl.thrq = 0.f;
    }
    pl.u = (double)u[(pl.A < g) ? g : g + 1];
    return pl;
}

__device__ __forceinline__ void st_plan(Plan* dst, const Plan& pl) { *dst = pl; }

// Residual mass r(v) = max(p(v) - q(v), 0) (or p(v) for the bonus draw) of one vector of the row
// pair.  Explicit round-to-nearest intrinsics keep the value bit-identical wherever it is
// recomputed (no contraction into FMA by the compiler).
template <int DT, int VEC>
__device__ __forceinline__ void residual_vec(const char* rowp, const char* rowq, long long v,
                                             const Plan& pl, float c, bool topk, float (&r)[VEC])
{
    float xp[VEC];
    load_vec<DT, VEC>(rowp, v, xp);
    if (rowq) {
        float xq[VEC];
        load_vec<DT, VEC>(rowq, v, xq);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float pp = __fmul_rn(ex2(fmaf(xp[e], c, -pl.MCp)), pl.invSp);
            float qq = __fmul_rn(ex2(fmaf(xq[e], c, -pl.MCq)), pl.invSq);
            if (topk) {
                if (!(xp[e] >= pl.thrp)) pp = 0.f;
                if (!(xq[e] >= pl.thrq)) qq = 0.f;
            }
            r[e] = fmaxf(__fsub_rn(pp, qq), 0.f);
        }
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float pp = __fmul_rn(ex2(fmaf(xp[e], c, -pl.MCp)), pl.invSp);
            if (topk && !(xp[e] >= pl.thrp)) pp = 0.f;
            r[e] = pp;
        }
    }
}

// fixed-order pairwise sum of a small array
template <int N>
__device__ __forceinline__ float tree_sum(const float (&r)[N])
{
    if constexpr (N == 1) {
        return r[0];
    } else {
        float t[N];
#pragma unroll
        for (int i = 0; i < N; ++i) t[i] = r[i];
#pragma unroll
        for (int w = 1; w < N; w <<= 1)
#pragma unroll
            for (int i = 0; i + w < N; i += 2 * w) t[i] = __fadd_rn(t[i], t[i + w]);
        return t[0];
    }
}

}  // namespace sv
