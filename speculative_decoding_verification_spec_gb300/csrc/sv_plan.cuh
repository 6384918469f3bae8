// sv_plan.cuh -- the per-request acceptance scan, run by one CTA once every logit row of the
// request has its normaliser.
//
// M7.1 section 0x03 / Module 16 "The Math: Speculative Sampling": draft token x_i is accepted when
// u_i < a_i = min(1, p_i(x_i) / q_i(x_i)); M7.1 section 0x03G: the round stops at the first
// rejection A; the correction row pair is (p_A, q_A), or the bonus row p_gamma when every draft
// token is accepted (M7.1 section 0x03H).  The ratio is formed in the log2 domain, in pairs of
// floats (about 48 bits):
//   log2 p_i(x) = fma(x, c, -MC_i) - log2(S_i)      (same exponent as the row's own sum)
// so that MC's rounding cancels exactly.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr double LN2 = 0.69314718055994530942;
constexpr float LN2_HI = 0.693147182464599609375f;   // fp32(ln 2)
constexpr float LN2_LO = -1.904654299957768e-09f;    // ln 2 - LN2_HI
constexpr float LOG2E_F = 1.44269504088896340736f;

// The normaliser fields of a row (one thread): from its maximum M, MC = fp32(M c), the sum
// S = hi + lo of 2^(fma(x, c, -MC)) over its (kept) tokens, and the logit xtok of the token it
// scores (tok_ok), kept when xtok >= thr:
//   lse = M / T + ln S - ln 2 (M c - MC)       natural log, over logits / T
//   lx  = fma(xtok, c, -MC) - log2 S           log2 p(xtok)
// log2 S = e + log2 m + log2(1 + lo / hi) with hi = m 2^e, m in [0.5, 1): the fp32 log2 of m has an
// absolute error of about 1e-7, and the integer e joins it exactly.  M c - MC, the rounding error
// of MC, is exact as fma(M, c, -MC).  Everything is carried in pairs of floats; only lx and S are
// widened to fp64 at the end.
__device__ __forceinline__ void row_norm(RowStats& st, float M, float MC, DFloat S, const SpecParams& P,
                                         bool tok_ok, float xtok, float thr)
{
    int e;
    const float m = frexpf(S.hi, &e);
    const float l2m = __fadd_rn(log2f(m), __fmul_rn(__fdiv_rn(S.lo, S.hi), LOG2E_F));
    DFloat l2S;
    two_sum((float)e, l2m, l2S.hi, l2S.lo);
    const float err = fmaf(M, P.c, -MC);
    const float a_hi = __fmul_rn(M, P.invT_hi);
    const DFloat a = df_make(a_hi, fmaf(M, P.invT_lo, fmaf(M, P.invT_hi, -a_hi)));
    DFloat d;
    d.hi = -err;
    d.lo = 0.f;
    const DFloat lse = df_add(a, df_mul(df_add(l2S, d), LN2_HI, LN2_LO));
    st.lse = __fadd_rn(lse.hi, lse.lo);
    st.invS = __frcp_rn(__fadd_rn(S.hi, S.lo));
    st.S = df_to_double(S);
    if (tok_ok) {
        const float t0 = fmaf(xtok, P.c, -MC);
        if (xtok >= thr && isfinite(t0)) {
            DFloat t;
            two_sum(t0, -l2S.hi, t.hi, t.lo);
            const DFloat lx = df_make(t.hi, __fsub_rn(t.lo, l2S.lo));
            st.lx_hi = lx.hi;
            st.lx_lo = lx.lo;
        } else {
            st.lx_hi = (xtok >= thr) ? t0 : NEG_INF;  // a -inf logit: p(x) = 0
            st.lx_lo = 0.f;
        }
    }
}

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
    r.lx_hi = __ldcg(&p->lx_hi);
    r.lx_lo = __ldcg(&p->lx_lo);
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

// The accept ratio a = min(1, 2^(lp - lq)) of log2 probabilities lp <= 0 and a finite lq.  The
// exponent's integer part n is applied as an exact power-of-two scale and 2^f of its fraction f in
// [0, 1) comes from the fp32 ex2 unit: relative error a few 1e-7, well inside the 1e-6 decision
// margin of the matching rules, with four fp64 operations (the fp64 pipe is very slow on this
// part).  a stays > 0 whenever p(x) > 0, so a uniform of exactly 0 is still accepted.
__device__ __forceinline__ double accept_ratio(double lp, double lq)
{
    if (!(lp < lq)) return 1.0;
    if (lp == -INFINITY) return 0.0;
    const double d = lp - lq;  // < 0
    const double n = floor(d);
    const float f = (float)(d - n);
    const int ni = (n < -1100.0) ? -1100 : (int)n;
    const double scale = (ni >= -1022) ? __longlong_as_double((long long)(ni + 1023) << 52)
                                       : 4.9406564584124654e-324;  // the smallest positive double
    return (double)ex2(f) * scale;
}

// The same ratio from log2 probabilities held as pairs of floats (no fp64 at all): the difference
// is formed exactly as a pair, its integer part n becomes an fp32 power of two and ex2 takes the
// fraction.  Returns a float > 0 whenever p(x) > 0.
__device__ __forceinline__ float accept_ratio_df(DFloat lp, DFloat lq)
{
    if (!(lp.hi < lq.hi || (lp.hi == lq.hi && lp.lo < lq.lo))) return 1.f;
    if (lp.hi == NEG_INF) return 0.f;
    float s, e;
    two_sum(lp.hi, -lq.hi, s, e);
    const DFloat d = df_make(s, __fadd_rn(e, __fsub_rn(lp.lo, lq.lo)));  // < 0
    const float n = floorf(d.hi);
    const float m = ex2(__fadd_rn(__fsub_rn(d.hi, n), d.lo));
    const int ni = (n < -200.f) ? -200 : (int)n;
    if (ni >= -126) return __fmul_rn(m, __int_as_float((ni + 127) << 23));
    if (ni >= -150) return __fmul_rn(__fmul_rn(m, __int_as_float((ni + 24 + 127) << 23)), 5.9604644775390625e-8f);
    return 1.40129846e-45f;  // the smallest positive float
}

__device__ __forceinline__ RowStats blank_rowstats()
{
    RowStats r;
    r.M = NEG_INF; r.MC = NEG_INF; r.S = 0.0; r.thr = NEG_INF;
    r.status = ROW_OK; r.klist_n = -1; r.dense = 0;
    r.lse = 0.f; r.invS = 0.f; r.lx_hi = 0.f; r.lx_lo = 0.f;
    return r;
}

__device__ __forceinline__ RowStats shfl_rowstats(const RowStats& r, int src)
{
    const unsigned FULL = 0xffffffffu;
    RowStats o;
    o.M = __shfl_sync(FULL, r.M, src);
    o.MC = __shfl_sync(FULL, r.MC, src);
    o.S = __shfl_sync(FULL, r.S, src);
    o.thr = __shfl_sync(FULL, r.thr, src);
    o.status = __shfl_sync(FULL, r.status, src);
    o.klist_n = __shfl_sync(FULL, r.klist_n, src);
    o.dense = __shfl_sync(FULL, r.dense, src);
    o.lse = __shfl_sync(FULL, r.lse, src);
    o.invS = __shfl_sync(FULL, r.invS, src);
    o.lx_hi = __shfl_sync(FULL, r.lx_hi, src);
    o.lx_lo = __shfl_sync(FULL, r.lx_lo, src);
    return o;
}

// The plan of request b from its rows' statistics held one row per lane (row r in lane r; R =
// 2 gamma + 1 <= 32), with the lse, 1/S and log2 p(x) of the scoring tokens filled in by whoever
// finished the rows.  One warp, every lane gets the plan; writes the aux outputs.  The request's
// tokens and uniforms are read here; everything else comes by shuffles.
__device__ __forceinline__ Plan plan_from_lanes(const SpecParams& P, int b, const RowStats& rs)
{
    const int g = P.gamma, R = P.R, lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const int x = (lane < g) ? __ldg(P.tokens + (size_t)b * g + lane) : 0;
    const int nu = P.smc ? 2 : g + 2;  // uniforms per request
    const float uu = (lane < nu) ? __ldg(P.uniforms + (size_t)b * nu + lane) : 0.f;
    const bool row = lane < R;
    const int nonfinite = __any_sync(FULL, row && rs.status != ROW_OK);
    const int timeout = __any_sync(FULL, row && rs.status == ROW_TIMEOUT);
    if (row) {
        const float lse = (rs.status == ROW_OK) ? rs.lse : __int_as_float(0x7fc00000);
        if (lane <= g) {
            if (P.aux_lse_p) P.aux_lse_p[(size_t)b * (g + 1) + lane] = lse;
        } else if (P.aux_lse_q) {
            P.aux_lse_q[(size_t)b * g + (lane - g - 1)] = lse;
        }
    }
    // position i = lane < g: log2 p_i(x_i) is this lane's row, log2 q_i(x_i) row g + 1 + i's
    DFloat lp, lq;
    lp.hi = rs.lx_hi;
    lp.lo = rs.lx_lo;
    lq.hi = __shfl_sync(FULL, rs.lx_hi, (lane + g + 1) & 31);
    lq.lo = __shfl_sync(FULL, rs.lx_lo, (lane + g + 1) & 31);
    int badtok = 0;
    bool reject = false;
    DFloat lr = df_make(0.f, 0.f);  // SMC: log2 p(x) - log2 q(x) of this position
    if (lane < g) {
        float a = __int_as_float(0x7fc00000);
        if (x < 0 || x >= P.V) {
            badtok = 1;
        } else if (!nonfinite) {
            if (lq.hi == NEG_INF) {
                badtok = 1;  // q(x) = 0: the draft cannot have proposed x
            } else {
                a = accept_ratio_df(lp, lq);
                reject = !P.smc && !(uu < a);
                lr = df_add(lp, df_make(-lq.hi, -lq.lo));
            }
        }
        if (P.aux_accept) P.aux_accept[(size_t)b * g + lane] = a;
    }
    badtok = __any_sync(FULL, badtok);
    const int badu = __any_sync(FULL, lane < nu && !(uu >= 0.0f && uu < 1.0f));
    const unsigned rej = __ballot_sync(FULL, reject);
    if (P.smc) {  // the block log-ratio, natural log (M16 "The Math: Reweight, Don't Reject")
        const DFloat l2 = warp_sum_df(lr);
        const DFloat ln = df_mul(l2, LN2_HI, LN2_LO);
        const bool okr = !nonfinite && !badtok && !badu;
        if (lane == 0) {
            const float v = okr ? ln.hi + ln.lo : __int_as_float(0x7fc00000);
            if (P.smc_log_ratio) P.smc_log_ratio[b] = v;
            P.smc_logw[b] = okr ? __ldg(P.smc_logw_in + b) + v : __int_as_float(0x7fc00000);
        }
    }

    Plan pl;
    pl.status = timeout ? ROW_TIMEOUT : nonfinite ? ROW_NONFINITE : badtok ? ROW_BAD_TOKEN : badu ? ROW_BAD_UNIFORM : ROW_OK;
    pl.A = rej ? __ffs(rej) - 1 : g;
    pl.rp = (pl.A < g) ? pl.A : g;
    pl.rq = (pl.A < g) ? g + 1 + pl.A : -1;
    const RowStats sp = shfl_rowstats(rs, pl.rp);
    const RowStats sq = shfl_rowstats(rs, pl.rq >= 0 ? pl.rq : 0);
    pl.MCp = sp.MC;
    pl.invSp = sp.invS;
    pl.thrp = sp.thr;
    pl.MCq = (pl.rq >= 0) ? sq.MC : 0.f;
    pl.invSq = (pl.rq >= 0) ? sq.invS : 0.f;
    pl.thrq = (pl.rq >= 0) ? sq.thr : 0.f;
    pl.u = (double)__shfl_sync(FULL, uu, P.smc ? 0 : (pl.A < g) ? g : g + 1);
    return pl;
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
    if constexpr (PRE) {
        if (R <= 32) {  // every row's statistics in one round of loads, one row per lane
            RowStats rs = blank_rowstats();
            if (lane < R) rs = ld_rowstats(P.rstats + (size_t)b * R + lane);
            return plan_from_lanes(P, b, rs);
        }
    }

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
    const int nu = P.smc ? 2 : g + 2;  // uniforms per request
    const float* u = P.uniforms + (size_t)b * nu;
    double lrsum = 0.0;  // SMC: sum of log2 p(x) - log2 q(x) over this lane's positions
    for (int i = lane; i < g; i += 32) {
        const int x = P.tokens[(size_t)b * g + i];
        double a = __longlong_as_double(0x7ff8000000000000ll);
        double plp = 0.0, plq = 0.0;
        if constexpr (PRE) {
            const RowStats* rp = P.rstats + (size_t)b * R + i;
            const RowStats* rq = P.rstats + (size_t)b * R + g + 1 + i;
            plp = (double)__ldcg(&rp->lx_hi) + (double)__ldcg(&rp->lx_lo);
            plq = (double)__ldcg(&rq->lx_hi) + (double)__ldcg(&rq->lx_lo);
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
                const float xp = masked_logit(P, b, i, DT, x);
                const float xq = masked_logit(P, b, g + 1 + i, DT, x);
                lp = row_log2prob(xp, rp, P.c, topk);
                lq = row_log2prob(xq, rq, P.c, topk);
            }
            if (lq == -INFINITY) {
                badtok = 1;  // q(x) = 0: the draft cannot have proposed x
            } else {
                a = accept_ratio(lp, lq);
                if (!P.smc && !((double)u[i] < a) && i < rej_first) rej_first = i;
                lrsum += lp - lq;
            }
        }
        if (P.aux_accept) P.aux_accept[(size_t)b * g + i] = (float)a;
    }
    badtok = __any_sync(FULL, badtok);
    int badu = 0;
    for (int i = lane; i < nu; i += 32) {
        const float v = u[i];
        if (!(v >= 0.0f && v < 1.0f)) badu = 1;
    }
    badu = __any_sync(FULL, badu);
    if (P.smc) {  // the block log-ratio, natural log (M16 "The Math: Reweight, Don't Reject")
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lrsum += __shfl_xor_sync(FULL, lrsum, o);
        const bool okr = !nonfinite && !badtok && !badu;
        if (lane == 0) {
            const float v = okr ? (float)(lrsum * LN2) : __int_as_float(0x7fc00000);
            if (P.smc_log_ratio) P.smc_log_ratio[b] = v;
            P.smc_logw[b] = okr ? P.smc_logw_in[b] + v : __int_as_float(0x7fc00000);
        }
    }

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
    pl.u = (double)u[P.smc ? 0 : (pl.A < g) ? g : g + 1];
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
