// sv_draw.cuh -- the correction / bonus draw of exact speculative sampling, shared by the residual
// kernels of the plain, grammar-masked and top-p paths (sv_softmax.cu, sv_topp.cu).
//
// M7.1 section 0x03C: after the first rejection at position A the token is drawn from the normalised
// positive residual max(p_A - q_A, 0); section 0x03H: when every draft token is accepted, the bonus
// is drawn from p_gamma.  The draw is an inverse CDF in ascending token order on the unnormalised
// mass: the first token whose running mass passes u * Z.  The mass of every vector is formed by
// residual_from (bit-identical wherever it is recomputed); a row pair is summed per segment of 32
// vectors, the segment sums are scanned to find the segment holding u * Z, and the token is resolved
// inside that segment.
#pragma once

#include "sv_plan.cuh"

namespace sv {

// Rows of the first pin_pairs row pairs (target row i and draft row i) are read with the L2
// evict-normal policy and the others evict-first, so that the row pair a correction rereads tends
// to still be in L2: the first positions are the likeliest rejections.
__device__ __forceinline__ bool pinned_row(const SpecParams& P, int r)
{
    if (r == P.gamma) return P.gamma < P.pin_pairs;  // the bonus row matters when all are accepted
    const int pos = (r < P.gamma) ? r : r - P.gamma - 1;
    return pos < P.pin_pairs;
}

// Top-p: a row keeps the tokens whose stored logit is >= its threshold (pl.thrp for the p row,
// pl.thrq for the q row); the rest become -inf.  The plain and masked paths carry -inf thresholds,
// for which this changes nothing.
template <int VEC>
__device__ __forceinline__ void apply_thresholds(float (&xp)[VEC], float (&xq)[VEC], bool has_q,
                                                 const Plan& pl)
{
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        if (!(xp[e] >= pl.thrp)) xp[e] = NEG_INF;
        if (has_q && !(xq[e] >= pl.thrq)) xq[e] = NEG_INF;
    }
}

// residual mass of one vector from already-loaded values (bit-identical wherever recomputed)
template <int VEC>
__device__ __forceinline__ void residual_from(const float (&xp)[VEC], const float (&xq)[VEC],
                                              bool has_q, const Plan& pl, float c, float (&r)[VEC])
{
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float pp = __fmul_rn(ex2(fmaf(xp[e], c, -pl.MCp)), pl.invSp);
        if (has_q) {
            const float qq = __fmul_rn(ex2(fmaf(xq[e], c, -pl.MCq)), pl.invSq);
            r[e] = fmaxf(__fsub_rn(pp, qq), 0.f);
        } else {
            r[e] = pp;
        }
    }
}

// Resolve the token inside the segment of 32 vectors starting at vbase (one per lane), given the
// mass t_local still to pass within it.  Runs in one warp; returns the token in every lane.  The
// scans inside the segment are fp32: the segment's mass is a small part of the total, so their
// rounding stays far below the 1e-6 decision margin.
template <int DT, int VEC>
__device__ int resolve_in_segment(const SpecParams& P, const char* rowp, const char* rowq,
                                  const uint32_t* mrow, const Plan& pl, long long vbase,
                                  double t_local)
{
    const int lane = threadIdx.x & 31;
    const long long v = vbase + lane;
    float r[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = 0.f;
    if (v < P.nvec) {
        float xp[VEC], xq[VEC];
        load_vec<DT, VEC>(rowp, v, xp);
        if (rowq) {
            load_vec<DT, VEC>(rowq, v, xq);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) xq[e] = 0.f;
        }
        if (mrow) {
            const uint32_t bits = allowed_bits<VEC>(mrow, v);
            mask_vals<VEC>(xp, bits);
            mask_vals<VEC>(xq, bits);
        }
        apply_thresholds<VEC>(xp, xq, rowq != nullptr, pl);
        residual_from<VEC>(xp, xq, rowq != nullptr, pl, P.c, r);
    }
    const float tl = (float)t_local;
    const float ls = tree_sum(r);
    const float incl = warp_incl_scan(ls);
    const float start = incl - ls;
    const unsigned hit = __ballot_sync(0xffffffffu, tl < incl && ls > 0.f);
    int owner;
    if (hit) {
        owner = __ffs(hit) - 1;
    } else {  // rounding left t_local past the segment: its last positive entry
        const unsigned pos = __ballot_sync(0xffffffffu, ls > 0.f);
        owner = pos ? 31 - __clz(pos) : 0;
    }
    int tok = -1;
    if (lane == owner) {
        float run = start;
        int last_pos = -1;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            if (r[e] > 0.f) last_pos = e;
            run += r[e];
            if (tok < 0 && hit && tl < run && r[e] > 0.f) tok = e;
        }
        if (tok < 0) tok = last_pos;
        tok = (tok < 0) ? -1 : (int)(v * VEC + tok);
    }
    return __shfl_sync(0xffffffffu, tok, owner);
}

// Request b's draw from its segment sums (one warp).  Returns the token, -1 if degenerate.  With up
// to 32 x DPL segments every lane holds its block of sums in registers (one round of loads), adds
// them pairwise in fp32 and the lane totals are scanned in fp64.
constexpr int DPL = 16;
template <int DT, int VEC>
__device__ int draw_from_segments(const SpecParams& P, int b, const Plan& pl, const char* rowp,
                                  const char* rowq)
{
    const int lane = threadIdx.x & 31;
    const float* segs = P.segs + (size_t)b * P.nseg;
    const uint32_t* mrow = P.mask ? spec_mask_row(P, b, pl.rp) : nullptr;
    const int per = (P.nseg + 31) / 32;
    const int s0 = min(lane * per, P.nseg), s1 = min(s0 + per, P.nseg);
    if (per <= DPL) {
        float v[DPL];
#pragma unroll
        for (int k = 0; k < DPL; ++k) v[k] = (s0 + k < s1) ? __ldcg(segs + s0 + k) : 0.f;
        const float lsum = tree_sum(v);
        const double mine = (double)lsum;
        const double incl = warp_incl_scan(mine);
        const double Z = __shfl_sync(0xffffffffu, incl, 31);
        if (!(Z > 0.0) || !isfinite(Z)) return -1;
        const double excl = incl - mine;
        const double t = pl.u * Z;
        unsigned own = __ballot_sync(0xffffffffu, mine > 0.0 && t < excl + mine);
        if (!own) {  // rounding: the last lane holding positive mass
            const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.0);
            own = pos ? (1u << (31 - __clz(pos))) : 0u;
            if (!own) return -1;
        }
        const int owner = __ffs(own) - 1;
        int seg = -1;
        double base = 0.0;
        if (lane == owner) {
            const float tr = (float)(t - excl);  // mass still to pass inside this lane's block
            float run = 0.f, lastrun = 0.f;
            int lastpos = -1;
            float before = 0.f;
#pragma unroll
            for (int k = 0; k < DPL; ++k) {
                if (seg < 0 && v[k] > 0.f) {
                    lastpos = s0 + k;
                    lastrun = run;
                    if (tr < run + v[k]) {
                        seg = s0 + k;
                        before = run;
                    }
                }
                run += v[k];
            }
            if (seg < 0) {
                seg = lastpos;
                before = lastrun;
            }
            base = excl + (double)before;
        }
        seg = __shfl_sync(0xffffffffu, seg, owner);
        base = __shfl_sync(0xffffffffu, base, owner);
        if (seg < 0) return -1;
        return resolve_in_segment<DT, VEC>(P, rowp, rowq, mrow, pl, (long long)seg * SEGV, t - base);
    }
    // more segments than the registers hold: each lane's block in batches of eight
    double mine = 0.0;
    for (int q0 = s0; q0 < s1; q0 += 8) {
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = (q0 + t < s1) ? __ldcg(segs + q0 + t) : 0.f;
        mine += (double)tree_sum(v);
    }
    const double incl = warp_incl_scan(mine);
    const double Z = __shfl_sync(0xffffffffu, incl, 31);
    if (!(Z > 0.0) || !isfinite(Z)) return -1;
    const double excl = incl - mine;
    const double t = pl.u * Z;
    unsigned own = __ballot_sync(0xffffffffu, mine > 0.0 && t < excl + mine);
    if (!own) {
        const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.0);
        own = pos ? (1u << (31 - __clz(pos))) : 0u;
        if (!own) return -1;
    }
    const int owner = __ffs(own) - 1;
    int seg = -1;
    double base = 0.0;
    if (lane == owner) {
        double run = 0.0, lastbase = excl;
        int lastpos = -1;
        for (int q = s0; q < s1 && seg < 0; ++q) {
            const double sv = (double)__ldcg(segs + q);
            if (sv > 0.0) { lastpos = q; lastbase = excl + run; }
            if (sv > 0.0 && t < excl + run + sv) { seg = q; base = excl + run; }
            else run += sv;
        }
        if (seg < 0) { seg = lastpos; base = lastbase; }
    }
    seg = __shfl_sync(0xffffffffu, seg, owner);
    base = __shfl_sync(0xffffffffu, base, owner);
    if (seg < 0) return -1;
    return resolve_in_segment<DT, VEC>(P, rowp, rowq, mrow, pl, (long long)seg * SEGV, t - base);
}

}  // namespace sv
