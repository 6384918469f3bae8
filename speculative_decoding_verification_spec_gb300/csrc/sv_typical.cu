// sv_typical.cu -- tree verify with typical acceptance.
//
// Module 16 "Verify the Tree": Medusa's sampling mode replaces the greedy check of each candidate by
// typical acceptance: the candidate passes when the target's probability of its token clears
// min(eps, delta exp(-H)), H the entropy of the target's distribution at that position.  The walk
// over the tree (valid = passes and parent valid, deepest valid node wins) is the greedy tree's;
// the token after the accepted path is drawn from the target's distribution at the accepted node.
//
// Kernel 1 (row statistics), one pass over every row of every request: per (row, chunk, warp) the
// maximum M, S = sum 2^y and E = sum 2^y y with y = x c - fp32(M c) and c = log2(e) / T, so that
//   p_v = 2^y_v / S,   H = -sum p ln p = ln 2 (log2 S - E / S).
// Rows of 16-byte vectors stream through the bulk-copy ring (typical_stream_kernel); any other
// layout uses plain loads (typical_stats_kernel).  Partials with maxima MC_k merge at the row's MC
// with d_k = MC_k - MC: S = sum 2^d_k S_k, E = sum 2^d_k (E_k + d_k S_k).
//
// Kernel 2 (typical_finish_kernel), one thread-block cluster of TYP_CL CTAs per request: the rows'
// statistics (shared among the CTAs), every node's test and the walk (CTA 0), then the inverse-CDF
// draw over the accepted node's row: per segment of 32 vectors the mass sum 2^y (the CTAs take a run
// of segments each), a scan of the segment sums in index order (pairs of floats), and the token
// resolved inside its segment (CTA 0).
#include <cooperative_groups.h>

#include "sv_plan.cuh"
#include "sv_tree_walk.cuh"
#include "sv_typical.cuh"

namespace cg = cooperative_groups;

namespace sv {

__device__ __forceinline__ const char* typ_row(const TypicalParams& P, int b, int r)
{
    return reinterpret_cast<const char*>(P.t.logits) +
           ((size_t)b * P.t.R + r) * (size_t)P.t.V * esize(P.t.dtype);
}

// one element's share of S and E: e = 2^y and e * y (0 for a -inf logit, whose y is -inf)
__device__ __forceinline__ void typ_acc(float x, float c, float MC, float& s, float& e)
{
    const float y = fmaf(x, c, -MC);
    const float w = ex2(y);
    s += w;
    e = fmaf(w, fmaxf(y, -3.0e38f), e);
}

// a < b for values held as pairs of floats (normalised: |lo| <= ulp(hi) / 2)
__device__ __forceinline__ bool df_lt(DFloat a, DFloat b)
{
    return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// ---------------------------------------------------------------- kernel 1: row statistics

// consumer groups per CTA of the streaming kernel (see ring_produce): two, in one CTA per SM.  Its
// chunks cost the most arithmetic of the streams, and two CTAs per SM finished unevenly.
constexpr int TYP_GROUPS = 2;

// Persistent CTAs over 32 KB chunks of the rows, fetched by bulk copies into shared-memory rings
// (a producer warp fills them, the consumer warps of each group release each stage on its "empty"
// mbarrier).  Each consumer warp writes one partial per chunk.  NaN or +inf anywhere makes the
// partial's S NaN.
template <int DT>
__global__ void __launch_bounds__(stream_threads<TYP_GROUPS>(), 1) typical_stream_kernel(TypicalParams P)
{
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    constexpr int ES = (DT == DT_BF16) ? 2 : 4;
    constexpr int CHUNK = NT * STREAM_NV * VEC;
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) uint64_t full[TYP_GROUPS * STREAM_STAGES];
    __shared__ __align__(8) uint64_t empty[TYP_GROUPS * STREAM_STAGES];
    __shared__ int sfail;

    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int S1 = P.S1, V = P.t.V;
    const int nch = P.t.B * P.t.R * S1;  // < 2^31 (checked on the host)
    const float c = P.c;
    if (tid == 0) {
        sfail = 0;
        for (int s = 0; s < TYP_GROUPS * STREAM_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == TYP_GROUPS * WARPS) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            ring_produce<TYP_GROUPS>(full, empty, &sfail, nch, P.t.wait_limit, [&](int s, int id) {
                const int row = id / S1, ci = id - row * S1;
                const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, V);
                bulk_load(ring + (size_t)s * NT * STREAM_NV,
                          reinterpret_cast<const char*>(P.t.logits) + ((size_t)row * V + cbase) * ES,
                          (unsigned)(cend - cbase) * ES, &full[s], pol);
            });
        }
        return;
    }
    const StreamGroup<TYP_GROUPS> sg;
    uint64_t* gfull = full + sg.g * STREAM_STAGES;
    uint64_t* gempty = empty + sg.g * STREAM_STAGES;
    const uint4* gring = ring + (size_t)sg.g * STREAM_STAGES * NT * STREAM_NV;

    bool failed = false;
    int stg = 0;
    unsigned phase = 0;
    for (int id = sg.vb, it = 0; id < nch; id += sg.stride, ++it) {
        if (it > 0 && ++stg == STREAM_STAGES) {
            stg = 0;
            phase ^= 1u;
        }
        const int row = id / S1, ci = id - row * S1;
        const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, V);
        if (!failed && *reinterpret_cast<volatile int*>(&sfail)) failed = true;
        bool ok = !failed && mbar_wait(&gfull[stg], phase, P.t.wait_limit);
        uint4 w[STREAM_NV];
        const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
        const uint4* sb = gring + (size_t)stg * NT * STREAM_NV + sg.t;
#pragma unroll
        for (int j = 0; j < STREAM_NV; ++j) {
            w[j] = make_uint4(pad, pad, pad, pad);
            if (ok && cbase + (j * NT + sg.t) * VEC < cend) w[j] = lds128(sb + j * NT);
        }
        ok = __all_sync(FULL, ok);
        if (ok) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gempty[stg]);
        } else if (!failed) {
            failed = true;
            if (lane == 0) *reinterpret_cast<volatile int*>(&sfail) = 1;
        }
        TypPartial pt;
        if (failed) {
            pt.M = __int_as_float(0x7fc00000);  // the chunk was not read: S < 0 marks a timeout
            pt.MC = pt.M;
            pt.S = -1.f;
            pt.E = 0.f;
        } else {
            float m;
            if constexpr (DT == DT_BF16) {
                uint32_t pm = w[0].x;
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) {
                    pm = bmax2(pm, w[j].x); pm = bmax2(pm, w[j].y);
                    pm = bmax2(pm, w[j].z); pm = bmax2(pm, w[j].w);
                }
                m = fmaxf(bf16lo(pm), bf16hi(pm));
            } else {
                m = NEG_INF;
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j)
                    m = fmaxf(fmaxf(m, __uint_as_float(w[j].x)), fmaxf(fmaxf(__uint_as_float(w[j].y),
                            __uint_as_float(w[j].z)), __uint_as_float(w[j].w)));
            }
            const float M = warp_max(m);
            const float MC = __fmul_rn(M, c);
            // s0, e0 take the low elements of each word (fp32: words x and z), s1, e1 the high ones
            // (y and w), two at a time with the packed fp32 instructions (each half rounds as the
            // scalar one would).  A -inf logit is raised to -1e30 first (NaN kept), so that its
            // y is finite and its e * y is 0, as typ_acc's clamp of y makes it.
            unsigned long long s01 = 0ull, e01 = 0ull;
            if (M != NEG_INF) {
                const unsigned long long c2 = f2_pack(c, c), nmc2 = f2_pack(-MC, -MC);
                auto acc2 = [&](float lo, float hi) {
                    const unsigned long long y2 = f2_fma(f2_pack(lo, hi), c2, nmc2);
                    float ylo, yhi;
                    f2_unpack(y2, ylo, yhi);
                    const unsigned long long w2 = f2_pack(ex2(ylo), ex2(yhi));
                    s01 = f2_add(s01, w2);
                    e01 = f2_fma(w2, y2, e01);
                };
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) {
                    if constexpr (DT == DT_BF16) {
                        constexpr uint32_t FLOOR2 = 0xf149f149u;  // bf16 -9.95e29, twice
                        const uint32_t q[4] = {bmax2_nan(w[j].x, FLOOR2), bmax2_nan(w[j].y, FLOOR2),
                                               bmax2_nan(w[j].z, FLOOR2), bmax2_nan(w[j].w, FLOOR2)};
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc2(bf16lo(q[k]), bf16hi(q[k]));
                    } else {
                        const float fl = -1.0e30f;
                        acc2(fmax_nan(__uint_as_float(w[j].x), fl), fmax_nan(__uint_as_float(w[j].y), fl));
                        acc2(fmax_nan(__uint_as_float(w[j].z), fl), fmax_nan(__uint_as_float(w[j].w), fl));
                    }
                }
            }
            float s0, s1, e0, e1;
            f2_unpack(s01, s0, s1);
            f2_unpack(e01, e0, e1);
            pt.M = M;
            pt.MC = MC;
            pt.S = warp_sum(s0 + s1);
            pt.E = warp_sum(e0 + e1);
        }
        if (lane == 0) P.partials[((size_t)row * S1 + ci) * WARPS + sg.w] = pt;
    }
}

// Scalar path (rows that are not 16-byte aligned): one warp per (row, slice of TYP_SLICE elements),
// plain loads, the slice's maximum first and then its sums.
template <int DT>
__global__ void __launch_bounds__(NT) typical_stats_kernel(TypicalParams P)
{
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long nt = (long long)P.t.B * P.t.R * P.S1;
    const long long gw = ((long long)blockIdx.x * NT + threadIdx.x) >> 5;
    const long long step = ((long long)gridDim.x * NT) >> 5;
    for (long long t = gw; t < nt; t += step) {
        const int row = (int)(t / P.S1), sl = (int)(t - (long long)row * P.S1);
        const char* rp = reinterpret_cast<const char*>(P.t.logits) + (size_t)row * P.t.V * esize(DT);
        const int v0 = sl * TYP_SLICE, v1 = min(v0 + TYP_SLICE, P.t.V);
        float m = NEG_INF;
        int nan = 0;
        for (int v = v0 + lane; v < v1; v += 32) {
            const float x = load_logit(rp, DT, v);
            if (x != x) nan = 1;
            m = fmaxf(m, x);
        }
        const float M = warp_max(m);
        const float MC = __fmul_rn(M, P.c);
        float s = 0.f, e = 0.f;
        if (M != NEG_INF)
            for (int v = v0 + lane; v < v1; v += 32) typ_acc(load_logit(rp, DT, v), P.c, MC, s, e);
        nan = __any_sync(0xffffffffu, nan);
        TypPartial pt;
        pt.M = M;
        pt.MC = MC;
        pt.S = nan ? __int_as_float(0x7fc00000) : warp_sum(s);
        pt.E = warp_sum(e);
        if (lane == 0) P.partials[(size_t)row * P.S1 + sl] = pt;
    }
}

// ---------------------------------------------------------------- kernel 2: per request

size_t typical_finish_smem(int N, int nseg)
{
    // par, tok, depth, valid, match [N] ints; MC, log2 S, H [N+1] floats; segment sums [nseg];
    // each node's token logit [N] floats
    return (size_t)5 * N * sizeof(int32_t) + (size_t)3 * (N + 1) * sizeof(float) +
           (size_t)nseg * sizeof(float) + (size_t)N * sizeof(float);
}

// The mass 2^y of each element of vector v of a row (0 past the row's end): recomputed bit for bit
// wherever it is needed.
template <int DT, int VEC>
__device__ __forceinline__ void typ_mass(const char* row, long long v, long long nvec, float c,
                                         float MC, float (&r)[VEC])
{
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = 0.f;
    if (v < nvec) {
        float x[VEC];
        load_vec<DT, VEC>(row, v, x);
#pragma unroll
        for (int e = 0; e < VEC; ++e) r[e] = ex2(fmaf(x[e], c, -MC));
    }
}

// One cluster of TYP_CL CTAs per request: the rows' statistics and the draw's segment sums are shared
// among the CTAs (remote stores into CTA 0's shared memory), the tests, the walk, the scan and the
// outputs run in CTA 0; four cluster barriers order the hand-offs.
template <int DT, int VEC>
__global__ void __launch_bounds__(TYP_NT) typical_finish_kernel(TypicalParams P)
{
    extern __shared__ __align__(16) int32_t ysm[];
    __shared__ int sh_bad;
    __shared__ TreeWalk sh_walk;
    __shared__ int sh_tok;
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = TYP_NT / 32;
    const int b = blockIdx.x / CL, N = P.t.N, R = P.t.R;
    const unsigned FULL = 0xffffffffu;
    int32_t* par = ysm;
    int32_t* tok = ysm + N;
    int32_t* depth = ysm + 2 * N;
    int32_t* valid = ysm + 3 * N;
    int32_t* match = ysm + 4 * N;
    float* rMC = reinterpret_cast<float*>(ysm + 5 * N);
    float* rL2S = rMC + R;
    float* rH = rL2S + R;
    float* segs = rH + R;
    float* xlog = segs + P.nseg;

    // the tree, each node's token logit and the uniform do not depend on kernel 1 (CTA 0 uses them)
    const char* row0 = typ_row(P, b, 0);
    if (rank == 0)
        for (int i = tid; i < N; i += TYP_NT) {
            const int p = __ldg(P.t.parents + (size_t)b * N + i), x = __ldg(P.t.tokens + (size_t)b * N + i);
            par[i] = p;
            tok[i] = x;
            xlog[i] = (p >= -1 && p < i && x >= 0 && x < P.t.V)
                          ? load_logit(row0 + (size_t)(p < 0 ? 0 : p + 1) * P.t.V * esize(DT), DT, x)
                          : 0.f;
        }
    const float u = __ldg(P.uniforms + b);
    if (tid == 0) sh_bad = 0;
    // every CTA of the cluster has started and CTA 0's flag is cleared before any CTA reports to it
    // (taken while kernel 1 still runs)
    cluster.sync();
    pdl_wait();  // the partials of kernel 1
    // CTA 0's copies: every CTA writes its rows' statistics and its segment sums there
    float* rMC0 = cluster.map_shared_rank(rMC, 0);
    float* rL2S0 = cluster.map_shared_rank(rL2S, 0);
    float* rH0 = cluster.map_shared_rank(rH, 0);
    float* segs0 = cluster.map_shared_rank(segs, 0);

    // ---- each row's statistics: one warp per row, the partials merged as pairs of floats.  CTA k of
    // the cluster takes rows k, k + CL, ...; a warp's rows (up to TYP_RPW of them) have their first 64
    // partials in flight together.
    constexpr int TYP_RPW = 3;
    int bad = 0;
    auto row_of = [&](int i) { return rank + CL * i; };
    for (int i0 = warp; row_of(i0) < R; i0 += nw * TYP_RPW) {
        float4 q[TYP_RPW][2];
#pragma unroll
        for (int t = 0; t < TYP_RPW; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = row_of(i0 + t * nw), k = lane + 32 * h;
                q[t][h] = make_float4(NEG_INF, NEG_INF, 0.f, 0.f);
                if (j < R && k < P.np)
                    q[t][h] = __ldcg(reinterpret_cast<const float4*>(P.partials + ((size_t)b * R + j) * P.np + k));
            }
#pragma unroll
        for (int t = 0; t < TYP_RPW; ++t) {
            const int j = row_of(i0 + t * nw);
            if (j >= R) break;  // the same for every lane
            const TypPartial* pp = P.partials + ((size_t)b * R + j) * P.np;
            float Mr = fmaxf(q[t][0].x, q[t][1].x);
            for (int k = lane + 64; k < P.np; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
            Mr = warp_max(Mr);
            const float MCr = __fmul_rn(Mr, P.c);
            DFloat S = df_make(0.f, 0.f), E = df_make(0.f, 0.f);
            int tmo = 0;
            auto merge = [&](const float4& e) {
                if (e.z < 0.f) tmo = 1;
                if (e.z != 0.f) {  // NaN and inf propagate through S
                    const float d = e.y - MCr;
                    const float f = ex2(d);
                    S = df_add(S, df_make(__fmul_rn(e.z, f), 0.f));
                    E = df_add(E, df_make(__fmul_rn(f, fmaf(d, e.z, e.w)), 0.f));
                }
            };
            merge(q[t][0]);
            merge(q[t][1]);
            for (int k = lane + 64; k < P.np; k += 32) merge(__ldcg(reinterpret_cast<const float4*>(pp + k)));
            S = warp_sum_df(S);
            E = warp_sum_df(E);
            tmo = __any_sync(FULL, tmo);
            const bool ok = !tmo && isfinite(S.hi) && S.hi > 0.f && Mr != NEG_INF && isfinite(Mr);
            float l2s = __int_as_float(0x7fc00000), H = l2s;
            if (ok) {
                // log2 S = e + log2 m + log2(1 + lo / hi), S.hi = m 2^e with m in [0.5, 1)
                int ex;
                const float mant = frexpf(S.hi, &ex);
                l2s = __fadd_rn((float)ex, __fadd_rn(log2f(mant), __fmul_rn(__fdiv_rn(S.lo, S.hi), LOG2E_F)));
                // H = ln 2 (log2 S - E / S); E <= 0, so both terms add
                const float mean = __fdiv_rn(__fadd_rn(E.hi, E.lo), __fadd_rn(S.hi, S.lo));
                H = __fmul_rn(__fsub_rn(l2s, mean), LN2_HI);
            } else {
                bad = max(bad, tmo ? 2 : 1);
            }
            if (lane == 0) {
                rMC0[j] = MCr;
                rL2S0[j] = l2s;
                rH0[j] = H;
                if (P.aux_entropy) P.aux_entropy[(size_t)b * R + j] = H;
            }
        }
    }
    if (bad && lane == 0) atomicMax(cluster.map_shared_rank(&sh_bad, 0), bad);
    cluster.sync();  // CTA 0 holds every row's statistics

    // ---- every node's own test: ln p_r(x) > min(ln eps, ln delta - H_r) (CTA 0)
    for (int i = tid; rank == 0 && i < N; i += TYP_NT) {
        const int p = par[i], x = tok[i];
        int m = 0;
        float lnp = __int_as_float(0x7fc00000);
        if (!sh_bad && p >= -1 && p < i && x >= 0 && x < P.t.V) {
            const int r = p < 0 ? 0 : p + 1;
            const float xl = xlog[i];
            lnp = __fmul_rn(__fsub_rn(fmaf(xl, P.c, -rMC[r]), rL2S[r]), LN2_HI);
            const float lthr = fminf(P.ln_eps, __fsub_rn(P.ln_delta, rH[r]));
            m = lnp > lthr;
        }
        match[i] = m;
        if (P.aux_logp) P.aux_logp[(size_t)b * N + i] = lnp;
    }
    __syncthreads();

    // ---- the walk (warp 0 of CTA 0)
    if (rank == 0 && warp == 0) {
        const int late = (u >= 0.f && u < 1.f) ? 0 : ROW_BAD_UNIFORM;
        const TreeWalk w = tree_walk(N, P.t.V, P.t.max_out, sh_bad, late, par, tok,
                                     [&](int i, int) { return match[i] != 0; }, depth, valid);
        if (lane == 0) {
            sh_walk = w;
            sh_tok = -1;
        }
    }
    cluster.sync();  // the walk is visible to every CTA
    const TreeWalk w = *cluster.map_shared_rank(&sh_walk, 0);

    // ---- the token after the path: inverse CDF over the accepted node's row with u
    const int r = w.node < 0 ? 0 : w.node + 1;
    const char* rp = row0 + (size_t)r * P.t.V * esize(DT);
    const long long nvec = P.t.nvec;
    if (w.st == ROW_OK) {  // the same in every CTA of the cluster
        const float MC = rMC0[r];
        // per segment of 32 vectors its mass: CTA k of the cluster takes the k-th run of segments, a
        // warp its segments in batches of TYP_SB, their loads in flight together
        const int sper = (P.nseg + CL - 1) / CL;
        const int ga = min(rank * sper, P.nseg), gz = min(ga + sper, P.nseg);
        constexpr int TYP_SB = 8;
        const uint64_t pol = policy_evict_first();
        for (int g0 = ga + warp; g0 < gz; g0 += nw * TYP_SB) {
            RawVec<DT, VEC> x[TYP_SB];  // raw bits until used: 4 registers per 16-byte vector
#pragma unroll
            for (int k = 0; k < TYP_SB; ++k) {
                const long long v = (long long)(g0 + k * nw) * 32 + lane;
                x[k].fill_neg_inf();
                if (g0 + k * nw < gz && v < nvec) x[k].load(rp, v, pol);
            }
#pragma unroll
            for (int k = 0; k < TYP_SB; ++k) {
                if (g0 + k * nw >= gz) break;  // the same for every lane
                float m[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) m[e] = ex2(fmaf(x[k].get(e), P.c, -MC));
                const float ws = warp_sum(tree_sum(m));
                if (lane == 0) segs0[g0 + k * nw] = ws;
            }
        }
    }
    cluster.sync();  // CTA 0 holds every segment sum; the other CTAs are done
    if (rank != 0) return;
    if (w.st == ROW_OK) {
        const float MC = rMC[r];
        if (warp == 0) {
            // lane totals of contiguous blocks of segments, scanned in index order as pairs of
            // floats (the fp64 pipe is slow on this part; a pair carries about 48 bits)
            const int per = (P.nseg + 31) / 32;
            const int s0 = min(lane * per, P.nseg), s1 = min(s0 + per, P.nseg);
            DFloat mine = df_make(0.f, 0.f);
            for (int k = s0; k < s1; ++k) mine = df_add(mine, df_make(segs[k], 0.f));
            DFloat incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                DFloat n;
                n.hi = __shfl_up_sync(FULL, incl.hi, o);
                n.lo = __shfl_up_sync(FULL, incl.lo, o);
                if (lane >= o) incl = df_add(incl, n);
            }
            DFloat Z;
            Z.hi = __shfl_sync(FULL, incl.hi, 31);
            Z.lo = __shfl_sync(FULL, incl.lo, 31);
            const DFloat t = df_mul(Z, u, 0.f);
            const DFloat excl = df_add(incl, df_make(-mine.hi, -mine.lo));
            const bool pos_mass = mine.hi > 0.f;
            unsigned own = __ballot_sync(FULL, pos_mass && df_lt(t, incl));
            if (!own) {  // rounding ran past the end: the last lane holding mass
                const unsigned pos = __ballot_sync(FULL, pos_mass);
                own = pos ? (1u << (31 - __clz(pos))) : 0u;
            }
            int seg = -1;
            DFloat base = df_make(0.f, 0.f);
            if (own) {
                const int owner = __ffs(own) - 1;
                if (lane == owner) {
                    DFloat run = excl, lastbase = excl;
                    int lastpos = -1;
                    for (int k = s0; k < s1 && seg < 0; ++k) {
                        const float sv = segs[k];
                        const DFloat nxt = df_add(run, df_make(sv, 0.f));
                        if (sv > 0.f) { lastpos = k; lastbase = run; }
                        if (sv > 0.f && df_lt(t, nxt)) { seg = k; base = run; }
                        else run = nxt;
                    }
                    if (seg < 0) { seg = lastpos; base = lastbase; }
                }
                seg = __shfl_sync(FULL, seg, owner);
                base.hi = __shfl_sync(FULL, base.hi, owner);
                base.lo = __shfl_sync(FULL, base.lo, owner);
            }
            int y = -1;
            if (seg >= 0) {  // inside the segment: lane masses, then the owner's elements
                float m[VEC];
                const long long v = (long long)seg * 32 + lane;
                typ_mass<DT, VEC>(rp, v, nvec, P.c, MC, m);
                const float tl = __fadd_rn(__fsub_rn(t.hi, base.hi), __fsub_rn(t.lo, base.lo));
                const float ls = tree_sum(m);
                const float inc = warp_incl_scan(ls);
                const unsigned hit = __ballot_sync(FULL, tl < inc && ls > 0.f);
                int owner;
                if (hit) {
                    owner = __ffs(hit) - 1;
                } else {
                    const unsigned pos = __ballot_sync(FULL, ls > 0.f);
                    owner = pos ? 31 - __clz(pos) : 0;
                }
                if (lane == owner) {
                    float run = inc - ls;
                    int last = -1, pick = -1;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if (m[e] > 0.f) last = e;
                        run += m[e];
                        if (pick < 0 && hit && tl < run && m[e] > 0.f) pick = e;
                    }
                    if (pick < 0) pick = last;
                    y = pick < 0 ? -1 : (int)(v * VEC + pick);
                }
                y = __shfl_sync(FULL, y, owner);
            }
            if (lane == 0) sh_tok = y;
        }
    }
    __syncthreads();
    if (warp == 0) tree_emit(P.t, b, w, par, tok, sh_tok);
}

template <int DT, int VEC>
static cudaError_t launch_finish(const TypicalParams& P, cudaStream_t st)
{
    const size_t smem = typical_finish_smem(P.t.N, P.nseg);
    set_smem_limit<typical_finish_kernel<DT, VEC>>(smem);
    return launch_dependent_cluster(typical_finish_kernel<DT, VEC>, (unsigned)((long long)P.t.B * TYP_CL),
                                    TYP_NT, smem, TYP_CL, st, P);
}

template <int DT>
static cudaError_t launch_typical(const TypicalParams& P, int sms, cudaStream_t st)
{
    mark_kernel_start(st);
    if (P.t.vec > 1) {
        constexpr auto K1 = typical_stream_kernel<DT>;
        constexpr int smem = TYP_GROUPS * STREAM_SMEM, nth = stream_threads<TYP_GROUPS>();
        K1<<<cta_grid<K1>(((long long)P.t.B * P.t.R * P.S1 + TYP_GROUPS - 1) / TYP_GROUPS, sms, smem, nth), nth,
             smem, st>>>(P);
    } else {
        constexpr auto K1 = typical_stats_kernel<DT>;
        K1<<<persistent_grid<K1>((long long)P.t.B * P.t.R * P.S1, sms), NT, 0, st>>>(P);
    }
    mark_kernel_stop(st);
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    return P.t.vec > 1 ? launch_finish<DT, VEC>(P, st) : launch_finish<DT, 1>(P, st);
}

cudaError_t launch_typical_path(const TypicalParams& P, int sms, cudaStream_t st)
{
    const cudaError_t e = (P.t.dtype == DT_BF16) ? launch_typical<DT_BF16>(P, sms, st)
                                                 : launch_typical<DT_F32>(P, sms, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sv
