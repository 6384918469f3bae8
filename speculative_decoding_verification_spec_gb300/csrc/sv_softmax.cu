// sv_softmax.cu -- exact speculative sampling without top-k: the one-pass row normalisers and
// the residual / bonus inverse-CDF draw.
//
// Kernel 1 (spec_stats_kernel): one CTA per (row, chunk of V).  Each thread streams 16-byte
// vectors, keeps an online (max, sum of 2^(x*c - max*c)) pair -- the online (m, l) merge over
// vocabulary blocks of M7.1 section 0x04J -- and the CTA writes one partial.  The last CTA of a row
// merges the row's partials (fp64), and the last row of a request runs the acceptance scan
// (sv_plan.cuh).  Completion is counted with atomics ("last CTA done"); nothing ever waits.
//
// Kernel 2 (spec_resample_kernel): one CTA per (request, chunk of V).  Each warp turns 32 vectors of
// the selected row pair into residual mass r = max(p - q, 0) (M7.1 section 0x03C; p alone for the
// bonus, 0x03H) and stores one segment sum.  The last CTA of the request scans the segment sums in
// fp64 in index order, finds the segment where the running mass passes u * Z, and one warp
// resolves the token inside that segment.
#include "sv_plan.cuh"

namespace sv {

// Row visiting order: all requests' bonus rows first, then draft pairs gamma-1 .. 0 (target row
// then draft row).  Pair 0 -- the most likely correction pair -- is read last, so it is the most
// likely to still sit in L2 when the resample kernel needs it.
__device__ __forceinline__ int slot_to_row(int slot, int gamma)
{
    if (slot == 0) return gamma;
    const int j = (slot - 1) >> 1;
    const int pos = gamma - 1 - j;
    return ((slot - 1) & 1) ? gamma + 1 + pos : pos;
}

// Online softmax statistics of vectors [v0, v1) of one row: per thread (m, mc, s) with
// mc = fp32(m*c) and s = sum 2^(fma(x, c, -mc)).
template <int DT, int VEC>
__device__ __forceinline__ void chunk_softmax_stats(const char* row, long long v0, long long v1,
                                                    float c, float& m, float& mc, float& s)
{
    constexpr int U = (VEC == 1) ? 8 : 4;  // vectors per thread per step
    for (long long base = v0 + threadIdx.x; base < v1; base += (long long)NT * U) {
        if constexpr (DT == DT_BF16 && VEC == 8) {
            uint4 w[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const long long v = base + (long long)j * NT;
                if (v < v1) w[j] = ld_stream_v4(row + v * 16);
                else w[j] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            }
            uint32_t pm = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
            for (int j = 1; j < U; ++j)
                pm = bmax2(pm, bmax2(bmax2(w[j].x, w[j].y), bmax2(w[j].z, w[j].w)));
            const float bm = fmaxf(bf16lo(pm), bf16hi(pm));
            if (bm > m) {
                const float mcn = bm * c;
                s *= ex2(mc - mcn);
                m = bm;
                mc = mcn;
            }
            if (mc != NEG_INF) {
                float acc[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const uint32_t q[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
                    float e[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        e[2 * k] = ex2(fmaf(bf16lo(q[k]), c, -mc));
                        e[2 * k + 1] = ex2(fmaf(bf16hi(q[k]), c, -mc));
                    }
                    acc[j] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
                }
                float t = acc[0];
#pragma unroll
                for (int j = 1; j < U; ++j) t += acc[j];
                s += t;
            }
        } else {
            float x[U][VEC];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const long long v = base + (long long)j * NT;
                if (v < v1) {
                    load_vec<DT, VEC>(row, v, x[j]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) x[j][e] = NEG_INF;
                }
            }
            float bm = NEG_INF;
#pragma unroll
            for (int j = 0; j < U; ++j)
#pragma unroll
                for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, x[j][e]);
            if (bm > m) {
                const float mcn = bm * c;
                s *= ex2(mc - mcn);
                m = bm;
                mc = mcn;
            }
            if (mc != NEG_INF) {
                float acc[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    float e[VEC];
#pragma unroll
                    for (int k = 0; k < VEC; ++k) e[k] = ex2(fmaf(x[j][k], c, -mc));
                    acc[j] = tree_sum(e);
                }
                s += tree_sum(acc);
            }
        }
    }
}

__device__ __forceinline__ Partial ld_partial(const Partial* p)
{
    Partial r;
    r.M = __ldcg(&p->M);
    r.MC = __ldcg(&p->MC);
    r.S = __ldcg(&p->S);
    return r;
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT) spec_stats_kernel(SpecParams P)
{
    __shared__ float sh_f[WARPS];
    __shared__ double sh_d[WARPS];
    __shared__ int sh_flag;

    const long long idx = blockIdx.x;
    const int chunk = (int)(idx % P.C1);
    const long long rs = idx / P.C1;
    const int slot = (int)(rs / P.B), b = (int)(rs % P.B);
    const int r = slot_to_row(slot, P.gamma);
    const char* row = spec_row_ptr(P, b, r);
    const long long v0 = (long long)chunk * P.cv1;
    const long long v1 = min(v0 + P.cv1, P.nvec);

    float m = NEG_INF, mc = NEG_INF, s = 0.f;
    chunk_softmax_stats<DT, VEC>(row, v0, v1, P.c, m, mc, s);

    const float M = block_max(m, sh_f);
    const float MC = M * P.c;
    const float sc = (mc == NEG_INF) ? 0.f : s * ex2(mc - MC);
    const double S = block_sum_f32(sc, sh_d);
    const int row_id = b * P.R + r;
    if (threadIdx.x == 0) {
        Partial pt;
        pt.M = M;
        pt.MC = MC;
        pt.S = S;
        P.partials[(size_t)row_id * P.C1 + chunk] = pt;
    }
    if (!arrive_last(&P.row_ctr[row_id], (unsigned)P.C1, &sh_flag)) return;

    // last CTA of this row: merge the chunk partials in chunk order
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const Partial* pp = P.partials + (size_t)row_id * P.C1;
        float Mr = NEG_INF;
        for (int k = lane; k < P.C1; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
        Mr = warp_max(Mr);
        const float MCr = Mr * P.c;
        double Sr = 0.0;
        for (int k = lane; k < P.C1; k += 32) {
            Partial q = ld_partial(pp + k);
            if (q.S != 0.0) Sr += q.S * exp2((double)q.MC - (double)MCr);
        }
        Sr = warp_sum(Sr);
        if (lane == 0) {
            RowStats st;
            st.M = Mr;
            st.MC = MCr;
            st.S = Sr;
            st.thr = NEG_INF;
            st.klist_n = -1;
            st.dense = 0;
            const bool ok = isfinite(Sr) && Sr > 0.0 && Mr != NEG_INF && isfinite(Mr);
            st.status = ok ? ROW_OK : ROW_NONFINITE;
            P.rstats[row_id] = st;
        }
    }
    if (!arrive_last(&P.req_ctr[b], (unsigned)P.R, &sh_flag)) return;

    // last row of this request: acceptance scan
    Plan pl = compute_plan<DT>(P, b, false);
    if (threadIdx.x == 0) P.plan[b] = pl;
}

// ---------------------------------------------------------------- resample

// Resolve the token inside segment s (vectors base .. base+31 of the chunk, one per lane) given
// the mass t_local still to pass within the segment.  Runs in one warp.  Returns the token.
template <int DT, int VEC>
__device__ int resolve_in_segment(const SpecParams& P, const char* rowp, const char* rowq,
                                  const Plan& pl, long long vbase, long long vend, double t_local)
{
    const int lane = threadIdx.x & 31;
    const long long v = vbase + lane;
    float r[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = 0.f;
    if (v < vend) residual_vec<DT, VEC>(rowp, rowq, v, pl, P.c, false, r);
    const float ls = tree_sum(r);
    const double incl = warp_incl_scan((double)ls);
    const double excl = __shfl_up_sync(0xffffffffu, incl, 1);
    const double start = lane ? excl : 0.0;
    const unsigned hit = __ballot_sync(0xffffffffu, t_local < incl);
    int owner;
    if (hit) {
        owner = __ffs(hit) - 1;
    } else {  // rounding left t_local past the segment: take its last positive entry
        const unsigned pos = __ballot_sync(0xffffffffu, ls > 0.f);
        owner = pos ? 31 - __clz(pos) : 0;
    }
    int tok = -1;
    if (lane == owner) {
        double run = start;
        int last_pos = -1;
        for (int e = 0; e < VEC; ++e) {
            if (r[e] > 0.f) last_pos = e;
            run += (double)r[e];
            if (hit && t_local < run && r[e] > 0.f) { tok = e; break; }
        }
        if (tok < 0) tok = last_pos;
        tok = (tok < 0) ? -1 : (int)(v * VEC + tok);
    }
    return __shfl_sync(0xffffffffu, tok, owner);
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT) spec_resample_kernel(SpecParams P)
{
    __shared__ double sh_d[WARPS];
    __shared__ int sh_flag, sh_owner, sh_seg;
    __shared__ double sh_base;

    const int b = blockIdx.x / P.C2, c = blockIdx.x % P.C2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Plan pl = ld_plan(P.plan + b);
    const int nseg_chunk = P.iters2 * WARPS;
    const char* rowp = spec_row_ptr(P, b, pl.rp);
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;

    if (pl.status == ROW_OK) {
        const long long cb = (long long)c * P.cv2;
        const long long ce = min(cb + P.cv2, P.nvec);
        float* segs = P.segs + ((size_t)b * P.C2 + c) * nseg_chunk;
        for (int it = 0; it < P.iters2; ++it) {
            const long long v = cb + (long long)it * NT + tid;
            float ls = 0.f;
            if (v < ce) {
                float r[VEC];
                residual_vec<DT, VEC>(rowp, rowq, v, pl, P.c, false, r);
                ls = tree_sum(r);
            }
            const float ws = warp_sum(ls);
            if (lane == 0) segs[it * WARPS + warp] = ws;
        }
    }
    if (!arrive_last(&P.res_ctr[b], (unsigned)P.C2, &sh_flag)) return;
    if (pl.status != ROW_OK) {
        emit_spec(P, b, pl.status, 0, -1);
        return;
    }

    // fp64 scan of the request's segment sums in index order
    const int nseg = P.C2 * nseg_chunk;
    const float* segs = P.segs + (size_t)b * nseg;
    const int per = (nseg + NT - 1) / NT;
    const int s0 = min(tid * per, nseg), s1 = min(s0 + per, nseg);
    double mine = 0.0;
    for (int s = s0; s < s1; ++s) mine += (double)__ldcg(segs + s);
    double Z;
    const double excl = block_excl_scan_f64(mine, sh_d, &Z);
    if (!(Z > 0.0) || !isfinite(Z)) {
        emit_spec(P, b, ROW_DEGENERATE, 0, -1);
        return;
    }
    const double t = pl.u * Z;
    if (tid == 0) sh_owner = NT;
    __syncthreads();
    if (s1 > s0 && mine > 0.0 && t < excl + mine) atomicMin(&sh_owner, tid);
    __syncthreads();
    int owner = sh_owner;
    if (owner == NT) {  // rounding: fall back to the last thread holding positive mass
        if (tid == 0) sh_owner = -1;
        __syncthreads();
        if (mine > 0.0) atomicMax(&sh_owner, tid);
        __syncthreads();
        owner = sh_owner;
    }
    if (tid == owner) {
        double run = 0.0;
        int seg = -1, lastpos = -1;
        double base = excl, lastbase = excl;
        for (int s = s0; s < s1; ++s) {
            const double sv = (double)__ldcg(segs + s);
            const double nx = run + sv;
            if (sv > 0.0) { lastpos = s; lastbase = excl + run; }
            if (t < excl + nx && sv > 0.0) { seg = s; base = excl + run; break; }
            run = nx;
        }
        if (seg < 0) { seg = lastpos; base = lastbase; }
        sh_seg = seg;
        sh_base = base;
    }
    __syncthreads();
    if (sh_seg < 0) {  // no segment holds positive mass (cannot happen when Z > 0)
        emit_spec(P, b, ROW_DEGENERATE, 0, -1);
        return;
    }
    if (warp == 0) {
        const int seg = sh_seg;
        const int cc = seg / nseg_chunk, rem = seg % nseg_chunk;
        const int it = rem / WARPS, w = rem % WARPS;
        const long long cb = (long long)cc * P.cv2;
        const long long ce = min(cb + P.cv2, P.nvec);
        const long long vbase = cb + (long long)it * NT + (long long)w * 32;
        const int tok = resolve_in_segment<DT, VEC>(P, rowp, rowq, pl, vbase, ce, t - sh_base);
        if (lane == 0) sh_seg = tok;
    }
    __syncthreads();
    const int tok = sh_seg;
    emit_spec(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}

cudaError_t launch_softmax_path(const SpecParams& P, unsigned g1, unsigned g2, cudaStream_t st)
{
    if (P.dtype == DT_BF16 && P.vec == 8) {
        spec_stats_kernel<DT_BF16, 8><<<g1, NT, 0, st>>>(P);
        spec_resample_kernel<DT_BF16, 8><<<g2, NT, 0, st>>>(P);
    } else if (P.dtype == DT_BF16) {
        spec_stats_kernel<DT_BF16, 1><<<g1, NT, 0, st>>>(P);
        spec_resample_kernel<DT_BF16, 1><<<g2, NT, 0, st>>>(P);
    } else if (P.vec == 4) {
        spec_stats_kernel<DT_F32, 4><<<g1, NT, 0, st>>>(P);
        spec_resample_kernel<DT_F32, 4><<<g2, NT, 0, st>>>(P);
    } else {
        spec_stats_kernel<DT_F32, 1><<<g1, NT, 0, st>>>(P);
        spec_resample_kernel<DT_F32, 1><<<g2, NT, 0, st>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace sv
