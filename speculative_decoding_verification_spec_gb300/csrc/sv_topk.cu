// sv_topk.cu -- exact speculative sampling with a top-k processor on p and q.
//
// M7.1 section 0x03D: truncation keeps the method exact when p and q are the truncated,
// renormalised distributions and q is the one that sampled the draft.  A row keeps every token
// whose stored logit is >= the row's k-th largest stored logit (counted with multiplicity), so ties
// at the threshold are all kept.
//
// Kernel 1 (topk_stats_kernel): one CTA per (row, chunk of NT*EPT elements), the chunk held in
// registers.  A lower bound tau of the chunk's k-th largest value is the k-th largest of the NT
// per-thread maxima (NT disjoint groups, so at least k chunk elements are >= tau); only elements
// >= tau -- a few dozen for k = 50 -- leave the registers.  The chunk's exact k-th largest value l_c
// is selected among them and every element >= l_c is listed.  Since the row's k-th largest value g
// satisfies g >= l_c for every chunk, the union of the chunk lists holds every element >= g, and the
// last CTA of the row selects g exactly from the union, keeps the entries >= g sorted by index, and
// forms (M, S) over them.  The last row of a request runs the acceptance scan and draws the
// correction / bonus token directly from the kept lists: the residual vanishes outside K_p, so no
// second pass over V is needed.
//
// Rows whose candidates overflow the on-chip capacities (massive ties, k > NT, ...) are marked
// dense and finished exactly by kernel 2 (topk_dense_kernel) with full-row passes.
#include <cuda_bf16.h>

#include "sv_plan.cuh"

namespace sv {

constexpr int CAP_S = 2048;  // candidate entries a chunk CTA holds on chip
constexpr int CAP_U = 2048;  // union entries the row epilogue holds on chip

// order-preserving 32-bit key of a float; -0 and +0 map to the same key
__device__ __forceinline__ uint32_t okey(float x)
{
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float fmax_nan_f(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Largest key P with count(key >= P) >= k over the n entries (the k-th largest key).  bf16-valued
// entries only differ in the top 16 key bits.  All threads of the CTA must call it.
template <int DT>
__device__ uint32_t block_kth_key(const TopkEntry* e, int n, int k, int* sh_red)
{
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        int cnt = 0;
        for (int i = threadIdx.x; i < n; i += NT) cnt += okey(e[i].x) >= want;
        cnt = block_sum_int(cnt, sh_red);
        if (cnt >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

// same over one value per thread
template <int DT>
__device__ uint32_t block_kth_key_per_thread(uint32_t key, int k)
{
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        if (__syncthreads_count(key >= want) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

// elements per thread held in registers, per dtype
template <int DT> struct TopkShape;
template <> struct TopkShape<DT_BF16> { static constexpr int EPT = 80, NREG = 40; };
template <> struct TopkShape<DT_F32> { static constexpr int EPT = 40, NREG = 40; };

// element index of register slot s of this thread (slot order = vector j, then lane e of it)
template <int VEC>
__device__ __forceinline__ long long slot_elem(long long cbase, int s)
{
    if constexpr (VEC == 1) return cbase + (long long)s * NT + threadIdx.x;
    else return cbase + ((long long)(s / VEC) * NT + threadIdx.x) * VEC + (s % VEC);
}

template <int DT, int VEC>
__device__ __forceinline__ float reg_value(const uint32_t (&w)[TopkShape<DT>::NREG], int s)
{
    if constexpr (DT == DT_BF16) return (s & 1) ? bf16hi(w[s >> 1]) : bf16lo(w[s >> 1]);
    else return __uint_as_float(w[s]);
}

// block exclusive scan of an int; returns exclusive prefix, total in *tot
__device__ __forceinline__ int block_excl_scan_int(int v, int* sh, int* tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int incl = warp_incl_scan(v);
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    int before = 0, t = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        if (w < warp) before += sh[w];
        t += sh[w];
    }
    *tot = t;
    return before + incl - v;
}

// bitonic sort of n entries by index (ascending), padded to a power of two with idx = INT_MAX
__device__ void block_sort_by_index(TopkEntry* e, int n)
{
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = n + threadIdx.x; i < m; i += NT) { e[i].idx = 0x7fffffff; e[i].x = NEG_INF; }
    __syncthreads();
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < m; i += NT) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    TopkEntry a = e[i], b = e[j];
                    if ((a.idx > b.idx) == up) { e[i] = b; e[j] = a; }
                }
            }
            __syncthreads();
        }
    }
}

struct TopkSmem {
    union {
        TopkEntry cand[CAP_S];  // chunk candidates, then the row's union
        double rr[CAP_S];       // request epilogue: residual mass of the kept list
    };
    TopkEntry kept[CAP_U];
    int red[WARPS];
    float redf[WARPS];
    int flag, n;
};

template <int DT, int VEC>
__global__ void __launch_bounds__(NT, 4) topk_stats_kernel(SpecParams P)
{
    using Shape = TopkShape<DT>;
    constexpr int EPT = Shape::EPT, NREG = Shape::NREG;
    static_assert(sizeof(TopkSmem) <= 48 * 1024, "static shared memory");
    __shared__ TopkSmem sm;

    const long long idx = blockIdx.x;
    const int chunk = (int)(idx % P.CT);
    const long long rs = idx / P.CT;
    const int b = (int)(rs / P.R), r = (int)(rs % P.R);
    const int row_id = b * P.R + r;
    const char* row = spec_row_ptr(P, b, r);
    const long long CE = (long long)NT * EPT;
    const long long cbase = (long long)chunk * CE;
    const long long cend = min(cbase + CE, (long long)P.V);
    const int k = P.top_k;

    // ---- load the chunk into registers (-inf padding)
    uint32_t w[NREG];
    if constexpr (VEC > 1) {
        constexpr int NV = EPT / VEC;  // vectors per thread
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const long long e0 = slot_elem<VEC>(cbase, j * VEC);
            uint4 q = make_uint4(0, 0, 0, 0);
            const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
            if (e0 < cend) q = ld_stream_v4(row + e0 * (DT == DT_BF16 ? 2 : 4));
            else q = make_uint4(pad, pad, pad, pad);
            w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
        }
    } else {
        if constexpr (DT == DT_BF16) {
            const unsigned short* rp = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
            for (int j = 0; j < NREG; ++j) {
                const long long e0 = slot_elem<1>(cbase, 2 * j), e1 = slot_elem<1>(cbase, 2 * j + 1);
                const uint32_t lo = e0 < cend ? __ldg(rp + e0) : 0xff80u;
                const uint32_t hi = e1 < cend ? __ldg(rp + e1) : 0xff80u;
                w[j] = lo | (hi << 16);
            }
        } else {
            const float* rp = reinterpret_cast<const float*>(row);
#pragma unroll
            for (int j = 0; j < NREG; ++j) {
                const long long e0 = slot_elem<1>(cbase, j);
                w[j] = e0 < cend ? __float_as_uint(__ldg(rp + e0)) : 0xff800000u;
            }
        }
    }

    // ---- group maxima (G registers each), thread maximum; NaN-propagating
    constexpr int G = 8, NG = NREG / G;
    static_assert(NREG % G == 0, "register groups");
    uint32_t gm[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        uint32_t m = w[g * G];
#pragma unroll
        for (int j = 1; j < G; ++j) {
            if constexpr (DT == DT_BF16) m = bmax2_nan(m, w[g * G + j]);
            else m = __float_as_uint(fmax_nan_f(__uint_as_float(m), __uint_as_float(w[g * G + j])));
        }
        gm[g] = m;
    }
    float tmax;
    if constexpr (DT == DT_BF16) {
        uint32_t pm = gm[0];
#pragma unroll
        for (int g = 1; g < NG; ++g) pm = bmax2_nan(pm, gm[g]);
        tmax = fmax_nan_f(bf16lo(pm), bf16hi(pm));
    } else {
        tmax = __uint_as_float(gm[0]);
#pragma unroll
        for (int g = 1; g < NG; ++g) tmax = fmax_nan_f(tmax, __uint_as_float(gm[g]));
    }
    if (threadIdx.x == 0) sm.n = 0;
    const int nonfinite = __syncthreads_or((tmax != tmax) || tmax == __int_as_float(0x7f800000));

    // ---- lower bound tau: k-th largest of the NT thread maxima (valid for k <= NT)
    uint32_t tau_key = okey(NEG_INF);
    if (!nonfinite && k <= NT) tau_key = block_kth_key_per_thread<DT>(okey(tmax), k);
    const float tau = key_value(tau_key);

    // ---- append every element >= tau to this chunk's list (unordered; the row merge sorts)
    TopkEntry* dst = P.clist + ((size_t)row_id * P.CT + chunk) * P.cap_w;
    const bool too_many = (k > NT) && (cend - cbase > P.cap_w);
    if (!nonfinite && !too_many) {
        auto append = [&](int slot, float x) {
            const long long e = slot_elem<VEC>(cbase, slot);
            if (e < cend) {
                const int pos = atomicAdd(&sm.n, 1);
                if (pos < P.cap_w) { TopkEntry en; en.x = x; en.idx = (int)e; dst[pos] = en; }
            }
        };
        if constexpr (DT == DT_BF16) {
            const __nv_bfloat162 t2 = __floats2bfloat162_rn(tau, tau);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                if (__hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&gm[g]), t2)) {
#pragma unroll
                    for (int j = g * G; j < g * G + G; ++j) {
                        const unsigned msk = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[j]), t2);
                        if (msk & 0xffffu) append(2 * j, bf16lo(w[j]));
                        if (msk >> 16) append(2 * j + 1, bf16hi(w[j]));
                    }
                }
            }
        } else {
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                if (__uint_as_float(gm[g]) >= tau) {
#pragma unroll
                    for (int j = g * G; j < g * G + G; ++j)
                        if (__uint_as_float(w[j]) >= tau) append(j, __uint_as_float(w[j]));
                }
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int n = sm.n;
        P.ccount[(size_t)row_id * P.CT + chunk] = nonfinite ? -2 : ((too_many || n > P.cap_w) ? -1 : n);
    }
    if (!arrive_last(&P.row_ctr[row_id], (unsigned)P.CT, &sm.flag)) return;

    // ==== last CTA of the row: exact threshold over the union of the chunk lists
    int bad = 0, over = 0, n_my = 0;
    for (int c = threadIdx.x; c < P.CT; c += NT) {
        const int n = __ldcg(P.ccount + (size_t)row_id * P.CT + c);
        if (n == -2) bad = 1;
        else if (n < 0) over = 1;
        else n_my += n;
    }
    bad = __syncthreads_or(bad);
    over = __syncthreads_or(over);
    const int utotal = block_sum_int(n_my, sm.red);
    RowStats st;
    st.M = NEG_INF; st.MC = NEG_INF; st.S = 0.0; st.thr = NEG_INF;
    st.status = ROW_OK; st.klist_n = -1; st.dense = 0;
    if (bad) {
        st.status = ROW_NONFINITE;
    } else if (over || utotal > CAP_U) {
        st.dense = 1;
    } else {
        // gather the union (chunk order)
        {
            int base = 0;
            for (int c = 0; c < P.CT; ++c) {
                const int n = __ldcg(P.ccount + (size_t)row_id * P.CT + c);
                const TopkEntry* src = P.clist + ((size_t)row_id * P.CT + c) * P.cap_w;
                for (int i = threadIdx.x; i < n; i += NT) {
                    TopkEntry en;
                    en.x = __ldcg(&src[i].x);
                    en.idx = __ldcg(&src[i].idx);
                    sm.cand[base + i] = en;
                }
                base += n;
            }
        }
        __syncthreads();
        const uint32_t gkey = (utotal >= k) ? block_kth_key<DT>(sm.cand, utotal, k, sm.red) : okey(NEG_INF);
        const float g = key_value(gkey);
        // keep entries >= g (stable order is not needed: they are sorted by index next)
        if (threadIdx.x == 0) sm.n = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < utotal; i += NT) {
            const TopkEntry en = sm.cand[i];
            if (okey(en.x) >= gkey) sm.kept[atomicAdd(&sm.n, 1)] = en;
        }
        __syncthreads();
        const int nk = sm.n;
        if (nk > P.cap_k) {
            st.dense = 1;
        } else {
            block_sort_by_index(sm.kept, nk);
            float mx = NEG_INF;
            for (int i = threadIdx.x; i < nk; i += NT) mx = fmaxf(mx, sm.kept[i].x);
            const float M = block_max(mx, sm.redf);
            const float MC = M * P.c;
            double S = 0.0;
            if (threadIdx.x < 32) {
                double acc = 0.0;
                if (M != NEG_INF)
                    for (int i = threadIdx.x; i < nk; i += 32) acc += (double)ex2(fmaf(sm.kept[i].x, P.c, -MC));
                S = warp_sum(acc);
            }
            TopkEntry* kl = P.klist + (size_t)row_id * P.cap_k;
            for (int i = threadIdx.x; i < nk; i += NT) kl[i] = sm.kept[i];
            st.M = M;
            st.MC = MC;
            st.S = S;
            st.thr = g;
            st.klist_n = nk;
            st.status = (M != NEG_INF && isfinite(M)) ? ROW_OK : ROW_NONFINITE;
        }
    }
    if (threadIdx.x == 0) P.rstats[row_id] = st;
    if (!arrive_last(&P.req_ctr[b], (unsigned)P.R, &sm.flag)) return;

    // ==== last row of the request
    int nd = 0;
    for (int rr = threadIdx.x; rr < P.R; rr += NT) nd += __ldcg(&P.rstats[(size_t)b * P.R + rr].dense);
    nd = block_sum_int(nd, sm.red);
    if (nd > 0) {  // finished by topk_dense_kernel
        if (threadIdx.x == 0) P.ndense[b] = nd;
        return;
    }
    __shared__ Plan sh_plan;
    if (threadIdx.x < 32) {
        const Plan p0 = compute_plan_warp<DT>(P, b, true);
        if (threadIdx.x == 0) sh_plan = p0;
    }
    __syncthreads();
    const Plan pl = sh_plan;
    if (pl.status != ROW_OK) {
        emit_spec(P, b, pl.status, 0, -1);
        return;
    }
    // residual over the kept list of the p row (index order); r vanishes outside K_p
    const RowStats sp = ld_rowstats(P.rstats + (size_t)b * P.R + pl.rp);
    const int nk = sp.klist_n;
    const TopkEntry* kl = P.klist + ((size_t)b * P.R + pl.rp) * P.cap_k;
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    for (int i = threadIdx.x; i < nk; i += NT) {
        const float xp = __ldcg(&kl[i].x);
        const int v = __ldcg(&kl[i].idx);
        float pp = __fmul_rn(ex2(fmaf(xp, P.c, -pl.MCp)), pl.invSp);
        float res = pp;
        if (rowq) {
            const float xq = load_logit(rowq, DT, v);
            const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, P.c, -pl.MCq)), pl.invSq) : 0.f;
            res = fmaxf(__fsub_rn(pp, qq), 0.f);
        }
        sm.rr[i] = (double)res;
        sm.kept[i].idx = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double Z = 0.0;
        for (int i = 0; i < nk; ++i) Z += sm.rr[i];
        int tok = -1;
        if (Z > 0.0 && isfinite(Z)) {
            const double t = pl.u * Z;
            double C = 0.0;
            int lastpos = -1;
            for (int i = 0; i < nk; ++i) {
                if (sm.rr[i] > 0.0) lastpos = i;
                C += sm.rr[i];
                if (t < C && sm.rr[i] > 0.0) { tok = sm.kept[i].idx; break; }
            }
            if (tok < 0 && lastpos >= 0) tok = sm.kept[lastpos].idx;
        }
        sm.n = tok;
    }
    __syncthreads();
    const int tok = sm.n;
    emit_spec(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}

// ---------------------------------------------------------------- exact fallback for dense rows

template <int DT>
__device__ __forceinline__ double topk_residual_at(const char* rowp, const char* rowq, long long v,
                                                   const Plan& pl, float c)
{
    const float xp = load_logit(rowp, DT, v);
    float pp = (xp >= pl.thrp) ? __fmul_rn(ex2(fmaf(xp, c, -pl.MCp)), pl.invSp) : 0.f;
    if (!rowq) return (double)pp;
    const float xq = load_logit(rowq, DT, v);
    const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, c, -pl.MCq)), pl.invSq) : 0.f;
    return (double)fmaxf(__fsub_rn(pp, qq), 0.f);
}

__device__ __forceinline__ double block_sum_f64(double v, double* sh)
{
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = 0.0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) r += sh[w];
    return r;
}

template <int DT>
__global__ void __launch_bounds__(NT) topk_dense_kernel(SpecParams P)
{
    __shared__ int sh_red[WARPS];
    __shared__ double sh_d[WARPS];
    __shared__ float sh_f[WARPS];
    __shared__ int sh_flag, sh_tok;

    const int row_id = blockIdx.x;
    const int b = row_id / P.R, r = row_id % P.R;
    if (!__ldcg(&P.rstats[row_id].dense)) return;
    const char* row = spec_row_ptr(P, b, r);
    const int V = P.V, k = P.top_k;

    // exact k-th largest key by bitwise search over full-row counts
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        int cnt = 0;
        for (int v = threadIdx.x; v < V; v += NT) cnt += okey(load_logit(row, DT, v)) >= want;
        if (block_sum_int(cnt, sh_red) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    const float g = key_value(prefix);
    float mx = NEG_INF;
    for (int v = threadIdx.x; v < V; v += NT) {
        const float x = load_logit(row, DT, v);
        if (x >= g) mx = fmaxf(mx, x);
    }
    const float M = block_max(mx, sh_f);
    const float MC = M * P.c;
    float s = 0.f;
    if (M != NEG_INF)
        for (int v = threadIdx.x; v < V; v += NT) {
            const float x = load_logit(row, DT, v);
            if (x >= g) s += ex2(fmaf(x, P.c, -MC));
        }
    const double S = block_sum_f32(s, sh_d);
    if (threadIdx.x == 0) {
        RowStats st;
        st.M = M; st.MC = MC; st.S = S; st.thr = g;
        st.status = (M != NEG_INF && isfinite(M) && S > 0.0) ? ROW_OK : ROW_NONFINITE;
        st.klist_n = -1;
        st.dense = 1;
        P.rstats[row_id] = st;
    }
    const unsigned nd = (unsigned)__ldcg(&P.ndense[b]);
    if (!arrive_last(&P.dense_ctr[b], nd, &sh_flag)) return;
    if (threadIdx.x == 0) P.ndense[b] = 0;

    __shared__ Plan sh_plan;
    if (threadIdx.x < 32) {
        const Plan p0 = compute_plan_warp<DT>(P, b, true);
        if (threadIdx.x == 0) sh_plan = p0;
    }
    __syncthreads();
    const Plan pl = sh_plan;
    if (pl.status != ROW_OK) {
        emit_spec(P, b, pl.status, 0, -1);
        return;
    }
    const char* rowp = spec_row_ptr(P, b, pl.rp);
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    // pass 1: total residual mass, tile by tile in index order (fp64)
    double Z = 0.0;
    for (int t0 = 0; t0 < V; t0 += NT) {
        const int v = t0 + threadIdx.x;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        Z += block_sum_f64(rv, sh_d);
    }
    if (!(Z > 0.0) || !isfinite(Z)) {
        emit_spec(P, b, ROW_DEGENERATE, 0, -1);
        return;
    }
    // pass 2: the tile where the running mass passes u*Z, then the element inside it
    const double t = pl.u * Z;
    double run = 0.0;
    int tok = -1;
    for (int t0 = 0; t0 < V; t0 += NT) {
        const int v = t0 + threadIdx.x;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        const double ts = block_sum_f64(rv, sh_d);
        if (t < run + ts) {  // uniform across the CTA
            double tot;
            const double excl = block_excl_scan_f64(rv, sh_d, &tot);
            if (threadIdx.x == 0) sh_tok = 0x7fffffff;
            __syncthreads();
            if (rv > 0.0 && t < run + excl + rv) atomicMin(&sh_tok, v);
            __syncthreads();
            tok = sh_tok;
            if (tok == 0x7fffffff) {  // rounding: last positive entry of the tile
                __syncthreads();
                if (threadIdx.x == 0) sh_tok = -1;
                __syncthreads();
                if (rv > 0.0) atomicMax(&sh_tok, v);
                __syncthreads();
                tok = sh_tok;
            }
            break;
        }
        run += ts;
    }
    if (tok < 0) {  // rounding ran past the end: last token with positive mass
        __syncthreads();
        if (threadIdx.x == 0) sh_tok = -1;
        __syncthreads();
        for (int v = threadIdx.x; v < V; v += NT)
            if (topk_residual_at<DT>(rowp, rowq, v, pl, P.c) > 0.0) atomicMax(&sh_tok, v);
        __syncthreads();
        tok = sh_tok;
    }
    emit_spec(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}

cudaError_t launch_topk_path(const SpecParams& P, unsigned g1, unsigned g2, cudaStream_t st)
{
    if (P.dtype == DT_BF16) {
        if (P.vec == 8) topk_stats_kernel<DT_BF16, 8><<<g1, NT, 0, st>>>(P);
        else topk_stats_kernel<DT_BF16, 1><<<g1, NT, 0, st>>>(P);
        topk_dense_kernel<DT_BF16><<<g2, NT, 0, st>>>(P);
    } else {
        if (P.vec == 4) topk_stats_kernel<DT_F32, 4><<<g1, NT, 0, st>>>(P);
        else topk_stats_kernel<DT_F32, 1><<<g1, NT, 0, st>>>(P);
        topk_dense_kernel<DT_F32><<<g2, NT, 0, st>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace sv
