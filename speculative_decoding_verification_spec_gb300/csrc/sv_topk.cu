// sv_topk.cu -- exact speculative sampling with a top-k processor on p and q.
//
// M7.1 section 0x03D: truncation keeps the method exact when p and q are the truncated,
// renormalised distributions and q is the one that sampled the draft.  A row keeps every token
// whose stored logit is >= the row's k-th largest stored logit (counted with multiplicity), so ties
// at the threshold are all kept.
//
// Kernel 1 (topk_stats_kernel): one CTA per (row, contiguous chunk of NT*EPT elements), the chunk
// held in registers.  A lower bound tau of the chunk's k-th largest value is the k-th largest of the
// NT per-thread maxima (NT disjoint groups, so at least k chunk elements are >= tau), selected by
// one warp; only elements >= tau -- a few dozen for k = 50 -- leave the registers: collected in
// shared memory, then appended to the row's union buffer with one reservation per chunk.  Since the
// row's k-th largest value g is >= every chunk's tau, the union holds every element >= g.  One warp of the last CTA of the row selects g exactly from
// the union, keeps the entries >= g sorted by index and forms (M, S) over them; one warp of the last
// row of a request runs the acceptance scan and draws the correction / bonus token directly from
// the kept list: the residual vanishes outside K_p, so no second pass over V is needed.
//
// Rows whose candidates overflow the capacities (massive ties, k > NT, ...) are marked dense and
// finished exactly by kernel 2 (topk_dense_kernel) with full-row passes.
#include <cuda_bf16.h>

#include "sv_plan.cuh"

namespace sv {

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

// The k-th largest key (largest P with count(key >= P) >= k) among n keys produced by key_at(i),
// by one warp: bitwise search from the top bit, counting with a warp reduction per bit.
// bf16-valued keys differ only in their top 16 bits.
template <int DT, class KeyAt>
__device__ uint32_t warp_kth_key(int n, int k, KeyAt key_at)
{
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        unsigned cnt = 0;
        for (int i = lane; i < n; i += 32) cnt += key_at(i) >= want;
        if ((int)__reduce_add_sync(0xffffffffu, cnt) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

// elements per thread held in registers, per dtype
template <int DT> struct TopkShape;
template <> struct TopkShape<DT_BF16> { static constexpr int EPT = 80, NREG = 40; };
template <> struct TopkShape<DT_F32> { static constexpr int EPT = 40, NREG = 40; };

// element index (within the row) of register slot s of this thread: vector j = s / VEC, element
// e = s % VEC of it; vectors of a thread are NT apart
template <int VEC>
__device__ __forceinline__ int slot_elem(int cbase, int s)
{
    if constexpr (VEC == 1) return cbase + s * NT + (int)threadIdx.x;
    else return cbase + ((s / VEC) * NT + (int)threadIdx.x) * VEC + (s % VEC);
}

// w[base + j] for a run-time j in [0, 8) and a compile-time base, by a select tree (no local memory)
template <int N>
__device__ __forceinline__ uint32_t select8(const uint32_t (&w)[N], int base, int j)
{
    const uint32_t a0 = (j & 1) ? w[base + 1] : w[base];
    const uint32_t a1 = (j & 1) ? w[base + 3] : w[base + 2];
    const uint32_t a2 = (j & 1) ? w[base + 5] : w[base + 4];
    const uint32_t a3 = (j & 1) ? w[base + 7] : w[base + 6];
    const uint32_t c0 = (j & 2) ? a1 : a0;
    const uint32_t c1 = (j & 2) ? a3 : a2;
    return (j & 4) ? c1 : c0;
}

constexpr int CAP_C = 1024;  // candidates a chunk CTA collects on chip

struct TopkSmem {
    union {
        TopkEntry cand[CAP_C];  // chunk phase: this chunk's candidates
        TopkEntry u[CAP_U];     // row epilogue: union of the chunks' candidates
        double rr[CAP_U];       // request epilogue: residual mass of the kept list
    };
    TopkEntry kept[CAP_U];
    float tmax[NT];
    float tau;
    int n, base, flag, nonfinite;
};

// append one candidate to the chunk's on-chip list (the slot beyond CAP_C only counts)
__device__ __forceinline__ void cand_push(TopkSmem& sm, float x, int e)
{
    const int pos = atomicAdd(&sm.n, 1);
    if (pos < CAP_C) {
        sm.cand[pos].x = x;
        sm.cand[pos].idx = e;
    }
}

// Warp-level bitonic sort of e[0..n) by index (ascending), padding to a power of two.
__device__ void warp_sort_by_index(TopkEntry* e, int n)
{
    const int lane = threadIdx.x & 31;
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = n + lane; i < m; i += 32) { e[i].idx = 0x7fffffff; e[i].x = NEG_INF; }
    __syncwarp();
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = lane; i < m; i += 32) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const TopkEntry a = e[i], b = e[j];
                    if ((a.idx > b.idx) == up) { e[i] = b; e[j] = a; }
                }
            }
            __syncwarp();
        }
    }
}

// One warp of the last CTA of a row: exact threshold over the union of the chunk lists, kept list
// sorted by index, normaliser over it.  Returns the row's stats.
template <int DT>
__device__ RowStats topk_row_epilogue(const SpecParams& P, TopkSmem& sm, int row_id)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    RowStats st;
    st.M = NEG_INF; st.MC = NEG_INF; st.S = 0.0; st.thr = NEG_INF;
    st.status = ROW_OK; st.klist_n = -1; st.dense = 0;
    const int flags = __ldcg(P.uflags + row_id);
    const int total = __ldcg(P.ucount + row_id);
    if (flags & 1) { st.status = ROW_NONFINITE; return st; }
    if ((flags & 2) || total > P.cap_u) { st.dense = 1; return st; }
    // the union, contiguous: independent loads, several in flight per lane
    const TopkEntry* src = P.ulist + (size_t)row_id * P.cap_u;
#pragma unroll 8
    for (int i = lane; i < total; i += 32) {
        TopkEntry en;
        en.x = __ldcg(&src[i].x);
        en.idx = __ldcg(&src[i].idx);
        sm.u[i] = en;
    }
    __syncwarp();
    const int k = P.top_k;
    const uint32_t gkey = (total >= k) ? warp_kth_key<DT>(total, k, [&](int i) { return okey(sm.u[i].x); })
                                       : okey(NEG_INF);
    // stable ballot compaction of the entries >= g
    int nk = 0;
    for (int i0 = 0; i0 < total; i0 += 32) {
        const int i = i0 + lane;
        const bool keep = i < total && okey(sm.u[i].x) >= gkey;
        const unsigned bal = __ballot_sync(FULL, keep);
        if (keep) sm.kept[nk + __popc(bal & ((1u << lane) - 1u))] = sm.u[i];
        nk += __popc(bal);
    }
    __syncwarp();
    if (nk > P.cap_k) { st.dense = 1; return st; }
    warp_sort_by_index(sm.kept, nk);
    float mx = NEG_INF;
    for (int i = lane; i < nk; i += 32) mx = fmaxf(mx, sm.kept[i].x);
    const float M = warp_max(mx);
    const float MC = M * P.c;
    double acc = 0.0;
    if (M != NEG_INF)
        for (int i = lane; i < nk; i += 32) acc += (double)ex2(fmaf(sm.kept[i].x, P.c, -MC));
    const double S = warp_sum(acc);
    TopkEntry* kl = P.klist + (size_t)row_id * P.cap_k;
    for (int i = lane; i < nk; i += 32) kl[i] = sm.kept[i];
    st.M = M;
    st.MC = MC;
    st.S = S;
    st.thr = key_value(gkey);
    st.klist_n = nk;
    st.status = (M != NEG_INF && isfinite(M)) ? ROW_OK : ROW_NONFINITE;
    return st;
}

// One warp: acceptance scan of request b and the correction / bonus draw from the kept list of
// the p row (index order); the residual is zero outside K_p.
template <int DT>
__device__ void topk_request_epilogue(const SpecParams& P, TopkSmem& sm, int b)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const Plan pl = compute_plan_warp<DT>(P, b, true);
    if (pl.status != ROW_OK) {
        emit_spec_warp(P, b, pl.status, 0, -1);
        return;
    }
    const RowStats sp = ld_rowstats(P.rstats + (size_t)b * P.R + pl.rp);
    const int nk = sp.klist_n;
    const TopkEntry* kl = P.klist + ((size_t)b * P.R + pl.rp) * P.cap_k;
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    // each lane owns a contiguous block of the kept list
    const int per = (nk + 31) / 32;
    const int i0 = min(lane * per, nk), i1 = min(i0 + per, nk);
    double mine = 0.0;
    for (int i = i0; i < i1; ++i) {
        const float xp = __ldcg(&kl[i].x);
        const int v = __ldcg(&kl[i].idx);
        const float pp = __fmul_rn(ex2(fmaf(xp, P.c, -pl.MCp)), pl.invSp);
        float res = pp;
        if (rowq) {
            const float xq = load_logit(rowq, DT, v);
            const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, P.c, -pl.MCq)), pl.invSq) : 0.f;
            res = fmaxf(__fsub_rn(pp, qq), 0.f);
        }
        sm.rr[i] = (double)res;
        mine += (double)res;
    }
    const double incl = warp_incl_scan(mine);
    const double Z = __shfl_sync(FULL, incl, 31);
    int tok = -1;
    if (Z > 0.0 && isfinite(Z)) {
        const double t = pl.u * Z, excl = incl - mine;
        unsigned own = __ballot_sync(FULL, mine > 0.0 && t < excl + mine);
        if (!own) {
            const unsigned pos = __ballot_sync(FULL, mine > 0.0);
            own = pos ? (1u << (31 - __clz(pos))) : 0u;
        }
        if (own) {
            const int owner = __ffs(own) - 1;
            if (lane == owner) {
                double run = excl;
                int lastpos = -1;
                for (int i = i0; i < i1; ++i) {
                    if (sm.rr[i] > 0.0) lastpos = i;
                    run += sm.rr[i];
                    if (t < run && sm.rr[i] > 0.0) { tok = __ldcg(&kl[i].idx); break; }
                }
                if (tok < 0 && lastpos >= 0) tok = __ldcg(&kl[lastpos].idx);
            }
            tok = __shfl_sync(FULL, tok, owner);
        }
    }
    emit_spec_warp(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT, 4) topk_stats_kernel(SpecParams P)
{
    using Shape = TopkShape<DT>;
    constexpr int EPT = Shape::EPT, NREG = Shape::NREG;
    static_assert(sizeof(TopkSmem) <= 48 * 1024, "static shared memory");
    __shared__ TopkSmem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x % P.CT;
    const int rs = blockIdx.x / P.CT;
    const int b = rs / P.R, r = rs % P.R;
    const int row_id = b * P.R + r;
    const char* row = spec_row_ptr(P, b, r);
    const int cbase = chunk * NT * EPT;
    const int cend = min(cbase + NT * EPT, P.V);
    const int k = P.top_k;
    const uint64_t pol = policy_evict_first();

    // ---- load the chunk into registers (-inf padding)
    uint32_t w[NREG];
    if constexpr (VEC > 1) {
        constexpr int NV = EPT / VEC;  // vectors per thread
        constexpr int ES = (DT == DT_BF16) ? 2 : 4;
        const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
        const char* tp = row + ((size_t)cbase + (size_t)tid * VEC) * ES;  // this thread's first vector
        if (cbase + NT * EPT <= cend) {  // full chunk: fixed offsets, no bounds checks
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint4 q = ld_stream_v4_pol(tp + (size_t)j * NT * VEC * ES, pol);
                w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const int e0 = cbase + (j * NT + tid) * VEC;
                const uint4 q = e0 < cend ? ld_stream_v4_pol(tp + (size_t)j * NT * VEC * ES, pol)
                                          : make_uint4(pad, pad, pad, pad);
                w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
            }
        }
    } else if constexpr (DT == DT_BF16) {
        const unsigned short* rp = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
        for (int j = 0; j < NREG; ++j) {
            const int e0 = slot_elem<1>(cbase, 2 * j), e1 = slot_elem<1>(cbase, 2 * j + 1);
            const uint32_t lo = e0 < cend ? __ldg(rp + e0) : 0xff80u;
            const uint32_t hi = e1 < cend ? __ldg(rp + e1) : 0xff80u;
            w[j] = lo | (hi << 16);
        }
    } else {
        const float* rp = reinterpret_cast<const float*>(row);
#pragma unroll
        for (int j = 0; j < NREG; ++j) {
            const int e0 = slot_elem<1>(cbase, j);
            w[j] = e0 < cend ? __float_as_uint(__ldg(rp + e0)) : 0xff800000u;
        }
    }

    // ---- group maxima (G registers each) and the thread maximum, NaN-propagating
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
    sm.tmax[tid] = tmax;
    __syncthreads();

    // ---- one warp: non-finite check and tau = k-th largest thread maximum (valid for k <= NT)
    if (warp == 0) {
        int bad = 0;
        for (int i = lane; i < NT; i += 32) {
            const float x = sm.tmax[i];
            if (x != x || x == __int_as_float(0x7f800000)) bad = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        uint32_t tk = okey(NEG_INF);
        if (!bad && k <= NT) {
            uint32_t keys[NT / 32];
#pragma unroll
            for (int i = 0; i < NT / 32; ++i) keys[i] = okey(sm.tmax[lane + 32 * i]);
            uint32_t prefix = 0;
            constexpr int lo = (DT == DT_BF16) ? 16 : 0;
            for (int bit = 31; bit >= lo; --bit) {
                const uint32_t want = prefix | (1u << bit);
                unsigned cnt = 0;
#pragma unroll
                for (int i = 0; i < NT / 32; ++i) cnt += keys[i] >= want;
                if ((int)__reduce_add_sync(0xffffffffu, cnt) >= k) prefix = want;
            }
            if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
            tk = prefix;
        }
        if (lane == 0) {
            sm.tau = key_value(tk);
            sm.nonfinite = bad;
            sm.n = 0;
        }
    }
    __syncthreads();
    const float tau = sm.tau;
    const int nonfinite = sm.nonfinite;

    // ---- collect every element >= tau on chip (unordered; the row merge sorts).  A group whose
    // maximum passes tau yields a bitmask of its passing slots; only the set bits are visited.
    const bool too_many = (k > NT) && (cend - cbase > CAP_C);
    if (!nonfinite && !too_many) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            uint32_t bits = 0;
            if constexpr (DT == DT_BF16) {
                const __nv_bfloat162 t2 = __floats2bfloat162_rn(tau, tau);
                if (__hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&gm[g]), t2)) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const uint32_t wd = w[g * G + j];
                        bits |= (__hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&wd), t2) & 0x00010001u) << j;
                    }
                }
            } else {
                if (__uint_as_float(gm[g]) >= tau) {
#pragma unroll
                    for (int j = 0; j < G; ++j) bits |= (uint32_t)(__uint_as_float(w[g * G + j]) >= tau) << j;
                }
            }
            while (bits) {
                const int bp = __ffs(bits) - 1;
                bits &= bits - 1;
                const int j = bp & 15, half = bp >> 4;  // register j of the group, bf16 half
                const uint32_t wd = select8(w, g * G, j);
                float x;
                int s;
                if constexpr (DT == DT_BF16) {
                    x = half ? bf16hi(wd) : bf16lo(wd);
                    s = 2 * (g * G + j) + half;
                } else {
                    x = __uint_as_float(wd);
                    s = g * G + j;
                }
                const int e = slot_elem<VEC>(cbase, s);
                if (e < cend) cand_push(sm, x, e);
            }
        }
    }
    __syncthreads();
    // ---- reserve room in the row's union and copy the candidates there (coalesced)
    if (tid == 0) {
        const int n = sm.n;
        int base = -1;
        if (nonfinite) atomicOr(P.uflags + row_id, 1);
        else if (too_many || n > CAP_C) atomicOr(P.uflags + row_id, 2);
        else if (n > 0) {
            base = atomicAdd(P.ucount + row_id, n);
            if (base + n > P.cap_u) { atomicOr(P.uflags + row_id, 2); base = -1; }
        }
        sm.base = base;
    }
    __syncthreads();
    if (sm.base >= 0) {
        TopkEntry* dst = P.ulist + (size_t)row_id * P.cap_u + sm.base;
        for (int i = tid; i < sm.n; i += NT) dst[i] = sm.cand[i];
    }
    if (!arrive_last(&P.row_ctr[row_id], (unsigned)P.CT, &sm.flag)) return;
    if (warp != 0) return;

    // ==== one warp of the last CTA of the row
    const RowStats st = topk_row_epilogue<DT>(P, sm, row_id);
    if (lane == 0) P.rstats[row_id] = st;
    if (!warp_arrive_last(&P.req_ctr[b], (unsigned)P.R)) return;

    // ==== the same warp, last row of the request
    int nd = 0;
    for (int rr = lane; rr < P.R; rr += 32) nd += __ldcg(&P.rstats[(size_t)b * P.R + rr].dense);
    nd = __reduce_add_sync(0xffffffffu, nd);
    if (nd > 0) {  // finished by topk_dense_kernel
        if (lane == 0) P.ndense[b] = nd;
        return;
    }
    topk_request_epilogue<DT>(P, sm, b);
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
