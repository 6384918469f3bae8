// sv_tree_sample.cu -- stochastic verification of a candidate tree by the residual update over a
// node's children ("M7.7 - Draft Sources, Dependent Heads, Hardware-Aware Trees", 0x09A; predictor
// row convention 0x07E; accept rule u < min(1, p(x)/q(x)) and the inverse-CDF draw of the Module 16
// speculative-decoding lesson, "The Math: Speculative Sampling").
//
// The walk over a tree is sequential: which row comes next depends on every earlier decision.  So a
// request is one thread-block cluster of CL CTAs that splits the vocabulary into CL slices (and each
// slice into one contiguous run per warp) and walks the tree in lock step, reading only the rows the
// walk visits:
//   - arrival at a node: each warp loads its run of the node's target row and of the first child's
//     proposal row and keeps the target run as fp32 mass 2^(x k2 - c_warp) in shared memory
//     (k2 = log2(e) / T, c_warp = k2 * the run's largest logit);
//   - after a rejection: each warp subtracts Rmass * q from its run in place (the positive residual)
//     and loads the next child's proposal row if it differs;
//   - every exchange: each warp writes its record (offset, mass, proposal offset and mass, and, in
//     the warp owning the next tested token, r(x) and its raw proposal logit), one CTA barrier, warp
//     0 folds the CTA's records into one, one cluster barrier; then every warp reads the CL CTA
//     records through distributed shared memory and takes the same decisions from the same values,
//     so the CTAs stay in step with no flag or spin-wait;
//   - the final token (correction from the residual, or bonus from a leaf's row) is drawn by the one
//     warp whose run holds the uniform's mass, scanning its elements in index order.
#include <cooperative_groups.h>

#include "sv_tree_sample.cuh"

namespace cg = cooperative_groups;

namespace sv {

namespace {

constexpr float TS_LOG2E = 1.4426950408889634f;
constexpr float TS_POS_INF = __builtin_huge_valf();

// One warp's (or CTA's) contribution to an exchange (log2 domain: v is kept as 2^(log2 v - c)).
struct __align__(16) TsRec {
    float c;    // arrival: k2 * the largest target logit (-inf: no finite entry); 0 after a rejection
    float s;    // residual mass at scale 2^-c
    float cq;   // a proposal row loaded in this phase: k2 * its largest logit in the run ...
    float sq;   // ... and the run's sum of 2^(x k2 - cq)
    float rx;   // the owner of the tested token: its residual value, at the scale of s
    float qx;   // ... and its raw proposal logit
    int bad;    // a loaded row holds NaN or +inf
    int pad;
};

__device__ __forceinline__ TsRec ts_blank()
{
    TsRec r;
    r.c = NEG_INF; r.s = 0.f; r.cq = NEG_INF; r.sq = 0.f;
    r.rx = 0.f; r.qx = NEG_INF; r.bad = 0; r.pad = 0;
    return r;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// element e of a 16-byte vector
template <int DT>
__device__ __forceinline__ float ts_val(const uint4& w, int e)
{
    if constexpr (DT == DT_BF16) {
        const uint32_t q = e < 2 ? w.x : e < 4 ? w.y : e < 6 ? w.z : w.w;
        return (e & 1) ? bf16hi(q) : bf16lo(q);
    } else {
        return __uint_as_float(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
    }
}

// elements 4h .. 4h+3 of a 16-byte vector
template <int DT>
__device__ __forceinline__ float4 ts_chunk(const uint4& w, int h)
{
    if constexpr (DT == DT_BF16) {
        const uint32_t a = h ? w.z : w.x, b = h ? w.w : w.y;
        return make_float4(bf16lo(a), bf16hi(a), bf16lo(b), bf16hi(b));
    } else {
        return make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                           __uint_as_float(w.w));
    }
}

// largest element of a vector, NaN if any element is NaN
template <int DT>
__device__ __forceinline__ float ts_vmax_nan(const uint4& w)
{
    if constexpr (DT == DT_BF16) {
        const uint32_t m = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
        return fmax_nan(bf16lo(m), bf16hi(m));
    } else {
        return fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

// Vector j (EPV consecutive elements) of a row: one 16-byte load, or element loads where rows are
// not 16-byte aligned.  Elements at or past V read as -inf.
template <int DT, bool VL>
__device__ __forceinline__ uint4 ts_load(const char* row, long long j, int V, uint64_t pol)
{
    if constexpr (VL) {
        return ld_stream_v4_pol(row + j * 16, pol);
    } else if constexpr (DT == DT_BF16) {
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const long long x = j * 8 + e;
            h[e] = x < V ? (uint32_t)ld_u16_pol(row + x * 2, pol) : 0xff80u;
        }
        return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                          h[6] | (h[7] << 16));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long x = j * 4 + e;
            w[e] = x < V ? ld_u32_pol(row + x * 4, pol) : 0xff800000u;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// element e of register vector i, for a runtime (i, e): a select chain, no local memory
template <int DT, int EPV>
__device__ __forceinline__ float ts_pick(const uint4 (&w)[TS_VPT], int i, int e)
{
    float r = 0.f;
#pragma unroll
    for (int ii = 0; ii < TS_VPT; ++ii)
#pragma unroll
        for (int ee = 0; ee < EPV; ++ee)
            if (ii == i && ee == e) r = ts_val<DT>(w[ii], ee);
    return r;
}

__device__ __forceinline__ float ts_comp(const float4& v, int c)
{
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// The smallest node index > after whose parent is cur (children follow their parent), or -1.
// Every warp computes it; the result is the same everywhere.
__device__ __forceinline__ int ts_next_child(const int* spar, int N, int cur, int after)
{
    const int lane = threadIdx.x & 31;
    for (int base = after + 1; base < N; base += 32) {
        const int i = base + lane;
        const unsigned m = __ballot_sync(0xffffffffu, i < N && spar[i] == cur);
        if (m) return base + __ffs(m) - 1;
    }
    return -1;
}

// Where element x lives: CTA rank, warp, lane, register vector and element within the vector.
struct TsOwner {
    int rank, warp, lane, i, e;
};
template <int EPV>
__device__ __forceinline__ TsOwner ts_owner(int x, int vpt)
{
    TsOwner o;
    const int j = x / EPV;
    const int per_cta = vpt * TS_NT;
    o.rank = j / per_cta;
    const int loc = j - o.rank * per_cta;
    o.warp = loc / (32 * vpt);
    const int r = loc - o.warp * 32 * vpt;
    o.i = r / 32;
    o.lane = r % 32;
    o.e = x % EPV;
    return o;
}

// residual values in shared memory, as float4: chunk h of this lane's vector i at
// ((warp * vpt + i) * RV + h) * 32 + lane, so that a warp's 16-byte accesses are contiguous
template <int RV>
__device__ __forceinline__ int ts_rr4(int warp, int vpt, int i, int h, int lane)
{
    return ((warp * vpt + i) * RV + h) * 32 + lane;
}

template <int DT, bool VL>
__global__ void __launch_bounds__(TS_NT, 2) tree_sample_kernel(const TreeSampleParams P)
{
    constexpr int EPV = DT == DT_BF16 ? 8 : 4;
    constexpr int RV = EPV / 4;
    constexpr uint32_t NEGW = DT == DT_BF16 ? 0xff80ff80u : 0xff800000u;
    const uint4 neg4 = make_uint4(NEGW, NEGW, NEGW, NEGW);

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / CL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = P.N, V = P.V, vpt = P.vpt;
    // first vector of this warp's run; lane l holds vectors vbase + i*32 + l
    const long long vbase = (long long)rank * vpt * TS_NT + (long long)warp * vpt * 32;
    const float k2 = P.invT * TS_LOG2E;

    extern __shared__ __align__(16) unsigned char ts_smem[];
    float4* rr4 = reinterpret_cast<float4*>(ts_smem);                          // residual values
    // the tree description, staged once so that the walk never waits on a global load for it
    int* spar = reinterpret_cast<int*>(rr4 + (size_t)TS_WARPS * vpt * RV * 32);  // [N] parents
    int* stok = spar + N;                                                        // [N] tokens
    int* sqrow = stok + N;                                                       // [N] proposal rows
    float* su = reinterpret_cast<float*>(sqrow + N);                             // [N+1] uniforms
    // outputs kept in shared memory until the walk ends (CTA 0), so that no global store sits
    // before a cluster barrier, whose release would wait for it
    float* sacc = su + N + 1;                                                    // [N] accept ratios
    int* spath = reinterpret_cast<int*>(sacc + N);                               // [N] path nodes
    __shared__ TsRec wrec[TS_WARPS];  // this CTA's warp records
    __shared__ TsRec crec[2];         // this CTA's record, read by the cluster; double-buffered
    __shared__ int s_draw;            // CTA 0: the drawn token, sent by the drawing warp

    const size_t es = DT == DT_BF16 ? 2 : 4;
    const char* tbase = static_cast<const char*>(P.target) + (size_t)b * (N + 1) * V * es;
    const char* dbase = static_cast<const char*>(P.draft) + (size_t)b * P.Nq * V * es;
    const int32_t* par_g = P.parents + (size_t)b * N;
    const int32_t* tok_g = P.tokens + (size_t)b * N;
    const int32_t* qrow_g = P.qrow + (size_t)b * N;
    const float* ug = P.uniforms + (size_t)b * (N + 1);
    const uint64_t pol = policy_evict_first();

    // ---- the tree description: into shared memory, and what it fixes before any row is read
    int e_par = 0, e_q = 0, e_tok = 0, e_u = 0;
    for (int i = tid; i < N; i += TS_NT) {
        const int pr = __ldg(par_g + i);
        spar[i] = pr;
        e_par |= (pr < -1 || pr >= i);
        const int qr = __ldg(qrow_g + i);
        sqrow[i] = qr;
        e_q |= (qr < 0 || qr >= P.Nq);
        const int tk = __ldg(tok_g + i);
        stok[i] = tk;
        e_tok |= (tk < 0 || tk >= V);
        sacc[i] = __int_as_float(0x7fc00000);
    }
    for (int i = tid; i <= N; i += TS_NT) {
        const float u = __ldg(ug + i);
        su[i] = u;
        e_u |= !(u >= 0.f && u < 1.f);
    }
    if (tid == 0) s_draw = -1;
    e_par = __syncthreads_or(e_par);
    e_q = __syncthreads_or(e_q);
    e_tok = __syncthreads_or(e_tok);
    e_u = __syncthreads_or(e_u);
    int st = e_par ? ROW_BAD_PARENT : e_q ? ROW_BAD_QROW : e_tok ? ROW_BAD_TOKEN
           : e_u ? ROW_BAD_UNIFORM : ROW_OK;

    // ---- the walk (identical control flow in every thread of every CTA of the cluster)
    int cur = -1, n = 0, ph = 0;
    int qcur = -1;       // proposal row held in qw
    float Cq = 0.f;      // its offset: k2 * its largest logit
    float Sq = 1.f;      // its sum of 2^(x k2 - Cq)
    float G = 0.f;       // offset of the current node's target row
    float Rmass = 0.f;   // mass of the current residual, at scale 2^-G
    float cw = NEG_INF;  // this warp's target offset at the last arrival
    float sc = 1.f;      // this warp's scale: residual value = rr * sc
    float ck = 0.f;      // lane k < CL: mass of CTA k's slice (for the draw)
    bool draw = false, last_arrival = false;
    uint4 qw[TS_VPT];
#pragma unroll
    for (int i = 0; i < TS_VPT; ++i) qw[i] = neg4;

    // loads this lane's vectors of a row
    auto load_row = [&](const char* row, uint4 (&w)[TS_VPT]) {
#pragma unroll
        for (int i = 0; i < TS_VPT; ++i) {
            const long long j = vbase + (long long)i * 32 + lane;
            w[i] = (i < vpt && j < P.nvec) ? ts_load<DT, VL>(row, j, V, pol) : neg4;
        }
    };
    // the run's statistics of the proposal row in qw: offset, sum of 2^(x k2 - offset), bad
    auto q_stats = [&](float& cq, float& sq, int& bad) {
        float m = NEG_INF;
#pragma unroll
        for (int i = 0; i < TS_VPT; ++i) m = fmax_nan(m, ts_vmax_nan<DT>(qw[i]));
        bad |= !(m == m) | (m == TS_POS_INF);
        m = warp_max(m);
        const float off = m == NEG_INF ? 0.f : m * k2;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < TS_VPT; ++i)
            if (i < vpt)
#pragma unroll
                for (int h = 0; h < RV; ++h) {
                    const float4 x = ts_chunk<DT>(qw[i], h);
                    s += (ex2(fmaf(x.x, k2, -off)) + ex2(fmaf(x.y, k2, -off))) +
                         (ex2(fmaf(x.z, k2, -off)) + ex2(fmaf(x.w, k2, -off)));
                }
        cq = m == NEG_INF ? NEG_INF : off;
        sq = warp_sum(s);
    };
    // one exchange: this warp's record (the warp owning token x adds r(x) and its raw proposal
    // logit), the CTA fold by warp 0, the cluster barrier; returns, in lane k < CL, CTA k's record
    auto exchange = [&](float c, float s, float cq, float sq, int bad, int x, TsOwner& o) {
        float rx = 0.f, qx = NEG_INF;
        if (x >= 0) {
            o = ts_owner<EPV>(x, vpt);
            if (rank == o.rank && warp == o.warp && lane == o.lane) {
                rx = ts_comp(rr4[ts_rr4<RV>(warp, vpt, o.i, o.e >> 2, lane)], o.e & 3);
                qx = ts_pick<DT, EPV>(qw, o.i, o.e);
            }
            rx = __shfl_sync(0xffffffffu, rx, o.lane);
            qx = __shfl_sync(0xffffffffu, qx, o.lane);
        }
        if (lane == 0) {
            TsRec R;
            R.c = c; R.s = s; R.cq = cq; R.sq = sq; R.rx = rx; R.qx = qx; R.bad = bad; R.pad = 0;
            wrec[warp] = R;
        }
        __syncthreads();
        if (warp == 0) {
            TsRec R = ts_blank();
            if (lane < TS_WARPS) R = wrec[lane];
            TsRec F;
            const float C = warp_max(R.c);
            const float f = (R.c == NEG_INF) ? 0.f : ex2(R.c - C);
            F.c = C;
            F.s = warp_sum(R.s * f);
            const float Cq2 = warp_max(R.cq);
            F.cq = Cq2;
            F.sq = warp_sum((R.cq == NEG_INF) ? 0.f : R.sq * ex2(R.cq - Cq2));
            F.rx = __shfl_sync(0xffffffffu, R.rx * f, o.warp);
            F.qx = __shfl_sync(0xffffffffu, R.qx, o.warp);
            F.bad = __any_sync(0xffffffffu, R.bad);
            F.pad = 0;
            if (lane == 0) crec[ph] = F;
        }
        cluster.sync();
        TsRec K = ts_blank();
        if (lane < CL) K = *cluster.map_shared_rank(&crec[ph], lane);
        ph ^= 1;
        return K;
    };
    // combined offset and mass of the CTA records: max c, and sum s * 2^(c - max) (also per lane)
    auto fold = [&](float c, float s, float& C, float& S) {
        C = warp_max(c);
        const float w = (c == NEG_INF) ? 0.f : s * ex2(c - C);
        S = warp_sum(w);
        return w;
    };

    while (st == ROW_OK) {
        // ---------------- arrival at node cur: its target row and its first child's proposal row
        int s = ts_next_child(spar, N, cur, cur);
        const int qr = s >= 0 ? sqrow[s] : -1;
        const bool newq = s >= 0 && qr != qcur;
        int bad = 0;
        float tm = NEG_INF, tsum = 0.f;
        {
            uint4 tw[TS_VPT];
            load_row(tbase + (size_t)(cur + 1) * V * es, tw);
            if (newq) load_row(dbase + (size_t)qr * V * es, qw);
#pragma unroll
            for (int i = 0; i < TS_VPT; ++i) tm = fmax_nan(tm, ts_vmax_nan<DT>(tw[i]));
            bad |= !(tm == tm) | (tm == TS_POS_INF);
            tm = warp_max(tm);
            const float off = tm == NEG_INF ? 0.f : tm * k2;
#pragma unroll
            for (int i = 0; i < TS_VPT; ++i)
                if (i < vpt)
#pragma unroll
                    for (int h = 0; h < RV; ++h) {
                        const float4 x = ts_chunk<DT>(tw[i], h);
                        float4 r;
                        r.x = ex2(fmaf(x.x, k2, -off));
                        r.y = ex2(fmaf(x.y, k2, -off));
                        r.z = ex2(fmaf(x.z, k2, -off));
                        r.w = ex2(fmaf(x.w, k2, -off));
                        rr4[ts_rr4<RV>(warp, vpt, i, h, lane)] = r;
                        tsum += (r.x + r.y) + (r.z + r.w);
                    }
            cw = tm == NEG_INF ? NEG_INF : off;
        }
        tsum = warp_sum(tsum);
        float qc = NEG_INF, qsum = 0.f;
        if (newq) q_stats(qc, qsum, bad);
        bad = __any_sync(0xffffffffu, bad);
        TsOwner o = {0, 0, 0, 0, 0};
        const TsRec K = exchange(cw, tsum, qc, qsum, bad, s >= 0 ? stok[s] : -1, o);
        float rx = 0.f, qx = NEG_INF;
        bool dead;
        {  // combine the CTA records (every warp, same values everywhere)
            ck = fold(K.c, K.s, G, Rmass);
            sc = (cw == NEG_INF) ? 0.f : ex2(cw - G);
            dead = __any_sync(0xffffffffu, K.bad) || G == NEG_INF;
            if (newq) {
                fold(K.cq, K.sq, Cq, Sq);
                qcur = qr;
                dead |= (Cq == NEG_INF);
            }
            if (s >= 0) {
                const float Ko = __shfl_sync(0xffffffffu, K.c, o.rank);
                rx = __shfl_sync(0xffffffffu, K.rx, o.rank) * ((Ko == NEG_INF) ? 0.f : ex2(Ko - G));
                qx = __shfl_sync(0xffffffffu, K.qx, o.rank);
            }
        }
        last_arrival = true;
        if (dead) {
            st = ROW_NONFINITE;
            break;
        }

        // ---------------- the children of cur, in ascending index, against the running residual
        bool moved = false;
        while (s >= 0) {
            if (qx == NEG_INF) {  // q(x) = 0: the proposal row could not have drawn x
                st = ROW_BAD_TOKEN;
                break;
            }
            // a = r(x) / (Rmass q(x)), with q(x) Sq = 2^(qx k2 - Cq)
            const float dq = fmaf(qx, k2, -Cq);
            float a;
            if (!(rx > 0.f)) a = 0.f;
            else if (dq > -120.f) a = fminf(1.f, rx * ex2(-dq) * (Sq / Rmass));
            else a = fminf(1.f, ex2(lg2(rx) - dq + lg2(Sq) - lg2(Rmass)));
            if (tid == 0) sacc[s] = a;
            if (su[s] < a) {  // accepted: the walk moves to s
                if (tid == 0) spath[n] = s;
                ++n;
                cur = s;
                moved = true;
                if (n + 1 > P.max_out) st = ROW_OVERFLOW;
                break;
            }
            // rejected: r <- max(r - Rmass * q_s, 0), with Rmass * q_s(v) = 2^(x_v k2 - Cq + c2)
            const float c2 = lg2(Rmass) - lg2(Sq);
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < TS_VPT; ++i)
                if (i < vpt)
#pragma unroll
                    for (int h = 0; h < RV; ++h) {
                        const int id = ts_rr4<RV>(warp, vpt, i, h, lane);
                        const float4 x = ts_chunk<DT>(qw[i], h);
                        float4 v = rr4[id];
                        v.x = fmaxf(fmaf(v.x, sc, -ex2(fmaf(x.x, k2, -Cq) + c2)), 0.f);
                        v.y = fmaxf(fmaf(v.y, sc, -ex2(fmaf(x.y, k2, -Cq) + c2)), 0.f);
                        v.z = fmaxf(fmaf(v.z, sc, -ex2(fmaf(x.z, k2, -Cq) + c2)), 0.f);
                        v.w = fmaxf(fmaf(v.w, sc, -ex2(fmaf(x.w, k2, -Cq) + c2)), 0.f);
                        rr4[id] = v;
                        psum += (v.x + v.y) + (v.z + v.w);
                    }
            psum = warp_sum(psum);
            sc = 1.f;
            const int s2 = ts_next_child(spar, N, cur, s);
            const int qr2 = s2 >= 0 ? sqrow[s2] : -1;
            const bool newq2 = s2 >= 0 && qr2 != qcur;
            float qc2 = NEG_INF, qsum2 = 0.f;
            int bad2 = 0;
            if (newq2) {  // the next child was drawn from another proposal row
                load_row(dbase + (size_t)qr2 * V * es, qw);
                q_stats(qc2, qsum2, bad2);
                bad2 = __any_sync(0xffffffffu, bad2);
            }
            TsOwner o2 = {0, 0, 0, 0, 0};
            const TsRec K2 = exchange(0.f, psum, qc2, qsum2, bad2, s2 >= 0 ? stok[s2] : -1, o2);
            bool dead2;
            {
                float unused;
                ck = fold(K2.c, K2.s, unused, Rmass);
                dead2 = __any_sync(0xffffffffu, K2.bad);
                if (newq2) {
                    fold(K2.cq, K2.sq, Cq, Sq);
                    qcur = qr2;
                    dead2 |= (Cq == NEG_INF);
                }
                if (s2 >= 0) {
                    rx = __shfl_sync(0xffffffffu, K2.rx, o2.rank);
                    qx = __shfl_sync(0xffffffffu, K2.qx, o2.rank);
                }
            }
            last_arrival = false;
            if (!(Rmass > 0.f)) {
                st = ROW_DEGENERATE;
                break;
            }
            if (dead2) {
                st = ROW_NONFINITE;
                break;
            }
            s = s2;
        }
        if (st != ROW_OK) break;
        if (moved) continue;
        draw = true;  // every child rejected (correction from r), or a leaf (bonus from p = r)
        break;
    }

    // ---- the final draw: the CTA, then the warp, whose run holds u * Rmass scans it in order
    if (draw) {
        const float tpos = su[N] * Rmass;
        const float cum = warp_incl_scan(lane < CL ? ck : 0.f);
        const unsigned hit = __ballot_sync(0xffffffffu, lane < CL && ck > 0.f && tpos < cum);
        const unsigned pos = __ballot_sync(0xffffffffu, lane < CL && ck > 0.f);
        const int kd = hit ? __ffs(hit) - 1 : 31 - __clz(pos);
        const float tp = tpos - __shfl_sync(0xffffffffu, cum - ck, kd & 31);
        if (rank == kd) {
            // this CTA's warp masses at the final scale (records of the last exchange)
            TsRec R = ts_blank();
            if (lane < TS_WARPS) R = wrec[lane];
            const float mwl = last_arrival ? ((R.c == NEG_INF) ? 0.f : R.s * ex2(R.c - G)) : R.s;
            const float cumw = warp_incl_scan(mwl);
            const unsigned hw = __ballot_sync(0xffffffffu, lane < TS_WARPS && mwl > 0.f && tp < cumw);
            const unsigned pw = __ballot_sync(0xffffffffu, lane < TS_WARPS && mwl > 0.f);
            const int wd = hw ? __ffs(hw) - 1 : 31 - __clz(pw);
            const float tq = tp - __shfl_sync(0xffffffffu, cumw - mwl, wd & 31);
            if (warp == wd) {
                // this warp's vectors in index order: i major, lane minor
                float vrun = 0.f, bstart = 0.f;
                int best = -1;
#pragma unroll
                for (int i = 0; i < TS_VPT; ++i) {
                    if (i < vpt) {
                        float w = 0.f;
#pragma unroll
                        for (int h = 0; h < RV; ++h) {
                            const float4 v = rr4[ts_rr4<RV>(warp, vpt, i, h, lane)];
                            w += (v.x + v.y) + (v.z + v.w);
                        }
                        w *= sc;
                        const float inc = warp_incl_scan(w);
                        const float start = vrun + (inc - w);
                        if (w > 0.f && start <= tq) {
                            best = i * 32 + lane;
                            bstart = start;
                        }
                        vrun += __shfl_sync(0xffffffffu, inc, 31);
                    }
                }
                int top = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
                if (top >= 0 && best == top) {
                    const int i = best / 32;
                    float c = bstart;
                    int y = -1, last = -1;
#pragma unroll
                    for (int h = 0; h < RV; ++h) {
                        const float4 v = rr4[ts_rr4<RV>(warp, vpt, i, h, lane)];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float val = ts_comp(v, e) * sc;
                            if (val > 0.f) {
                                last = h * 4 + e;
                                c += val;
                                if (y < 0 && tq < c) y = h * 4 + e;
                            }
                        }
                    }
                    if (y < 0) y = last;
                    *cluster.map_shared_rank(&s_draw, 0) = (int)((vbase + best) * EPV + y);
                }
            }
        }
    }

    // the drawn token reaches CTA 0; after this barrier no CTA touches another's shared memory
    cluster.sync();

    // ---- outputs of the request (CTA 0)
    if (rank == 0) {
        if (draw && s_draw < 0) st = ROW_DEGENERATE;  // no positive mass found (underflow)
        const bool ok = (st == ROW_OK);
        int32_t* out = P.out_tokens + (size_t)b * P.max_out;
        for (int i = tid; i < P.max_out; i += TS_NT)
            out[i] = !ok ? -1 : i < n ? stok[spath[i]] : i == n ? s_draw : -1;
        if (P.out_nodes) {
            int32_t* onodes = P.out_nodes + (size_t)b * (P.max_out - 1);
            for (int i = tid; i < P.max_out - 1; i += TS_NT) onodes[i] = (ok && i < n) ? spath[i] : -1;
        }
        if (P.aux_accept)
            for (int i = tid; i < N; i += TS_NT) P.aux_accept[(size_t)b * N + i] = sacc[i];
        if (tid == 0) {
            P.accepted_len[b] = ok ? n : -1;
            if (P.row_status) P.row_status[b] = st;
        }
    }
}

template <int DT, bool VL>
cudaError_t launch_one(const TreeSampleParams& P, int CL, size_t smem, cudaStream_t st)
{
    auto* k = tree_sample_kernel<DT, VL>;
    // static records (16 KB) plus the dynamic part can pass the 48 KB default: always opt in
    static size_t smem_set = 0;
    if (smem > smem_set) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)P.B * CL));
    cfg.blockDim = dim3(TS_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (CL > 8) {  // above the portable cluster size: opt in, and make sure one cluster fits
        static bool opted = false;
        if (!opted) {
            const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            opted = true;
        }
        int clusters = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
    }
    mark_kernel_start(st);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, P);
    mark_kernel_stop(st);
    return e;
}

}  // namespace

size_t tree_sample_smem(int vpt, int dtype, int N)
{
    const int EPV = dtype == DT_BF16 ? 8 : 4;
    return (size_t)vpt * EPV * TS_NT * sizeof(float) + (size_t)(6 * N + 1) * sizeof(int);
}

cudaError_t launch_tree_sample(const TreeSampleParams& P, int CL, bool vec16, cudaStream_t st)
{
    const size_t smem = tree_sample_smem(P.vpt, P.dtype, P.N);
    if (P.dtype == DT_BF16)
        return vec16 ? launch_one<DT_BF16, true>(P, CL, smem, st) : launch_one<DT_BF16, false>(P, CL, smem, st);
    return vec16 ? launch_one<DT_F32, true>(P, CL, smem, st) : launch_one<DT_F32, false>(P, CL, smem, st);
}

}  // namespace sv
