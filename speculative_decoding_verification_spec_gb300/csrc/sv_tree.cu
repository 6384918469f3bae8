// sv_tree.cu -- Medusa-style greedy tree verify (Module 16 lesson, "Verify the Tree -- and Why It's
// Exact"; M7.7 section 0x07E for the predictor-row convention).
//
// Rows of 16-byte vectors: one CTA per contiguous chunk, loaded into registers (see
// tree_argmax_chunk_kernel).  Other rows: persistent warps with plain loads, where a warp task is
// (request, row, slice of TV1 vectors) and the hot loop keeps, per lane, only the running maximum
// and the step where it was first reached; after the task, the lanes holding the warp maximum
// re-read that one step to find the first index of the maximum, so ties go to the lowest index.  The warp that completes a
// request merges the partials of every row in slice order, walks the tree in node order (a node's
// parent always precedes it), picks the deepest valid node and writes the path and the bonus.
#include "sv_tree_walk.cuh"

namespace sv {

// (value, index) order: larger value first, then the lower index
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

// maximum of one step (U1 vectors per lane); NaN if any element is NaN
template <int DT, int VEC>
__device__ __forceinline__ float step_max(const char* row, long long base, long long t1, uint64_t pol)
{
    if constexpr (DT == DT_BF16 && VEC == 8) {
        uint4 w[U1];
#pragma unroll
        for (int u = 0; u < U1; ++u) {
            const long long v = base + u * 32;
            if (v < t1) w[u] = ld_stream_v4_pol(row + v * 16, pol);
            else w[u] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
        }
        uint32_t pm = bmax2_nan(bmax2_nan(w[0].x, w[0].y), bmax2_nan(w[0].z, w[0].w));
#pragma unroll
        for (int u = 1; u < U1; ++u)
            pm = bmax2_nan(pm, bmax2_nan(bmax2_nan(w[u].x, w[u].y), bmax2_nan(w[u].z, w[u].w)));
        return fmax_nan(bf16lo(pm), bf16hi(pm));
    } else {
        float x[U1][VEC];
#pragma unroll
        for (int u = 0; u < U1; ++u) {
            const long long v = base + u * 32;
            if (v < t1) {
                load_vec_pol<DT, VEC>(row, v, pol, x[u]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) x[u][e] = NEG_INF;
            }
        }
        float bm = NEG_INF;
#pragma unroll
        for (int u = 0; u < U1; ++u)
#pragma unroll
            for (int e = 0; e < VEC; ++e) bm = fmax_nan(bm, x[u][e]);
        return bm;
    }
}

// first element index equal to `target` in one step of this lane (index order), or INT_MAX; all
// U1 loads are issued before the first compare
template <int DT, int VEC>
__device__ __forceinline__ int step_find(const char* row, long long base, long long t1, float target)
{
    RawVec<DT, VEC> x[U1];
#pragma unroll
    for (int u = 0; u < U1; ++u) {
        x[u].fill_neg_inf();
        if (base + u * 32 < t1) x[u].load(row, base + u * 32, policy_evict_first());
    }
    int found = 0x7fffffff;
#pragma unroll
    for (int u = U1 - 1; u >= 0; --u)
#pragma unroll
        for (int e = VEC - 1; e >= 0; --e)
            if (base + u * 32 < t1 && x[u].get(e) == target) found = (int)((base + u * 32) * VEC + e);
    return found;
}

__device__ void tree_walk_and_emit(const TreeParams& P, int b, int bad, const int32_t* par,
                                   const int32_t* tok, const int32_t* am, int32_t* depth,
                                   int32_t* valid);

// The warp that completed request b: per-row argmax in slice order, the walk, the outputs.
__device__ void tree_finish_request(const TreeParams& P, int b)
{
    const int lane = threadIdx.x & 31;
    // ---- this warp completed the request: per-row argmax in slice order
    int bad = 0;
    for (int j = lane; j < P.R; j += 32) {
        const ArgmaxPartial* pp = P.partials + ((size_t)b * P.R + j) * P.S1;
        float bv = NEG_INF;
        int bi = 0x7fffffff, bn = 0;
        for (int k = 0; k < P.S1; ++k) {
            const float v = __ldcg(&pp[k].best);
            const int i = __ldcg(&pp[k].idx);
            bn |= __ldcg(&pp[k].nan);
            if (better(v, i, bv, bi)) { bv = v; bi = i; }
        }
        const bool ok = !bn && bi != 0x7fffffff && bv != NEG_INF;  // all -inf: no token
        if (!ok) bad = 1;
        P.amax[(size_t)b * P.R + j] = ok ? bi : -1;
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    int32_t* depth = P.scratch + (size_t)b * P.N * 2;
    tree_walk_and_emit(P, b, bad, P.parents ? P.parents + (size_t)b * P.N : nullptr,
                       P.tokens + (size_t)b * P.N,
                       P.amax + (size_t)b * P.R, depth, depth + P.N);
}

// One warp: the greedy walk (a node passes when its token is its predictor row's argmax, am[row])
// and the outputs, with the argmax of the accepted node's own row as the token after the path.
__device__ void tree_walk_and_emit(const TreeParams& P, int b, int bad, const int32_t* par,
                                   const int32_t* tok, const int32_t* am, int32_t* depth,
                                   int32_t* valid)
{
    const TreeWalk w = tree_walk(P.N, P.V, P.max_out, bad, 0, par, tok,
                                 [&](int i, int p) { return tok[i] == am[p < 0 ? 0 : p + 1]; },
                                 depth, valid);
    tree_emit(P, b, w, par, tok, w.st == ROW_OK ? am[w.node < 0 ? 0 : w.node + 1] : -1);
}

// End of an argmax task: the lanes holding the warp maximum locate its first index (ties to the
// lowest index), lane 0 stores the slice partial, and the warp completing the request finishes it.
template <int DT, int VEC>
__device__ __forceinline__ void tree_finalize(const TreeParams& P, const char* row, int b, int r, int s,
                                              long long t1, float best, int best_step, int nan)
{
    const int lane = threadIdx.x & 31;
    const long long t0 = (long long)s * TV1;
    const float W = warp_max(best);
    int idx = 0x7fffffff;
    if (best == W && best_step >= 0)
        idx = step_find<DT, VEC>(row, t0 + (long long)best_step * 32 * U1 + lane, t1, W);
    idx = __reduce_min_sync(0xffffffffu, idx);
    nan = __any_sync(0xffffffffu, nan);
    if (lane == 0) {
        ArgmaxPartial pt;
        pt.best = W;
        pt.idx = idx;
        pt.nan = nan;
        pt.pad = 0;
        P.partials[((size_t)b * P.R + r) * P.S1 + s] = pt;
    }
    if (warp_arrive_last(&P.req_ctr[b], (unsigned)(P.R * P.S1))) tree_finish_request(P, b);
}

__device__ __forceinline__ void decode_tree_task(const TreeParams& P, long long t, int& b, int& r, int& s)
{
    s = (int)(t % P.S1);
    const long long rr = t / P.S1;
    b = (int)(rr / P.R);
    r = (int)(rr % P.R);
}

__device__ __forceinline__ const char* tree_row(const TreeParams& P, int b, int r)
{
    const size_t es = (P.dtype == DT_BF16) ? 2 : 4;
    return reinterpret_cast<const char*>(P.logits) + ((size_t)b * P.R + r) * (size_t)P.V * es;
}

// Scalar-path kernel (rows not 16-byte aligned).
template <int DT, int VEC>
__global__ void __launch_bounds__(NT) tree_argmax_kernel(TreeParams P)
{
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    long long t = claim_task(&P.work[0]);
    while (t < P.tasks) {
        const long long next = claim_task(&P.work[0]);
        int b, r, s;
        decode_tree_task(P, t, b, r, s);
        const char* row = tree_row(P, b, r);
        const long long t0 = (long long)s * TV1;
        const long long t1 = min(t0 + TV1, P.nvec);
        float best = NEG_INF;
        int best_step = -1, nan = 0;
#pragma unroll 1
        for (int step = 0; step < ST1; ++step) {
            const long long sb = t0 + (long long)step * 32 * U1;
            if (sb >= t1) break;
            const float bm = step_max<DT, VEC>(row, sb + lane, t1, pol);
            if (bm != bm) nan = 1;
            else if (bm > best) { best = bm; best_step = step; }
        }
        tree_finalize<DT, VEC>(P, row, b, r, s, t1, best, best_step, nan);
        t = next;
    }
}

// consumer groups per CTA of the streaming argmax (see ring_produce): one, with two CTAs per SM;
// two groups in one CTA per SM gave the same time
constexpr int TREE_GROUPS = 1;

// Streaming argmax for rows of 16-byte vectors: persistent CTAs take 32 KB chunks round-robin,
// fetched by bulk copies into a ring of shared-memory stages.  Each thread finds its maximum (via
// the maxima of its vectors) and the first of its elements equal to it -- its vectors and their
// elements are in index order -- and each warp reduces (value, index) with ties to the lower
// index into one partial per (chunk, warp).  A NaN anywhere marks the partial.  Warp-specialised:
// a producer warp fills the ring (ring_produce) and the consumer warps release each stage on its
// "empty" mbarrier, so they never wait for one another.
template <int DT>
__global__ void __launch_bounds__(stream_threads<TREE_GROUPS>(), 2 / TREE_GROUPS) tree_stream_kernel(TreeParams P)
{
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    constexpr int ES = (DT == DT_BF16) ? 2 : 4;
    constexpr int CHUNK = NT * STREAM_NV * VEC;
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) uint64_t full[TREE_GROUPS * STREAM_STAGES];
    __shared__ __align__(8) uint64_t empty[TREE_GROUPS * STREAM_STAGES];
    __shared__ int sfail;  // a wait ran out in this CTA: nothing more is read
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int nch = P.B * P.R * P.S1;
    if (tid == 0) {
        sfail = 0;
        for (int s = 0; s < TREE_GROUPS * STREAM_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == TREE_GROUPS * WARPS) {  // the producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            ring_produce<TREE_GROUPS>(full, empty, &sfail, nch, P.wait_limit, [&](int s, int id) {
                const int row_id = id / P.S1, ci = id - row_id * P.S1;
                const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, P.V);
                bulk_load(ring + (size_t)s * NT * STREAM_NV,
                          reinterpret_cast<const char*>(P.logits) + ((size_t)row_id * P.V + cbase) * ES,
                          (unsigned)(cend - cbase) * ES, &full[s], pol);
            });
        }
        return;
    }
    const StreamGroup<TREE_GROUPS> sg;
    uint64_t* gfull = full + sg.g * STREAM_STAGES;
    uint64_t* gempty = empty + sg.g * STREAM_STAGES;
    const uint4* gring = ring + (size_t)sg.g * STREAM_STAGES * NT * STREAM_NV;
    const int tid_g = sg.t;  // thread within the group

    bool failed = false;
    int stg = 0;          // it % STREAM_STAGES
    unsigned phase = 0;   // (it / STREAM_STAGES) & 1
    // chunk id = row_id * S1 + ci, advanced by the stride without a division per chunk
    int row_id = sg.vb / P.S1, ci = sg.vb - row_id * P.S1;
    const int drow = sg.stride / P.S1, dci = sg.stride - drow * P.S1;
    for (int id = sg.vb; id < nch; id += sg.stride) {
        if (id != sg.vb) {
            row_id += drow;
            ci += dci;
            if (ci >= P.S1) {
                ci -= P.S1;
                ++row_id;
            }
            if (++stg == STREAM_STAGES) {
                stg = 0;
                phase ^= 1u;
            }
        }
        const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, P.V);
        const int s = stg;
        if (!failed && *reinterpret_cast<volatile int*>(&sfail)) failed = true;
        bool ok = !failed && mbar_wait(&gfull[s], phase, P.wait_limit);
        const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
        const uint4* sb = gring + (size_t)s * NT * STREAM_NV;
        uint4 w[STREAM_NV];
        float vmax[STREAM_NV];
        int nin = 0;  // vectors of this thread inside the row
#pragma unroll
        for (int j = 0; j < STREAM_NV; ++j) {
            const bool in = cbase + (j * NT + tid_g) * VEC < cend;
            nin += in;
            w[j] = make_uint4(pad, pad, pad, pad);
            if (ok && in) w[j] = lds128(sb + j * NT + tid_g);
        }
        // release the stage once every lane has read it; a warp whose wait ran out never releases
        // it (its copy may still land), which stops the producer
        ok = __all_sync(FULL, ok);
        if (ok) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gempty[s]);
        } else if (!failed) {
            failed = true;
            if (lane == 0) *reinterpret_cast<volatile int*>(&sfail) = 1;
        }
        ArgmaxPartial pt;
        pt.pad = 0;
        if (failed) {
            pt.best = NEG_INF;
            pt.idx = 0x7fffffff;
            pt.nan = 2;  // the chunk was not read
        } else {
            float tm = NEG_INF;
#pragma unroll
            for (int j = 0; j < STREAM_NV; ++j) {
                if constexpr (DT == DT_BF16) {
                    const uint32_t pm = bmax2_nan(bmax2_nan(w[j].x, w[j].y), bmax2_nan(w[j].z, w[j].w));
                    vmax[j] = fmax_nan(bf16lo(pm), bf16hi(pm));
                } else {
                    vmax[j] = fmax_nan(fmax_nan(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                                       fmax_nan(__uint_as_float(w[j].z), __uint_as_float(w[j].w)));
                }
                tm = fmax_nan(tm, vmax[j]);
            }
            const int nan = tm != tm;
            int idx = 0x7fffffff;
            if (!nan && nin > 0) {
                int jf = 0;
#pragma unroll
                for (int j = STREAM_NV - 1; j >= 0; --j)
                    if (vmax[j] == tm) jf = j;
                uint4 v = w[0];
#pragma unroll
                for (int j = 1; j < STREAM_NV; ++j)
                    if (j == jf) v = w[j];
                int ef = 0;
                if constexpr (DT == DT_BF16) {
                    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 7; e >= 0; --e) {
                        const float x = (e & 1) ? bf16hi(q[e >> 1]) : bf16lo(q[e >> 1]);
                        if (x == tm) ef = e;
                    }
                } else {
                    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 3; e >= 0; --e)
                        if (__uint_as_float(q[e]) == tm) ef = e;
                }
                idx = cbase + (jf * NT + tid_g) * VEC + ef;
            }
            // warp: maximum value, then the lowest index holding it
            float bv = nan ? NEG_INF : tm;
            int bi = idx;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            pt.best = bv;
            pt.idx = bi;
            pt.nan = __any_sync(0xffffffffu, nan);
        }
        if (lane == 0) P.partials[((size_t)row_id * P.S1 + ci) * WARPS + sg.w] = pt;
    }
}

// One CTA per request: the warps merge the rows' partials (rows round-robin, every partial of a
// warp's rows in flight together), then warp 0 walks the tree.  When the tree fits
// (N <= TREE_SMEM_NODES) the walk runs entirely in shared memory -- parents, tokens, the rows'
// argmaxes, depth and validity: dynamic shared memory of 4 N + R ints.
constexpr int TREE_SMEM_NODES = 4096;

template <int DT>
__global__ void __launch_bounds__(NT) tree_finish_kernel(TreeParams P)
{
    extern __shared__ int32_t tsm[];  // par[N], tok[N], depth[N], valid[N], am[R]
    __shared__ int sh_bad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, N = P.N, R = P.R;
    const bool staged = N <= TREE_SMEM_NODES;
    const int32_t* par = staged ? tsm : P.parents ? P.parents + (size_t)b * N : nullptr;
    const int32_t* tok = staged ? tsm + N : P.tokens + (size_t)b * N;
    int32_t* depth = staged ? tsm + 2 * N : P.scratch + (size_t)b * N * 2;
    int32_t* valid = staged ? tsm + 3 * N : P.scratch + (size_t)b * N * 2 + N;
    int32_t* am = staged ? tsm + 4 * N : P.amax + (size_t)b * R;
    if (staged)
        for (int i = tid; i < N; i += NT) {
            tsm[i] = P.parents ? __ldg(P.parents + (size_t)b * N + i) : i - 1;  // null: a chain
            tsm[N + i] = __ldg(P.tokens + (size_t)b * N + i);
        }
    if (tid == 0) sh_bad = 0;
    pdl_wait();  // the partials of the streaming kernel
    __syncthreads();
    const int np = P.S1 * WARPS;  // partials per row
    int bad = 0;
    constexpr int RPW = 9;  // rows of a warp in flight together (one round trip for R <= 72)
    for (int j0 = warp; j0 < R; j0 += WARPS * RPW) {
        int4 q[RPW][2];  // (best, idx, nan, pad) of two partials per lane for each row
#pragma unroll
        for (int t = 0; t < RPW; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = j0 + t * WARPS, k = lane + 32 * h;
                q[t][h] = make_int4(__float_as_int(NEG_INF), 0x7fffffff, 0, 0);
                if (j < R && k < np)
                    q[t][h] = __ldcg(reinterpret_cast<const int4*>(P.partials + ((size_t)b * R + j) * np + k));
            }
#pragma unroll
        for (int t = 0; t < RPW; ++t) {
            const int j = j0 + t * WARPS;
            if (j >= R) break;  // j is the same for every lane
            float bv = __int_as_float(q[t][0].x);
            int bi = q[t][0].y, bn = max(q[t][0].z, q[t][1].z);
            if (better(__int_as_float(q[t][1].x), q[t][1].y, bv, bi)) { bv = __int_as_float(q[t][1].x); bi = q[t][1].y; }
            for (int k = lane + 64; k < np; k += 32) {  // rows with more than 64 partials
                const int4 e = __ldcg(reinterpret_cast<const int4*>(P.partials + ((size_t)b * R + j) * np + k));
                bn = max(bn, e.z);
                if (better(__int_as_float(e.x), e.y, bv, bi)) { bv = __int_as_float(e.x); bi = e.y; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            const int btmo = __any_sync(0xffffffffu, bn == 2);
            bn = __any_sync(0xffffffffu, bn);
            const bool ok = !bn && bi != 0x7fffffff && bv != NEG_INF;  // all -inf: no token
            if (!ok) bad = btmo ? 2 : max(bad, 1);
            if (lane == 0) am[j] = ok ? bi : -1;
        }
    }
    if (bad && lane == 0) atomicMax(&sh_bad, bad);
    __syncthreads();
    if (warp == 0) tree_walk_and_emit(P, b, sh_bad, par, tok, am, depth, valid);
}

template <int DT, int VEC>
static void launch_tree_plain(const TreeParams& P, int sms, cudaStream_t st)
{
    mark_kernel_start(st);
    tree_argmax_kernel<DT, VEC><<<persistent_grid<tree_argmax_kernel<DT, VEC>>(P.tasks, sms), NT, 0, st>>>(P);
    mark_kernel_stop(st);
}

template <int DT>
static void launch_tree_chunk(const TreeParams& P, int sms, cudaStream_t st)
{
    constexpr auto K1 = tree_stream_kernel<DT>;
    mark_kernel_start(st);
    constexpr int ssm = TREE_GROUPS * STREAM_SMEM, nth = stream_threads<TREE_GROUPS>();
    K1<<<cta_grid<K1>(((long long)P.B * P.R * P.S1 + TREE_GROUPS - 1) / TREE_GROUPS, sms, ssm, nth), nth, ssm,
         st>>>(P);
    mark_kernel_stop(st);
    const size_t smem = P.N <= TREE_SMEM_NODES ? (size_t)(4 * P.N + P.R) * sizeof(int32_t) : 0;
    set_smem_limit<tree_finish_kernel<DT>>(smem);
    launch_dependent(tree_finish_kernel<DT>, (unsigned)P.B, NT, smem, st, P);
}

cudaError_t launch_tree_path(const TreeParams& P, int sms, cudaStream_t st)
{
    if (P.dtype == DT_BF16) {
        if (P.vec == 8) launch_tree_chunk<DT_BF16>(P, sms, st);
        else launch_tree_plain<DT_BF16, 1>(P, sms, st);
    } else {
        if (P.vec == 4) launch_tree_chunk<DT_F32>(P, sms, st);
        else launch_tree_plain<DT_F32, 1>(P, sms, st);
    }
    return cudaGetLastError();
}

}  // namespace sv
