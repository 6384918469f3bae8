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
#include "sv_common.cuh"

namespace sv {

__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

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
        const bool ok = !bn && bi != 0x7fffffff;
        if (!ok) bad = 1;
        P.amax[(size_t)b * P.R + j] = ok ? bi : -1;
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    // ---- walk (lane 0; parents precede children)
    const int N = P.N, mo = P.max_out;
    int32_t* out = P.out_tokens + (size_t)b * mo;
    int32_t* onodes = P.out_nodes ? P.out_nodes + (size_t)b * (mo - 1) : nullptr;
    int st = bad ? ROW_NONFINITE : ROW_OK, bestd = 0;
    if (lane == 0) {
        const int32_t* par = P.parents + (size_t)b * N;
        const int32_t* tok = P.tokens + (size_t)b * N;
        const int32_t* am = P.amax + (size_t)b * P.R;
        int32_t* depth = P.scratch + (size_t)b * N * 2;
        int32_t* valid = depth + N;
        if (st == ROW_OK) {
            int badp = 0, badt = 0;
            for (int i = 0; i < N; ++i) {
                const int p = par[i];
                if (p < -1 || p >= i) badp = 1;
                const int tk = tok[i];
                if (tk < 0 || tk >= P.V) badt = 1;
            }
            st = badp ? ROW_BAD_PARENT : (badt ? ROW_BAD_TOKEN : ROW_OK);
        }
        int bestn = -1;
        if (st == ROW_OK) {
            for (int i = 0; i < N; ++i) {
                const int p = par[i];
                const int predictor = p < 0 ? 0 : p + 1;
                const int vi = (tok[i] == am[predictor]) && (p < 0 || valid[p]);
                const int d = p < 0 ? 1 : depth[p] + 1;
                valid[i] = vi;
                depth[i] = d;
                if (vi && d > bestd) { bestd = d; bestn = i; }
            }
            if (bestd + 1 > mo) st = ROW_OVERFLOW;
        }
        P.accepted_len[b] = (st == ROW_OK) ? bestd : -1;
        if (P.row_status) P.row_status[b] = st;
        if (st == ROW_OK) {  // path written back to front, then the bonus
            int n = bestd;
            out[n] = am[bestn < 0 ? 0 : bestn + 1];
            for (int i = bestn; i >= 0; i = par[i]) {
                --n;
                out[n] = tok[i];
                if (onodes) onodes[n] = i;
            }
        }
    }
    st = __shfl_sync(0xffffffffu, st, 0);
    bestd = __shfl_sync(0xffffffffu, bestd, 0);
    const int A = (st == ROW_OK) ? bestd : -1;
    for (int i = lane; i < mo; i += 32) {
        if (st != ROW_OK || i > A) out[i] = -1;
        if (onodes && i < mo - 1 && (st != ROW_OK || i >= A)) onodes[i] = -1;
    }

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

// Chunk kernel for 16-byte vectors: one CTA per (request, row, chunk of CHUNK_VECS contiguous
// vectors), U1 vectors per thread loaded at a time into registers.  Each thread keeps its running
// maximum and the first vector where it was reached (strictly greater replaces, and a thread sees
// its vectors in index order); after the CTA maximum is known, the threads holding it re-read that
// one vector to locate the element, and the lowest such index is the chunk's argmax.
template <int DT>
__global__ void __launch_bounds__(NT) tree_argmax_chunk_kernel(TreeParams P)
{
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    __shared__ float sh_f[WARPS];
    __shared__ int sh_i[WARPS], sh_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x % P.S1;
    const int rr = blockIdx.x / P.S1;
    const int b = rr / P.R, r = rr % P.R;
    const char* row = tree_row(P, b, r);
    const int c0 = c * CHUNK_VECS;
    const int c1 = (int)min((long long)c0 + CHUNK_VECS, P.nvec);
    const uint64_t pol = policy_evict_first();
    float best = NEG_INF;
    int bvec = -1, nan = 0;
#pragma unroll
    for (int it = 0; it < CV / U1; ++it) {
        const int vb = c0 + it * U1 * NT + tid;
        if (vb >= c1) break;
        uint4 w[U1];
#pragma unroll
        for (int u = 0; u < U1; ++u) {
            const int v = vb + u * NT;
            const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;  // -inf
            w[u] = v < c1 ? ld_stream_v4_pol(row + (size_t)v * 16, pol) : make_uint4(pad, pad, pad, pad);
        }
#pragma unroll
        for (int u = 0; u < U1; ++u) {
            float vm;
            if constexpr (DT == DT_BF16) {
                const uint32_t pm = bmax2_nan(bmax2_nan(w[u].x, w[u].y), bmax2_nan(w[u].z, w[u].w));
                vm = fmax_nan(bf16lo(pm), bf16hi(pm));
            } else {
                vm = fmax_nan(fmax_nan(__uint_as_float(w[u].x), __uint_as_float(w[u].y)),
                              fmax_nan(__uint_as_float(w[u].z), __uint_as_float(w[u].w)));
            }
            if (vm != vm) nan = 1;
            else if (vm > best) { best = vm; bvec = vb + u * NT; }
        }
    }
    const float W = block_max(best, sh_f);
    const int anynan = __syncthreads_or(nan);
    int idx = 0x7fffffff;
    if (best == W && bvec >= 0) {  // re-read the vector where this thread first reached W
        RawVec<DT, VEC> x;
        x.load(row, bvec, pol);
#pragma unroll
        for (int e = VEC - 1; e >= 0; --e)
            if (x.get(e) == W) idx = bvec * VEC + e;
    }
    idx = __reduce_min_sync(0xffffffffu, idx);
    if (lane == 0) sh_i[warp] = idx;
    __syncthreads();
    if (tid == 0) {
        int bi = sh_i[0];
        for (int w = 1; w < WARPS; ++w) bi = min(bi, sh_i[w]);
        ArgmaxPartial pt;
        pt.best = W;
        pt.idx = bi;
        pt.nan = anynan;
        pt.pad = 0;
        P.partials[((size_t)b * P.R + r) * P.S1 + c] = pt;
    }
    if (!arrive_last(&P.req_ctr[b], (unsigned)(P.R * P.S1), &sh_flag)) return;
    if (warp == 0) tree_finish_request(P, b);
}

template <int DT, int VEC>
static void launch_tree_plain(const TreeParams& P, int sms, cudaStream_t st)
{
    mark_kernel_start(st);
    tree_argmax_kernel<DT, VEC><<<persistent_grid<tree_argmax_kernel<DT, VEC>>(P.tasks, sms), NT, 0, st>>>(P);
    mark_kernel_stop(st);
}

template <int DT>
static void launch_tree_chunk(const TreeParams& P, cudaStream_t st)
{
    mark_kernel_start(st);
    tree_argmax_chunk_kernel<DT><<<(unsigned)((long long)P.B * P.R * P.S1), NT, 0, st>>>(P);
    mark_kernel_stop(st);
}

cudaError_t launch_tree_path(const TreeParams& P, int sms, cudaStream_t st)
{
    if (P.dtype == DT_BF16) {
        if (P.vec == 8) launch_tree_chunk<DT_BF16>(P, st);
        else launch_tree_plain<DT_BF16, 1>(P, sms, st);
    } else {
        if (P.vec == 4) launch_tree_chunk<DT_F32>(P, st);
        else launch_tree_plain<DT_F32, 1>(P, sms, st);
    }
    return cudaGetLastError();
}

}  // namespace sv
