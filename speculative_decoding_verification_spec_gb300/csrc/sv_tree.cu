// sv_tree.cu -- Medusa-style greedy tree verify (Module 16 lesson, "Verify the Tree -- and Why It's
// Exact"; M7.7 section 0x07E for the predictor-row convention).
//
// One kernel.  Each CTA takes one (row, chunk of V) and finds the chunk's argmax (first index of
// the maximum) with packed bf16x2 maxima per 16-byte vector; the last CTA of a request merges the
// partials in chunk order (so ties keep the lowest index), walks the tree in node order (a node's
// parent always precedes it), picks the deepest valid node and writes the path and the bonus.
#include "sv_common.cuh"

namespace sv {

__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// (best, idx) ordering: larger value first, then the lower index
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

template <int DT, int VEC>
__device__ __forceinline__ void chunk_argmax(const char* row, long long v0, long long v1,
                                             float& best, int& bidx, int& nan)
{
    constexpr int U = (VEC == 1) ? 8 : 4;
    for (long long base = v0 + threadIdx.x; base < v1; base += (long long)NT * U) {
        float x[U][VEC];
        float bm;
        if constexpr (DT == DT_BF16 && VEC == 8) {
            uint4 w[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const long long v = base + (long long)j * NT;
                if (v < v1) w[j] = ld_stream_v4(row + v * 16);
                else w[j] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            }
            uint32_t pm = bmax2_nan(bmax2_nan(w[0].x, w[0].y), bmax2_nan(w[0].z, w[0].w));
#pragma unroll
            for (int j = 1; j < U; ++j)
                pm = bmax2_nan(pm, bmax2_nan(bmax2_nan(w[j].x, w[j].y), bmax2_nan(w[j].z, w[j].w)));
            bm = fmax_nan(bf16lo(pm), bf16hi(pm));
            if (bm > best) {
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    x[j][0] = bf16lo(w[j].x); x[j][1] = bf16hi(w[j].x);
                    x[j][2] = bf16lo(w[j].y); x[j][3] = bf16hi(w[j].y);
                    x[j][4] = bf16lo(w[j].z); x[j][5] = bf16hi(w[j].z);
                    x[j][6] = bf16lo(w[j].w); x[j][7] = bf16hi(w[j].w);
                }
            }
        } else {
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
            bm = NEG_INF;
#pragma unroll
            for (int j = 0; j < U; ++j)
#pragma unroll
                for (int e = 0; e < VEC; ++e) bm = fmax_nan(bm, x[j][e]);
        }
        if (bm != bm) {
            nan = 1;
        } else if (bm > best) {  // strictly greater: earlier indices win ties
            int found = -1;
#pragma unroll
            for (int j = 0; j < U; ++j)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (found < 0 && x[j][e] == bm) found = j * VEC + e;
            const int j = found / VEC, e = found % VEC;
            best = bm;
            bidx = (int)((base + (long long)j * NT) * VEC + e);
        }
    }
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT) tree_argmax_kernel(TreeParams P)
{
    __shared__ float sh_v[WARPS];
    __shared__ int sh_i[WARPS], sh_n[WARPS];
    __shared__ int sh_flag, sh_status, sh_A;

    const long long idx = blockIdx.x;
    const int chunk = (int)(idx % P.C);
    const long long rr = idx / P.C;
    const int b = (int)(rr / P.R), r = (int)(rr % P.R);
    const size_t es = (DT == DT_BF16) ? 2 : 4;
    const char* row = reinterpret_cast<const char*>(P.logits) + ((size_t)b * P.R + r) * (size_t)P.V * es;
    const long long v0 = (long long)chunk * P.cv;
    const long long v1 = min(v0 + P.cv, P.nvec);

    float best = NEG_INF;
    int bidx = 0x7fffffff, nan = 0;
    chunk_argmax<DT, VEC>(row, v0, v1, best, bidx, nan);

    // block reduction of (best, bidx), NaN flag
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (better(ov, oi, best, bidx)) { best = ov; bidx = oi; }
    }
    nan = __any_sync(0xffffffffu, nan);
    if (lane == 0) { sh_v[warp] = best; sh_i[warp] = bidx; sh_n[warp] = nan; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bv = sh_v[0];
        int bi = sh_i[0], bn = sh_n[0];
        for (int w = 1; w < WARPS; ++w) {
            if (better(sh_v[w], sh_i[w], bv, bi)) { bv = sh_v[w]; bi = sh_i[w]; }
            bn |= sh_n[w];
        }
        ArgmaxPartial pt;
        pt.best = bv;
        pt.idx = bi;
        pt.nan = bn;
        pt.pad = 0;
        P.partials[((size_t)b * P.R + r) * P.C + chunk] = pt;
    }
    if (!arrive_last(&P.req_ctr[b], (unsigned)(P.R * P.C), &sh_flag)) return;

    // ---- last CTA of the request: per-row argmax in chunk order
    if (threadIdx.x == 0) sh_status = ROW_OK;
    __syncthreads();
    int bad = 0;
    for (int j = threadIdx.x; j < P.R; j += NT) {
        const ArgmaxPartial* pp = P.partials + ((size_t)b * P.R + j) * P.C;
        float bv = NEG_INF;
        int bi = 0x7fffffff, bn = 0;
        for (int k = 0; k < P.C; ++k) {
            const float v = __ldcg(&pp[k].best);
            const int i = __ldcg(&pp[k].idx);
            bn |= __ldcg(&pp[k].nan);
            if (better(v, i, bv, bi)) { bv = v; bi = i; }
        }
        const bool ok = !bn && bi != 0x7fffffff;
        if (!ok) bad = 1;
        P.amax[(size_t)b * P.R + j] = ok ? bi : -1;
    }
    bad = __syncthreads_or(bad);

    // ---- walk (one thread; parents precede children)
    const int N = P.N, mo = P.max_out;
    int32_t* out = P.out_tokens + (size_t)b * mo;
    int32_t* onodes = P.out_nodes ? P.out_nodes + (size_t)b * (mo - 1) : nullptr;
    if (threadIdx.x == 0) {
        int st = bad ? ROW_NONFINITE : ROW_OK;
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
                const int t = tok[i];
                if (t < 0 || t >= P.V) badt = 1;
            }
            st = badp ? ROW_BAD_PARENT : (badt ? ROW_BAD_TOKEN : ROW_OK);
        }
        int bestn = -1, bestd = 0;
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
        sh_status = st;
        sh_A = bestd;
        P.accepted_len[b] = (st == ROW_OK) ? bestd : -1;
        if (P.row_status) P.row_status[b] = st;
        if (st == ROW_OK) {
            // path written back to front
            int n = bestd;
            out[n] = am[bestn < 0 ? 0 : bestn + 1];
            for (int i = bestn; i >= 0; i = par[i]) {
                --n;
                out[n] = tok[i];
                if (onodes) onodes[n] = i;
            }
        }
    }
    __syncthreads();
    const int st = sh_status;
    const int A = (st == ROW_OK) ? sh_A : -1;
    for (int i = threadIdx.x; i < mo; i += NT) {
        if (st != ROW_OK || i > A) out[i] = -1;
        if (onodes && i < mo - 1 && (st != ROW_OK || i >= A)) onodes[i] = -1;
    }
}

cudaError_t launch_tree_path(const TreeParams& P, unsigned grid, cudaStream_t st)
{
    if (P.dtype == DT_BF16) {
        if (P.vec == 8) tree_argmax_kernel<DT_BF16, 8><<<grid, NT, 0, st>>>(P);
        else tree_argmax_kernel<DT_BF16, 1><<<grid, NT, 0, st>>>(P);
    } else {
        if (P.vec == 4) tree_argmax_kernel<DT_F32, 4><<<grid, NT, 0, st>>>(P);
        else tree_argmax_kernel<DT_F32, 1><<<grid, NT, 0, st>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace sv
