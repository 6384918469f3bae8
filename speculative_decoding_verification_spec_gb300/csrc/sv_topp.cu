// sv_topp.cu -- exact speculative sampling with a top-p (nucleus) processor on p and q.
//
// "Exact speculative and assisted decoding for TinyRustLM": top-p is one of the declared processors
// that both distributions pass through before the ratio is formed; M7.1 section 0x03D: truncation
// keeps the round exact when q is the truncated distribution that sampled the draft.  A row keeps
// the tokens of largest probability, whole groups of equal stored logit at a time, until the kept
// mass (after temperature) first reaches top_p: the kept set is {v : x_v >= g}, and p is
// renormalised over it.
//
// Kernel 1: the plain path's row statistics (M, MC, S per chunk and warp).
// Kernel 2 (topp_row_kernel), one CTA per row: the row's M, MC and full mass, then g by a
// mass-weighted radix select over the order-preserving key of the stored logits (16-bit for bf16,
// 32-bit for fp32), four bits per pass over the row.  Each pass adds the fixed-point mass
// 2^40 * 2^y (rounded toward zero), y = x c - MC, of every element whose key matches the digits
// chosen so far to the thread's own bin of its next digit (integer sums: exact and order-free, so
// g does not depend on scheduling); the digit is where the mass above it first reaches
// top_p * (total).  The kept mass is the select's own sum above g.  The row's lse, 1/S and
// log2 p(x) of the token it scores are then formed as on the plain path; the last CTA of a request
// runs the acceptance scan.
// Kernel 3: the plain path's residual pass with each row's threshold applied.
#include "sv_plan.cuh"

namespace sv {

// Monotone key of a float (x < y iff key(x) < key(y)); -0 is folded into +0 first, since the two
// compare equal.
__device__ __forceinline__ uint32_t order_key(float x)
{
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// The fixed-point mass 2^40 w (rounded toward zero) of w in [0, 1], from the float's bits with
// integer operations only (a conversion to a 64-bit integer is not a fast-pipe instruction).
__device__ __forceinline__ unsigned long long fixed_mass(float w)
{
    const uint32_t u = __float_as_uint(w);
    const int e = (int)(u >> 23);  // biased exponent; w >= 0
    if (e == 0) return 0ull;       // zero (the exponential flushes subnormals)
    const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
    const int sh = e - 127 - 23 + 40;  // 2^40 w = m 2^sh, sh <= 17
    return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT) topp_row_kernel(SpecParams P)
{
    constexpr int KB = (DT == DT_BF16) ? 16 : 32;  // key bits that carry information
    __shared__ unsigned long long hist[16 * NT];   // digit-major, one column per thread (32 KB)
    __shared__ unsigned long long tot[16];
    __shared__ float sh_M;
    __shared__ DFloat sh_S;
    __shared__ int sh_st;
    __shared__ uint32_t sh_prefix;
    __shared__ unsigned long long sh_above, sh_kept;
    __shared__ double sh_target;
    __shared__ int sh_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int row_id = blockIdx.x, b = row_id / P.R, r = row_id - b * P.R, g = P.gamma;
    const char* row = spec_row_ptr(P, b, r);

    // the token this row scores and its logit: inputs, read before waiting for kernel 1
    const int pos = (r < g) ? r : (r > g) ? r - g - 1 : -1;
    const int tok = (pos >= 0) ? __ldg(P.tokens + (size_t)b * g + pos) : -1;
    const bool tok_ok = tok >= 0 && tok < P.V;
    const float xtok = tok_ok ? load_logit(row, DT, tok) : 0.f;
    pdl_wait();  // the partials of kernel 1

    // ---- the row's maximum and full mass (warp 0), as on the plain path
    if (warp == 0) {
        const int np = P.vec > 1 ? P.S1 * WARPS : P.S1;
        const Partial* pp = P.partials + (size_t)row_id * np;
        float Mr = NEG_INF;
        for (int k = lane; k < np; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
        Mr = warp_max(Mr);
        const float MCr = __fmul_rn(Mr, P.c);
        DFloat S = df_make(0.f, 0.f);
        int tmo = 0;
        for (int k = lane; k < np; k += 32) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(pp + k));
            if (q.z < 0.f) tmo = 1;
            if (q.z != 0.f) S = df_add(S, df_make(__fmul_rn(q.z, ex2(q.y - MCr)), 0.f));
        }
        S = warp_sum_df(S);
        tmo = __any_sync(FULL, tmo);
        if (lane == 0) {
            const bool ok = !tmo && isfinite(S.hi) && S.hi > 0.f && Mr != NEG_INF && isfinite(Mr);
            sh_M = Mr;
            sh_S = S;
            sh_st = tmo ? ROW_TIMEOUT : ok ? ROW_OK : ROW_NONFINITE;
            sh_prefix = 0;
            sh_above = 0;
        }
    }
    __syncthreads();
    const float M = sh_M, MC = __fmul_rn(M, P.c);
    float thr = NEG_INF;
    DFloat S = sh_S;

    // ---- the nucleus threshold: a radix select on the key, weighted by fixed-point mass
    if (sh_st == ROW_OK && P.top_p < 1.0f) {
        for (int lvl = 0; lvl < KB / 4; ++lvl) {
            const int shift = 32 - 4 * (lvl + 1);  // this level's digit of the 32-bit key
            const uint32_t prefix = sh_prefix;
#pragma unroll
            for (int d = 0; d < 16; ++d) hist[d * NT + tid] = 0ull;
            // consecutive elements of a thread mostly share a digit: their masses are added in a
            // register and reach the thread's bin when the digit changes
            unsigned long long run = 0ull;
            int cur = 0;
            for (long long v = tid; v < P.nvec; v += NT) {
                float x[VEC];
                load_vec<DT, VEC>(row, v, x);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const uint32_t key = order_key(x[e]);
                    if (lvl == 0 || (key >> (shift + 4)) == prefix) {
                        const int d = (int)((key >> shift) & 15u);
                        const unsigned long long fx = fixed_mass(ex2(fmaf(x[e], P.c, -MC)));
                        if (d != cur) {
                            hist[cur * NT + tid] += run;
                            cur = d;
                            run = fx;
                        } else {
                            run += fx;
                        }
                    }
                }
            }
            hist[cur * NT + tid] += run;
            __syncthreads();
            // digit totals: warp w adds the columns of digits 2w and 2w + 1
            for (int d = 2 * warp; d < 2 * warp + 2; ++d) {
                unsigned long long s = 0ull;
                for (int t = lane; t < NT; t += 32) s += hist[d * NT + t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
                if (lane == 0) tot[d] = s;
            }
            __syncthreads();
            if (tid == 0) {
                if (lvl == 0) {
                    unsigned long long all = 0ull;
                    for (int d = 0; d < 16; ++d) all += tot[d];
                    sh_target = (double)P.top_p * (double)all;
                }
                // the largest digit whose mass, with everything above it, reaches the target
                unsigned long long above = sh_above;
                int dsel = 0;
                for (int d = 15; d >= 0; --d) {
                    if ((double)(above + tot[d]) >= sh_target || d == 0) {
                        dsel = d;
                        break;
                    }
                    above += tot[d];
                }
                sh_above = above;
                sh_kept = above + tot[dsel];
                sh_prefix = (prefix << 4) | (uint32_t)dsel;
            }
            __syncthreads();
        }
        // the threshold's full key: for bf16 the low 16 bits of a key are all 0 (x >= 0) or all 1
        uint32_t gk = sh_prefix << (32 - KB);
        if (KB < 32 && !(gk & 0x80000000u)) gk |= (1u << (32 - KB)) - 1u;
        thr = key_float(gk);
        // the kept mass as a pair of floats (2^-40 units, exact in fp64 up to 2^53)
        const double kept = (double)sh_kept * (1.0 / 1099511627776.0);
        const float hi = (float)kept;
        S = df_make(hi, (float)(kept - (double)hi));
    }

    // ---- the row's statistics, as the plain path's row plan forms them
    if (tid == 0) {
        RowStats st = blank_rowstats();
        st.M = M;
        st.MC = MC;
        st.S = (double)S.hi;
        st.status = sh_st;
        st.lse = __int_as_float(0x7fc00000);
        st.lx_hi = __int_as_float(0x7fc00000);
        st.lx_lo = 0.f;
        if (sh_st == ROW_OK) {
            row_norm(st, M, MC, S, P, tok_ok, xtok, thr);
            st.thr = thr;
        }
        P.rstats[row_id] = st;
    }
    // ---- the last row of the request: the acceptance scan
    if (!arrive_last(&P.dense_ctr[b], (unsigned)P.R, &sh_flag)) return;
    if (warp == 0) {
        const Plan pl = compute_plan_warp<DT, true>(P, b, true);
        if (lane == 0) P.plan[b] = pl;
    }
}

cudaError_t launch_topp_path(const SpecParams& P, int sms, cudaStream_t st)
{
    cudaError_t e = launch_softmax_stats(P, sms, st);
    if (e != cudaSuccess) return e;
    const unsigned rows = (unsigned)((long long)P.B * P.R);
    if (P.dtype == DT_BF16)
        e = P.vec > 1 ? launch_dependent(topp_row_kernel<DT_BF16, 8>, rows, NT, 0, st, P)
                      : launch_dependent(topp_row_kernel<DT_BF16, 1>, rows, NT, 0, st, P);
    else
        e = P.vec > 1 ? launch_dependent(topp_row_kernel<DT_F32, 4>, rows, NT, 0, st, P)
                      : launch_dependent(topp_row_kernel<DT_F32, 1>, rows, NT, 0, st, P);
    if (e != cudaSuccess) return e;
    return launch_softmax_resample_thr(P, sms, st);
}

}  // namespace sv
