// sv_smc.cu -- the group step of an SMC-SD verify round (Module 16 speculative-decoding lesson,
// "SMC Speculative Decoding: Resample, Don't Reject", "The Math: Reweight, Don't Reject", Algorithm 1
// step 5).  The particles' block log-ratios and extension tokens come from the plain round's kernels
// run without acceptance test; this kernel takes each group of Np particles (one CTA per group):
//   - ESS = (sum w)^2 / sum w^2 of the updated weights w = exp(logw - max);
//   - ESS < eta: particle n's ancestor is the inverse-CDF draw over the normalised weights, in
//     particle order, with its own uniform (i.i.d. draws), and every weight is reset to 1/Np;
//   - a group holding a particle whose status is not OK gets ESS NaN, resampled -1, ancestors -1 and
//     weights NaN.
#include "sv_smc.cuh"

namespace sv {

namespace {

__global__ void __launch_bounds__(SMC_NT) smc_group_kernel(const SmcGroupParams S)
{
    extern __shared__ float cw[];  // [Np] inclusive prefix of the weights, particle order
    __shared__ float red[2][SMC_NT / 32];
    __shared__ float carry;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Np = S.Np;
    const size_t b0 = (size_t)g * Np;
    pdl_wait();  // the plans and mid-round weights of the plain round

    int ok = 1;
    float m = NEG_INF;
    for (int n = tid; n < Np; n += SMC_NT) {
        ok &= (S.plan[b0 + n].status == ROW_OK);
        m = fmaxf(m, S.logw[b0 + n]);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        for (int n = tid; n < Np; n += SMC_NT) {
            S.logw[b0 + n] = __int_as_float(0x7fc00000);
            if (S.ancestors) S.ancestors[b0 + n] = -1;
        }
        if (tid == 0) {
            if (S.ess) S.ess[g] = __int_as_float(0x7fc00000);
            if (S.resampled) S.resampled[g] = -1;
        }
        return;
    }
    // the largest log weight, then sum w and sum w^2 (fixed order: lanes, then warps)
    m = warp_max(m);
    if (lane == 0) red[0][warp] = m;
    __syncthreads();
    m = red[0][0];
#pragma unroll
    for (int w = 1; w < SMC_NT / 32; ++w) m = fmaxf(m, red[0][w]);
    __syncthreads();
    float s1 = 0.f, s2 = 0.f;
    for (int n = tid; n < Np; n += SMC_NT) {
        const float w = expf(S.logw[b0 + n] - m);
        s1 += w;
        s2 += w * w;
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if (lane == 0) {
        red[0][warp] = s1;
        red[1][warp] = s2;
    }
    __syncthreads();
    s1 = 0.f;
    s2 = 0.f;
#pragma unroll
    for (int w = 0; w < SMC_NT / 32; ++w) {
        s1 += red[0][w];
        s2 += red[1][w];
    }
    const float ess = s1 * s1 / s2;
    const bool rs = ess < S.eta;
    if (tid == 0) {
        if (S.ess) S.ess[g] = ess;
        if (S.resampled) S.resampled[g] = rs ? 1 : 0;
    }
    if (!rs) {
        if (S.ancestors)
            for (int n = tid; n < Np; n += SMC_NT) S.ancestors[b0 + n] = n;
        return;
    }
    // inclusive prefix of the weights in particle order, tile by tile
    if (tid == 0) carry = 0.f;
    __syncthreads();
    for (int base = 0; base < Np; base += SMC_NT) {
        const int n = base + tid;
        const float w = n < Np ? expf(S.logw[b0 + n] - m) : 0.f;
        const float inc = warp_incl_scan(w);
        if (lane == 31) red[0][warp] = inc;
        __syncthreads();
        float off = carry;
        for (int w2 = 0; w2 < warp; ++w2) off += red[0][w2];
        if (n < Np) cw[n] = off + inc;
        __syncthreads();
        if (tid == SMC_NT - 1) {
            float t = carry;
            for (int w2 = 0; w2 < SMC_NT / 32; ++w2) t += red[0][w2];
            carry = t;
        }
        __syncthreads();
    }
    const float total = cw[Np - 1];
    const float reset = -logf((float)Np);
    for (int n = tid; n < Np; n += SMC_NT) {
        // the smallest m with u * total < cw[m]; past the end by rounding: the last particle with
        // positive weight
        const float t = __ldg(S.uniforms + (b0 + n) * 2 + 1) * total;
        int lo = 0, hi = Np;  // first index with t < cw[index]
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (t < cw[mid]) hi = mid;
            else lo = mid + 1;
        }
        int a = lo;
        if (a >= Np) {
            a = Np - 1;
            while (a > 0 && !(cw[a] > cw[a - 1])) --a;
        }
        if (S.ancestors) S.ancestors[b0 + n] = a;
    }
    __syncthreads();  // every weight read before any is reset
    for (int n = tid; n < Np; n += SMC_NT) S.logw[b0 + n] = reset;
}

}  // namespace

cudaError_t launch_smc_groups(const SmcGroupParams& S, cudaStream_t st)
{
    const size_t smem = (size_t)S.Np * sizeof(float);
    set_smem_limit<smc_group_kernel>(smem);
    return launch_dependent(smc_group_kernel, (unsigned)S.G, SMC_NT, smem, st, S);
}

}  // namespace sv
