// sv_typical.cuh -- tree verify with typical acceptance (sv_typical.cu): Medusa's sampling mode, in
// which a candidate passes when the target's probability clears min(eps, delta exp(-H)).
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int TYP_NT = 1024;          // threads of each CTA of the per-request finish cluster
constexpr int TYP_CL = 4;             // CTAs of the per-request finish cluster
constexpr int TYP_MAX_NODES = 2048;   // the tree is staged in shared memory
constexpr int TYP_MAX_SEGS = 16384;   // draw segments of one row (32 vectors each) in shared memory
constexpr int TYP_SLICE = 1024;       // elements per partial on the scalar path

struct __align__(16) TypPartial {  // one (row, chunk, warp) of the row statistics
    float M;   // maximum of the raw logits (-inf if none)
    float MC;  // fp32(M * c)
    float S;   // sum of 2^y, y = fma(x, c, -MC); < 0: the chunk was not read
    float E;   // sum of 2^y * y (the entropy's first moment)
};

struct TypicalParams {
    TreeParams t;           // logits, parents, tokens, sizes and outputs (t.partials unused)
    const float* uniforms;  // [B] the token after the path
    float c;                // log2(e) / T
    float ln_eps, ln_delta; // natural logs of eps and delta (-inf for 0)
    float* aux_entropy;     // [B, N+1] or null: natural-log entropy of each row after temperature
    float* aux_logp;        // [B, N] or null: ln p_r(token) of each node under its predictor row
    TypPartial* partials;   // [B*R*np]
    int np;                 // partials per row
    int S1;                 // stream chunks per row (16-byte vectors) or slices (scalar path)
    int nseg;               // draw segments per row: ceil(nvec / 32)
};

// row statistics (streaming or scalar kernel) then one finish CTA per request (dependent launch)
cudaError_t launch_typical_path(const TypicalParams& P, int sms, cudaStream_t st);
size_t typical_finish_smem(int N, int nseg);

}  // namespace sv
