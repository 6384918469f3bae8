// sv_smc.cuh -- the group step of an SMC-SD verify round (sv_smc.cu): effective sample size of each
// group's updated weights and, below the threshold, the particles' ancestors.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int SMC_NT = 256;                 // threads per group CTA
constexpr int SMC_MAX_PARTICLES = 4096;     // a group's weight prefix is kept in shared memory

struct SmcGroupParams {
    const Plan* plan;       // [B] the plain round's plans (status of each particle)
    const float* uniforms;  // [B, 2] slot 1: the particle's ancestor draw
    float* logw;            // [B] in: logw_in + block log-ratio; out: reset to -log(Np) if resampled
    int G, Np;
    float eta;
    float* ess;             // [G] or null
    int32_t* resampled;     // [G] or null: 1, 0, or -1 when a particle of the group failed
    int32_t* ancestors;     // [B] or null: index of the ancestor within the group
};

// one CTA per group, launched as a dependent grid after the plain round's kernels
cudaError_t launch_smc_groups(const SmcGroupParams& S, cudaStream_t st);

}  // namespace sv
