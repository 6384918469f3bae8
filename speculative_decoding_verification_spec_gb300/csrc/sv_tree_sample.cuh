// sv_tree_sample.cuh -- parameters and launch of the stochastic tree verify (sv_tree_sample.cu):
// one thread-block cluster of CL CTAs per request, each CTA one slice of the vocabulary.
#pragma once

#include "sv_common.cuh"

namespace sv {

enum { ROW_BAD_QROW = 8 };  // a node's proposal row index is outside [0, Nq)

constexpr int TS_NT = 512;               // threads per CTA
constexpr int TS_WARPS = TS_NT / 32;
constexpr int TS_VPT = 4;                // 16-byte vectors of a row per thread (registers)
constexpr int TS_MAX_CLUSTER = 16;
constexpr int TS_MAX_NODES = 4096;       // the tree description is kept in shared memory

struct TreeSampleParams {
    const void* target;       // [B, N+1, V]
    const void* draft;        // [B, Nq, V]
    const int32_t* parents;   // [B, N]
    const int32_t* tokens;    // [B, N]
    const int32_t* qrow;      // [B, N]
    const float* uniforms;    // [B, N+1]
    int B, N, Nq, V, max_out;
    int dtype;
    float invT;
    long long nvec;           // vectors of EPV elements per row (the last may be partial)
    int vpt;                  // vectors per thread: a CTA's slice is vpt * TS_NT vectors, a warp's
                              // a contiguous run of vpt * 32 of them
    int32_t* accepted_len;
    int32_t* out_tokens;
    int32_t* out_nodes;
    int32_t* row_status;
    float* aux_accept;        // [B, N] or null
};

// dynamic shared memory of one CTA, and the clustered launch (one kernel per call)
size_t tree_sample_smem(int vpt, int dtype, int N);
cudaError_t launch_tree_sample(const TreeSampleParams& P, int CL, bool vec16, cudaStream_t st);

}  // namespace sv
