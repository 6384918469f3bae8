// sv_noalloc.cu -- spec_verify_noalloc: spec_verify with its scratch in a fixed device array, for
// callers that cannot allocate device memory (include/spec_verify.h says who and why).
//
// The array below is a file-scope __device__ object, so every GPU on which this library's code is
// loaded holds SPEC_NOALLOC_SCRATCH_BYTES for it until the process exits.  Host code sees only a
// host-side stand-in under its name; the device address comes from cudaGetSymbolAddress, looked
// up once per device with that device current and cached here.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/spec_verify.h"

namespace {

__device__ __align__(256) unsigned char noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* scratch_ptr[MAX_DEVICES] = {};
std::mutex scratch_mu;

// Device address of noalloc_scratch on the current device (nullptr if it cannot be had).
void* scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(scratch_mu);
    if (!scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, noalloc_scratch) != cudaSuccess || !p) return nullptr;
        scratch_ptr[dev] = p;
    }
    return scratch_ptr[dev];
}

}  // namespace

extern "C" spec_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                           spec_dtype dtype, const int32_t* draft_tokens,
                                           const float* uniforms, int B, int gamma, int V,
                                           float temperature, int32_t* accepted_len,
                                           int32_t* out_tokens, int32_t* row_status,
                                           float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                                           void* stream)
{
    const size_t need = spec_workspace_bytes(B, gamma, V, 0, 0);
    if (need == 0) return SPEC_ERR_INVALID_ARG;
    if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_TOO_LARGE;
    void* ws = scratch_on_current_device();
    if (!ws) return SPEC_ERR_CUDA;
    // spec_verify clears its completion counters on `stream` before its kernels run, so what the
    // previous call left in the array does not matter.
    return spec_verify(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma, V,
                       temperature, accepted_len, out_tokens, row_status, aux_lse_p, aux_lse_q,
                       aux_accept, ws, SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
