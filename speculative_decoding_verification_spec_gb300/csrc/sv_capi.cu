// sv_capi.cu -- the C ABI (include/spec_verify.h): host-side validation, task geometry, workspace
// layout and kernel launches.  No allocation, no host synchronisation.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"
#include "sv_smc.cuh"
#include "sv_tree_sample.cuh"
#include "sv_typical.cuh"

namespace sv {

KernelEvents g_kernel_events;
// polls of a ring or segment wait before it gives up (spec_set_wait_limit); read at every call
static int g_wait_limit = MBAR_SPIN_LIMIT;
// tree_verify_sample's cluster size when forced (spec_set_tree_sample_cluster), else 0
static int g_ts_cluster = 0;

constexpr size_t ALIGN = 256;
static inline size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }
static inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// --------------------------------------------------------------------------- geometry

struct Shape {
    int vec;
    long long nvec;
};

static Shape row_shape(int V, int vec)
{
    Shape s;
    s.vec = vec;
    s.nvec = (vec == 1) ? V : V / vec;
    return s;
}

static long long slices1(const Shape& s) { return std::max(1LL, cdiv(s.nvec, TV1)); }
// 32 KB chunks of a row of 16-byte vectors (the streaming kernels)
static long long stream_chunks(const Shape& s) { return std::max(1LL, cdiv(s.nvec, (long long)NT * STREAM_NV)); }
// softmax partials per row: one per warp task (scalar path) or one per warp of each stream chunk
static long long partials_per_row(const Shape& s)
{
    return s.vec > 1 ? stream_chunks(s) * WARPS : slices1(s);
}
static long long slices2(const Shape& s) { return std::max(1LL, cdiv(s.nvec, TV2)); }
static long long nsegs(const Shape& s) { return std::max(1LL, cdiv(s.nvec, SEGV)); }

// L2 budget for the row pairs most likely to be corrected (read evict_last by the stats kernel)
constexpr double PIN_BYTES = 80e6;

// top-k chunks are 32 KB of one row: 16384 bf16 or 8192 fp32 elements
static long long topk_chunk_elems(int dtype) { return dtype == DT_BF16 ? 16384 : 8192; }
static int topk_chunks(int dtype, int V) { return (int)cdiv(V, topk_chunk_elems(dtype)); }
// Candidate lists of a row hold at most TK_UNION entries in all (the finish kernel keeps them in
// registers), one list per (segment, warp of the streaming kernel).  A row is split into up to 4
// segments (runs of chunks) so that the streaming kernel's ~2 CTAs per SM have at least a dozen
// segments each (load balance at small B), as far as every segment's lists can still hold a
// generous estimate of its candidates: 64 per chunk plus 2k + 64.
constexpr int TK_MAX_SEGR = 4;
constexpr int TK_UNION = 1024;
static int topk_segments(long long rows, int CT, int sms, int k)
{
    const long long want = cdiv(24LL * sms, std::max(1LL, rows));
    int ns = (int)std::max(1LL, std::min<long long>(want, std::min(TK_MAX_SEGR, CT)));
    while (ns > 1 && (long long)ns * (64 * cdiv(CT, ns) + 2 * std::min(k, NT) + 64) > TK_UNION) --ns;
    return (int)cdiv(CT, cdiv(CT, ns));
}
// per-chunk candidate slot: 2k + 64 entries
static int topk_slot_cap(int k) { return (int)((2LL * std::min(k, NT) + 64 + 31) / 32 * 32); }
// per-row kept list: the same, rounded up to a power of two (the on-chip sort pads to one)
static int topk_kept_cap(int k)
{
    int c = 1;
    while (c < topk_slot_cap(k)) c <<= 1;
    return c;
}

// --------------------------------------------------------------------------- workspace layout

struct SpecLayout {
    size_t ctr_bytes = 0, bytes = 0;
    size_t o_row_ctr = 0, o_req_ctr = 0, o_res_ctr = 0, o_dense_ctr = 0, o_ndense = 0, o_work = 0;
    size_t o_partials = 0, o_rstats = 0, o_plan = 0, o_segs = 0;
    size_t o_clist = 0, o_cdata = 0, o_ccount = 0, o_cbound = 0, o_klist = 0;
};

// Byte layout for `ppr` softmax partials per row, nseg residual segments per request and (top-k)
// (top-k) `nsegr` segment lists of `cap_s` candidates per row and kept lists of `cap_k` entries.
// All counters sit at the front so one memset clears them.
static SpecLayout spec_layout(int B, int R, long long ppr, long long nseg, bool topk, int nsegr,
                              int cap_s, int cap_k)

{
    SpecLayout L;
    size_t o = 0;
    L.o_row_ctr = o; o += (size_t)B * R * sizeof(unsigned);
    L.o_req_ctr = o; o += (size_t)B * sizeof(unsigned);
    L.o_res_ctr = o; o += (size_t)B * sizeof(unsigned);
    L.o_dense_ctr = o; o += (size_t)B * sizeof(unsigned);
    L.o_ndense = o; o += (size_t)B * sizeof(int);
    L.o_work = o; o += 2 * sizeof(unsigned);
    L.ctr_bytes = o;
    o = align_up(o);
    L.o_partials = o; o = align_up(o + (size_t)B * R * ppr * sizeof(Partial));
    L.o_rstats = o; o = align_up(o + (size_t)B * R * sizeof(RowStats));
    L.o_plan = o; o = align_up(o + (size_t)B * sizeof(Plan));
    L.o_segs = o; o = align_up(o + (size_t)B * nseg * sizeof(float));
    if (topk) {
        L.o_clist = o; o = align_up(o + (size_t)B * R * nsegr * cap_s * sizeof(TopkEntry));
        L.o_cdata = o; o = align_up(o + (size_t)B * R * nsegr * cap_s * sizeof(uint4));
        L.o_ccount = o; o = align_up(o + (size_t)B * R * nsegr * sizeof(int));
        L.o_cbound = o; o = align_up(o + (size_t)B * R * nsegr * sizeof(float));
        L.o_klist = o; o = align_up(o + (size_t)B * R * cap_k * sizeof(TopkEntry));
    }
    L.bytes = o;
    return L;
}

struct TreeLayout {
    size_t ctr_bytes = 0, bytes = 0;
    size_t o_req_ctr = 0, o_work = 0, o_partials = 0, o_amax = 0, o_scratch = 0;
};

static TreeLayout tree_layout(int B, int N, long long S1)
{
    TreeLayout L;
    const int R = N + 1;
    size_t o = 0;
    L.o_req_ctr = o; o += (size_t)B * sizeof(unsigned);
    L.o_work = o; o += sizeof(unsigned);
    L.ctr_bytes = o;
    o = align_up(o);
    L.o_partials = o; o = align_up(o + (size_t)B * R * S1 * sizeof(ArgmaxPartial));
    L.o_amax = o; o = align_up(o + (size_t)B * R * sizeof(int32_t));
    L.o_scratch = o; o = align_up(o + (size_t)B * (N > 0 ? N : 1) * 2 * sizeof(int32_t));
    L.bytes = o;
    return L;
}

// --------------------------------------------------------------------------- device queries

static int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int pick_vec(int dtype, int V, const void* a, const void* b)
{
    const size_t es = dtype == DT_BF16 ? 2 : 4;
    const int vec = dtype == DT_BF16 ? 8 : 4;
    if (((size_t)V * es) % 16 != 0) return 1;
    if (!aligned(a, 16)) return 1;
    if (b && !aligned(b, 16)) return 1;
    return vec;
}

// --------------------------------------------------------------------------- the calls

// the SMC-SD group step of smc_verify (null for the speculative-sampling calls)
struct SmcArgs {
    const float* logw_in;
    float* logw_out;
    float* log_ratio;
    int groups, particles;
    float eta;
    float* ess;
    int32_t* resampled;
    int32_t* ancestors;
};

static spec_status spec_common(const void* target, const void* draft, spec_dtype dtype,
                               const int32_t* tokens, const float* uniforms, int B, int gamma,
                               int V, float temperature, int top_k, int32_t* accepted_len,
                               int32_t* out_tokens, int32_t* row_status, float* aux_lse_p,
                               float* aux_lse_q, float* aux_accept, void* workspace,
                               size_t workspace_bytes, void* stream, const SmcArgs* smc = nullptr,
                               const uint32_t* allowed = nullptr, float top_p = 1.0f)
{
    if (B < 0 || gamma < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
    const double T = (double)temperature;
    const float c = (float)(1.4426950408889634 / T);
    if (!std::isfinite(c) || !(c > 0.0f)) return SPEC_ERR_INVALID_ARG;
    if (top_k < 0 || top_k > V) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    const int R = 2 * gamma + 1;
    if ((long long)B * R > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
    const size_t es = dtype == SPEC_BF16 ? 2 : 4;
    if (!target || !aligned(target, es)) return SPEC_ERR_INVALID_ARG;
    if (gamma > 0 && (!draft || !aligned(draft, es) || !tokens || !aligned(tokens, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
    if (!accepted_len || !out_tokens || !aligned(accepted_len, 4) || !aligned(out_tokens, 4))
        return SPEC_ERR_INVALID_ARG;
    if ((row_status && !aligned(row_status, 4)) || (aux_lse_p && !aligned(aux_lse_p, 4)) ||
        (aux_lse_q && !aligned(aux_lse_q, 4)) || (aux_accept && !aligned(aux_accept, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return SPEC_ERR_WORKSPACE;
    if (allowed && (!aligned(allowed, 4) || top_k != 0 || smc)) return SPEC_ERR_INVALID_ARG;
    if (!(top_p > 0.0f) || std::isnan(top_p)) return SPEC_ERR_INVALID_ARG;
    const bool topp = top_p < 1.0f;
    if (topp && (top_k != 0 || allowed || smc)) return SPEC_ERR_INVALID_ARG;

    const bool topk = top_k > 0 && top_k < V;
    const int dt = (dtype == SPEC_BF16) ? DT_BF16 : DT_F32;
    const int vec = pick_vec(dt, V, target, gamma > 0 ? draft : nullptr);
    const Shape sh = row_shape(V, vec);
    const int sms = sm_count();

    SpecParams P;
    std::memset(&P, 0, sizeof P);
    P.target = target;
    P.draft = draft;
    P.tokens = tokens;
    P.uniforms = uniforms;
    P.B = B; P.gamma = gamma; P.V = V; P.R = R;
    P.dtype = dt; P.vec = vec; P.nvec = sh.nvec;
    P.c = c; P.T = T; P.invT = 1.0 / T; P.top_k = top_k;
    P.wait_limit = g_wait_limit;
    P.invT_hi = (float)P.invT;
    P.invT_lo = (float)(P.invT - (double)P.invT_hi);
    // 16-byte vectors: 32 KB stream chunks (statistics) and 2048-vector residual chunks; the
    // scalar path's persistent warps take TV1 / TV2 vectors per task
    P.S1 = (int)(vec > 1 ? stream_chunks(sh) : slices1(sh));
    P.S2 = (int)(vec > 1 ? std::max(1LL, cdiv(sh.nvec, NT * RCV)) : slices2(sh));
    P.nseg = (int)nsegs(sh);
    P.tasks1 = (long long)B * R * P.S1;
    P.tasks2 = (long long)B * P.S2;
    P.pin_pairs = (int)std::min(2.0, std::floor(PIN_BYTES / ((double)B * 2.0 * (double)V * (double)es)));
    if (topk) {
        P.CT = topk_chunks(dt, V);
        P.nsegr = topk_segments((long long)B * R, P.CT, sms, top_k);
        P.sps = (int)cdiv(P.CT, P.nsegr);
        P.cap_s = TK_UNION / P.nsegr;
        P.cap_k = topk_kept_cap(top_k);
    }
    const SpecLayout L = spec_layout(B, R, partials_per_row(sh), P.nseg, topk, P.nsegr, P.cap_s, P.cap_k);
    if (workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
    if ((long long)B * R * (topk ? P.CT : 1) >= (1LL << 31) || P.tasks1 >= (1LL << 31) ||
        (long long)B * R * P.S1 >= (1LL << 31) ||
        (long long)B * R * TK_MAX_SEGR * WARPS >= (1LL << 31))
        return SPEC_ERR_INVALID_ARG;

    char* ws = static_cast<char*>(workspace);
    P.accepted_len = accepted_len;
    P.out_tokens = out_tokens;
    P.row_status = row_status;
    P.aux_lse_p = aux_lse_p;
    P.aux_lse_q = aux_lse_q;
    P.aux_accept = aux_accept;
    P.mask = allowed;
    P.mwords = (int)cdiv(V, 32);
    P.top_p = topp ? top_p : 1.0f;
    if (smc) {
        P.smc = 1;
        P.smc_logw_in = smc->logw_in;
        P.smc_log_ratio = smc->log_ratio;
        P.smc_logw = smc->logw_out;
    }
    P.row_ctr = reinterpret_cast<unsigned*>(ws + L.o_row_ctr);
    P.req_ctr = reinterpret_cast<unsigned*>(ws + L.o_req_ctr);
    P.res_ctr = reinterpret_cast<unsigned*>(ws + L.o_res_ctr);
    P.dense_ctr = reinterpret_cast<unsigned*>(ws + L.o_dense_ctr);
    P.ndense = reinterpret_cast<int*>(ws + L.o_ndense);
    P.work = reinterpret_cast<unsigned*>(ws + L.o_work);
    P.partials = reinterpret_cast<Partial*>(ws + L.o_partials);
    P.rstats = reinterpret_cast<RowStats*>(ws + L.o_rstats);
    P.plan = reinterpret_cast<Plan*>(ws + L.o_plan);
    P.segs = reinterpret_cast<float*>(ws + L.o_segs);
    if (topk) {
        P.clist = reinterpret_cast<TopkEntry*>(ws + L.o_clist);
        P.cdata = reinterpret_cast<uint4*>(ws + L.o_cdata);
        P.ccount = reinterpret_cast<int*>(ws + L.o_ccount);
        P.cbound = reinterpret_cast<float*>(ws + L.o_cbound);
        P.klist = reinterpret_cast<TopkEntry*>(ws + L.o_klist);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // streaming paths (16-byte vectors) clear the counters in their first kernel; the scalar
    // paths' persistent kernels claim work from counters, so those are cleared beforehand
    if (vec > 1) {
        P.ctr_clear = reinterpret_cast<unsigned*>(ws);
        P.ctr_words = (int)(L.ctr_bytes / sizeof(unsigned));
    } else if (cudaMemsetAsync(ws, 0, L.ctr_bytes, st) != cudaSuccess) {
        return SPEC_ERR_CUDA;
    }
    cudaError_t err;
    if (topp) {
        err = launch_topp_path(P, sms, st);
    } else if (!topk) {
        err = launch_softmax_path(P, sms, st);
    } else {
        err = launch_topk_path(P, sms, st);
    }
    if (err == cudaSuccess && smc) {
        SmcGroupParams S;
        S.plan = P.plan;
        S.uniforms = uniforms;
        S.logw = smc->logw_out;
        S.G = smc->groups;
        S.Np = smc->particles;
        S.eta = smc->eta;
        S.ess = smc->ess;
        S.resampled = smc->resampled;
        S.ancestors = smc->ancestors;
        err = launch_smc_groups(S, st);
    }
    return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_workspace_bytes(int B, int gamma, int V, int top_k, int tree_nodes)
{
    if (B < 0 || gamma < 0 || V < 1 || top_k < 0 || tree_nodes < 0) return 0;
    size_t best = ALIGN;
    for (int vec : {1, 4, 8}) {
        const Shape sh = row_shape(V, vec);
        if (tree_nodes > 0) {
            best = std::max(best, tree_layout(B, tree_nodes, sh.vec > 1 ? stream_chunks(sh) * WARPS
                                                                           : slices1(sh)).bytes);
        } else {
            const bool topk = top_k > 0 && top_k < V;
            // lists: nsegr * cap_s = TK_UNION groups per row, at most TK_MAX_SEGR lists
            const SpecLayout L = spec_layout(B, 2 * gamma + 1, partials_per_row(sh), nsegs(sh), topk,
                                             TK_MAX_SEGR, topk ? TK_UNION / TK_MAX_SEGR : 0,
                                             topk ? topk_kept_cap(top_k) : 0);
            best = std::max(best, L.bytes);
        }
    }
    return best;
}

spec_status spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                        const int32_t* draft_tokens, const float* uniforms, int B, int gamma, int V,
                        float temperature, int32_t* accepted_len, int32_t* out_tokens,
                        int32_t* row_status, float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                        void* workspace, size_t workspace_bytes, void* stream)
{
    return spec_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma, V,
                       temperature, 0, accepted_len, out_tokens, row_status, aux_lse_p, aux_lse_q,
                       aux_accept, workspace, workspace_bytes, stream);
}

spec_status spec_verify_topk(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* draft_tokens, const float* uniforms, int B, int gamma,
                             int V, float temperature, int top_k, int32_t* accepted_len,
                             int32_t* out_tokens, int32_t* row_status, float* aux_lse_p,
                             float* aux_lse_q, float* aux_accept, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    if (top_k < 1 || top_k > V) return SPEC_ERR_INVALID_ARG;
    return spec_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma, V,
                       temperature, top_k, accepted_len, out_tokens, row_status, aux_lse_p,
                       aux_lse_q, aux_accept, workspace, workspace_bytes, stream);
}

spec_status spec_verify_topp(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* draft_tokens, const float* uniforms, int B, int gamma,
                             int V, float temperature, float top_p, int32_t* accepted_len,
                             int32_t* out_tokens, int32_t* row_status, float* aux_lse_p,
                             float* aux_lse_q, float* aux_accept, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    if (!(top_p > 0.0f) || std::isnan(top_p)) return SPEC_ERR_INVALID_ARG;
    if ((long long)B * (2 * (long long)gamma + 1) >= (1LL << 31)) return SPEC_ERR_INVALID_ARG;
    return spec_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma, V,
                       temperature, 0, accepted_len, out_tokens, row_status, aux_lse_p, aux_lse_q,
                       aux_accept, workspace, workspace_bytes, stream, nullptr, nullptr, top_p);
}

spec_status spec_verify_masked(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const float* uniforms,
                               const uint32_t* allowed, int B, int gamma, int V, float temperature,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                               float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                               void* workspace, size_t workspace_bytes, void* stream)
{
    if (B > 0 && !allowed) return SPEC_ERR_INVALID_ARG;
    return spec_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma, V,
                       temperature, 0, accepted_len, out_tokens, row_status, aux_lse_p, aux_lse_q,
                       aux_accept, workspace, workspace_bytes, stream, nullptr, allowed);
}

spec_status smc_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                       const int32_t* draft_tokens, const float* log_weights_in,
                       const float* uniforms, int groups, int particles, int K, int V,
                       float temperature, float ess_threshold, int32_t* accepted_len,
                       int32_t* out_tokens, float* log_weights_out, float* block_log_ratio,
                       float* ess, int32_t* resampled, int32_t* ancestors, int32_t* row_status,
                       void* workspace, size_t workspace_bytes, void* stream)
{
    if (groups < 0 || particles < 1 || particles > SMC_MAX_PARTICLES) return SPEC_ERR_INVALID_ARG;
    if ((long long)groups * particles > 0x7fffffffLL) return SPEC_ERR_INVALID_ARG;
    if (!std::isfinite(ess_threshold)) return SPEC_ERR_INVALID_ARG;
    if (groups > 0 && (!log_weights_in || !aligned(log_weights_in, 4) || !log_weights_out ||
                       !aligned(log_weights_out, 4)))
        return SPEC_ERR_INVALID_ARG;
    if ((block_log_ratio && !aligned(block_log_ratio, 4)) || (ess && !aligned(ess, 4)) ||
        (resampled && !aligned(resampled, 4)) || (ancestors && !aligned(ancestors, 4)))
        return SPEC_ERR_INVALID_ARG;
    SmcArgs a;
    a.logw_in = log_weights_in;
    a.logw_out = log_weights_out;
    a.log_ratio = block_log_ratio;
    a.groups = groups;
    a.particles = particles;
    a.eta = ess_threshold;
    a.ess = ess;
    a.resampled = resampled;
    a.ancestors = ancestors;
    return spec_common(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                       groups * particles, K, V, temperature, 0, accepted_len, out_tokens,
                       row_status, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream, &a);
}

// greedy tree verify; chain: parents is ignored and node i's parent is i - 1 (spec_verify_greedy)
static spec_status tree_common(const void* logits, spec_dtype dtype, const int32_t* parents,
                               const int32_t* tokens, int B, int N, int V, int max_out,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                               int32_t* row_status, void* workspace, size_t workspace_bytes,
                               void* stream, bool chain)
{
    if (B < 0 || N < 0 || V < 1 || max_out < 1) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    const int R = N + 1;
    if ((long long)B * R > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
    const size_t es = dtype == SPEC_BF16 ? 2 : 4;
    if (!logits || !aligned(logits, es)) return SPEC_ERR_INVALID_ARG;
    if (chain) parents = nullptr;
    if (N > 0 && ((!chain && (!parents || !aligned(parents, 4))) || !tokens || !aligned(tokens, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!accepted_len || !out_tokens || !aligned(accepted_len, 4) || !aligned(out_tokens, 4))
        return SPEC_ERR_INVALID_ARG;
    if ((out_nodes && !aligned(out_nodes, 4)) || (row_status && !aligned(row_status, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return SPEC_ERR_WORKSPACE;

    const int dt = (dtype == SPEC_BF16) ? DT_BF16 : DT_F32;
    const int vec = pick_vec(dt, V, logits, nullptr);
    const Shape sh = row_shape(V, vec);
    TreeParams P;
    std::memset(&P, 0, sizeof P);
    P.logits = logits;
    P.parents = parents;
    P.tokens = tokens;
    P.B = B; P.N = N; P.V = V; P.R = R;
    P.dtype = dt; P.vec = vec; P.nvec = sh.nvec;
    // 16-byte vectors: 32 KB stream chunks (a partial per chunk and warp); scalar path: slices
    P.S1 = (int)(vec > 1 ? stream_chunks(sh) : slices1(sh));
    P.tasks = (long long)B * R * P.S1;
    P.max_out = max_out;
    P.wait_limit = g_wait_limit;
    if (P.tasks >= (1LL << 31)) return SPEC_ERR_INVALID_ARG;
    const TreeLayout L = tree_layout(B, N, vec > 1 ? (long long)P.S1 * WARPS : P.S1);
    if (workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    P.accepted_len = accepted_len;
    P.out_tokens = out_tokens;
    P.out_nodes = (max_out > 1) ? out_nodes : nullptr;
    P.row_status = row_status;
    P.req_ctr = reinterpret_cast<unsigned*>(ws + L.o_req_ctr);
    P.work = reinterpret_cast<unsigned*>(ws + L.o_work);
    P.partials = reinterpret_cast<ArgmaxPartial*>(ws + L.o_partials);
    P.amax = reinterpret_cast<int32_t*>(ws + L.o_amax);
    P.scratch = reinterpret_cast<int32_t*>(ws + L.o_scratch);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the streaming path (16-byte vectors) uses no counters; the scalar path claims work from them
    if (vec == 1 && cudaMemsetAsync(ws, 0, L.ctr_bytes, st) != cudaSuccess) return SPEC_ERR_CUDA;
    const cudaError_t err = launch_tree_path(P, sm_count(), st);
    return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status tree_verify_greedy(const void* logits, spec_dtype dtype, const int32_t* parents,
                               const int32_t* tokens, int B, int N, int V, int max_out,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                               int32_t* row_status, void* workspace, size_t workspace_bytes,
                               void* stream)
{
    return tree_common(logits, dtype, parents, tokens, B, N, V, max_out, accepted_len, out_tokens,
                       out_nodes, row_status, workspace, workspace_bytes, stream, false);
}

spec_status spec_verify_greedy(const void* target_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, int B, int gamma, int V,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                               void* workspace, size_t workspace_bytes, void* stream)
{
    if (gamma < 0) return SPEC_ERR_INVALID_ARG;
    return tree_common(target_logits, dtype, nullptr, draft_tokens, B, gamma, V, gamma + 1,
                       accepted_len, out_tokens, nullptr, row_status, workspace, workspace_bytes,
                       stream, true);
}

spec_status tree_verify_typical(const void* logits, spec_dtype dtype, const int32_t* parents,
                                const int32_t* tokens, const float* uniforms, int B, int N, int V,
                                float temperature, float epsilon, float delta, int max_out,
                                int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                                int32_t* row_status, float* aux_entropy, float* aux_logp,
                                void* workspace, size_t workspace_bytes, void* stream)
{
    if (B < 0 || N < 0 || N > TYP_MAX_NODES || V < 1 || max_out < 1) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
    const double T = (double)temperature;
    const float c = (float)(1.4426950408889634 / T);
    if (!std::isfinite(c) || !(c > 0.0f)) return SPEC_ERR_INVALID_ARG;
    if (!(epsilon >= 0.f) || !std::isfinite(epsilon) || !(delta >= 0.f) || !std::isfinite(delta))
        return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    const int R = N + 1;
    if ((long long)B * R > (1LL << 30)) return SPEC_ERR_INVALID_ARG;
    const size_t es = dtype == SPEC_BF16 ? 2 : 4;
    if (!logits || !aligned(logits, es)) return SPEC_ERR_INVALID_ARG;
    if (N > 0 && (!parents || !aligned(parents, 4) || !tokens || !aligned(tokens, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
    if (!accepted_len || !out_tokens || !aligned(accepted_len, 4) || !aligned(out_tokens, 4))
        return SPEC_ERR_INVALID_ARG;
    if ((out_nodes && !aligned(out_nodes, 4)) || (row_status && !aligned(row_status, 4)) ||
        (aux_entropy && !aligned(aux_entropy, 4)) || (aux_logp && !aligned(aux_logp, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return SPEC_ERR_WORKSPACE;

    const int dt = (dtype == SPEC_BF16) ? DT_BF16 : DT_F32;
    const int vec = pick_vec(dt, V, logits, nullptr);
    const Shape sh = row_shape(V, vec);
    TypicalParams P;
    std::memset(&P, 0, sizeof P);
    P.t.logits = logits;
    P.t.parents = parents;
    P.t.tokens = tokens;
    P.t.B = B; P.t.N = N; P.t.V = V; P.t.R = R;
    P.t.dtype = dt; P.t.vec = vec; P.t.nvec = sh.nvec;
    P.t.max_out = max_out;
    P.t.wait_limit = g_wait_limit;
    P.t.accepted_len = accepted_len;
    P.t.out_tokens = out_tokens;
    P.t.out_nodes = (max_out > 1) ? out_nodes : nullptr;
    P.t.row_status = row_status;
    P.uniforms = uniforms;
    P.c = c;
    P.ln_eps = epsilon > 0.f ? (float)std::log((double)epsilon) : -INFINITY;
    P.ln_delta = delta > 0.f ? (float)std::log((double)delta) : -INFINITY;
    P.aux_entropy = aux_entropy;
    P.aux_logp = aux_logp;
    // 16-byte vectors: 32 KB stream chunks, a partial per chunk and warp; scalar path: slices of
    // TYP_SLICE elements (as many as slices1, so the tree workspace size holds them)
    P.S1 = (int)(vec > 1 ? stream_chunks(sh) : cdiv(V, TYP_SLICE));
    P.np = vec > 1 ? P.S1 * WARPS : P.S1;
    P.nseg = (int)cdiv(sh.nvec, 32);
    if (P.nseg > TYP_MAX_SEGS) return SPEC_ERR_INVALID_ARG;
    if ((long long)B * R * P.S1 >= (1LL << 31)) return SPEC_ERR_INVALID_ARG;
    const TreeLayout L = tree_layout(B, N, P.np);
    if (workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
    P.partials = reinterpret_cast<TypPartial*>(static_cast<char*>(workspace) + L.o_partials);
    const cudaError_t err = launch_typical_path(P, sm_count(), static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status tree_verify_sample(const void* target_logits, const void* draft_logits,
                               spec_dtype dtype, const int32_t* parents, const int32_t* tokens,
                               const int32_t* qrow, const float* uniforms, int B, int N, int Nq,
                               int V, float temperature, int max_out, int32_t* accepted_len,
                               int32_t* out_tokens, int32_t* out_nodes, int32_t* row_status,
                               float* aux_accept, void* stream)
{
    if (B < 0 || N < 0 || Nq < 0 || V < 1 || max_out < 1) return SPEC_ERR_INVALID_ARG;
    if (N > TS_MAX_NODES) return SPEC_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    const size_t es = dtype == SPEC_BF16 ? 2 : 4;
    if (!target_logits || !aligned(target_logits, es)) return SPEC_ERR_INVALID_ARG;
    if (N > 0) {
        if (Nq < 1 || !draft_logits || !aligned(draft_logits, es)) return SPEC_ERR_INVALID_ARG;
        if (!parents || !tokens || !qrow || !aligned(parents, 4) || !aligned(tokens, 4) ||
            !aligned(qrow, 4))
            return SPEC_ERR_INVALID_ARG;
    }
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_INVALID_ARG;
    if (!accepted_len || !out_tokens || !aligned(accepted_len, 4) || !aligned(out_tokens, 4))
        return SPEC_ERR_INVALID_ARG;
    if ((out_nodes && !aligned(out_nodes, 4)) || (row_status && !aligned(row_status, 4)) ||
        (aux_accept && !aligned(aux_accept, 4)))
        return SPEC_ERR_INVALID_ARG;

    const int dt = (dtype == SPEC_BF16) ? DT_BF16 : DT_F32;
    const int EPV = dt == DT_BF16 ? 8 : 4;
    const long long nvec = cdiv(V, EPV);
    // the smallest cluster whose slices fit TS_VPT vectors per thread ...
    int CL = 1;
    while (CL <= TS_MAX_CLUSTER && cdiv(nvec, (long long)CL * TS_NT) > TS_VPT) CL *= 2;
    if (CL > TS_MAX_CLUSTER) return SPEC_ERR_INVALID_ARG;  // V above the cluster's capacity
    if (g_ts_cluster > 0) {  // a forced size (measurement aid), if its slices hold the row
        if (cdiv(nvec, (long long)g_ts_cluster * TS_NT) > TS_VPT) return SPEC_ERR_INVALID_ARG;
        CL = g_ts_cluster;
    } else {
        // ... widened, up to the portable 8, while the doubled cluster still leaves every CTA an
        // SM of its own and each thread at least one vector (a wider cluster shares a row among
        // more SMs, but every exchange between them then costs more)
        const int sms = sm_count();
        while (CL < 8 && 2LL * B * CL <= sms && nvec >= 2LL * CL * TS_NT) CL *= 2;
    }
    if ((long long)B * CL > 0x7fffffffLL) return SPEC_ERR_INVALID_ARG;

    TreeSampleParams P;
    std::memset(&P, 0, sizeof P);
    P.target = target_logits;
    P.draft = draft_logits;
    P.parents = parents;
    P.tokens = tokens;
    P.qrow = qrow;
    P.uniforms = uniforms;
    P.B = B; P.N = N; P.Nq = Nq; P.V = V; P.max_out = max_out;
    P.dtype = dt;
    P.invT = 1.0f / temperature;
    P.nvec = nvec;
    P.vpt = (int)cdiv(nvec, (long long)CL * TS_NT);
    P.accepted_len = accepted_len;
    P.out_tokens = out_tokens;
    P.out_nodes = (max_out > 1) ? out_nodes : nullptr;
    P.row_status = row_status;
    P.aux_accept = aux_accept;
    // 16-byte loads when every row starts on a 16-byte boundary
    const bool vec16 = ((size_t)V * es) % 16 == 0 && aligned(target_logits, 16) &&
                       (N == 0 || aligned(draft_logits, 16));
    const cudaError_t err = launch_tree_sample(P, CL, vec16, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

void spec_set_kernel_events(void* start, void* stop)
{
    g_kernel_events.start = static_cast<cudaEvent_t>(start);
    g_kernel_events.stop = static_cast<cudaEvent_t>(stop);
}

int spec_set_tree_sample_cluster(int cl)
{
    const int prev = g_ts_cluster;
    g_ts_cluster = (cl == 1 || cl == 2 || cl == 4 || cl == 8 || cl == 16) ? cl : 0;
    return prev;
}

int spec_set_wait_limit(int polls)
{
    const int prev = g_wait_limit;
    g_wait_limit = polls < 0 ? MBAR_SPIN_LIMIT : std::min(polls, MBAR_SPIN_LIMIT);
    return prev;
}

const char* spec_status_string(spec_status s)
{
    switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_CUDA: return "CUDA launch error";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_TOO_LARGE: return "sizes need more scratch than the no-allocation entry point holds";
    }
    return "unknown status";
}

}  // extern "C"
