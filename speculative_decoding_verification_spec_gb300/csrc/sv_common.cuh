// sv_common.cuh -- shared device helpers, parameter blocks and workspace layout of the GB300
// speculative-decoding verify kernels.
//
// Arithmetic conventions used by every kernel:
//   * logits are read as fp32 (bf16 is widened exactly by a 16-bit shift);
//   * with c = log2(e)/T in fp32, a row's normaliser is kept as (MC, S) with MC = fp32(M * c),
//     M the row maximum, and S = sum_v 2^(fma(x_v, c, -MC)), so that p(v) = 2^(fma(x_v,c,-MC)) / S.
//     fma() rounds once after the exact product, so the exponent carries only a small error near
//     the row maximum, where probability mass sits; the rounding of MC shifts every exponent of a
//     row equally and cancels between numerator and S.
//   * per-thread and per-warp partial sums are fp32 (two at a time with the packed fp32
//     instructions where a loop carries pairs); sums across warps, chunks and segments are pairs of
//     floats (about 48 bits) or fp64 lane totals, and masses that decide a kept set are fixed-point
//     integers; every sum is taken in a fixed order or is exact, so results do not depend on CTA
//     scheduling.
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int NT = 256;           // threads per CTA, every kernel
constexpr int WARPS = NT / 32;
constexpr float NEG_INF = -__builtin_huge_valf();

enum { DT_F32 = 0, DT_BF16 = 1 };
enum {
    ROW_OK = 0,
    ROW_NONFINITE = 1,
    ROW_DEGENERATE = 2,
    ROW_BAD_TOKEN = 3,
    ROW_TIMEOUT = 4,
    ROW_BAD_PARENT = 5,
    ROW_OVERFLOW = 6,
    ROW_BAD_UNIFORM = 7
};

// ---------------------------------------------------------------- workspace records

struct __align__(16) Partial {  // one (row, chunk) of the softmax statistics
    float M;          // chunk maximum of the raw logits (-inf if none)
    float MC;         // fp32(M * c)
    float S;          // sum over the chunk of 2^(fma(x, c, -MC)); < 0: the chunk was not read
    float pad;
};

struct RowStats {     // one logit row after its chunks are combined
    float M, MC;
    double S;
    float thr;        // top-k threshold on the stored logit (-inf without top-k)
    int status;       // ROW_OK or ROW_NONFINITE
    int klist_n;      // top-k: number of kept (index, value) pairs listed, -1 if not listed
    int dense;        // top-k: row needs the exact fallback path
    // filled in advance by the top-k finish kernel (the plan reads them when `pre` is set)
    float lse;        // natural-log normaliser of logits / T over the kept tokens
    float invS;       // fp32(1 / S)
    float lx_hi, lx_lo;  // log2 p(x) of the token this row scores as a pair of floats (hi NaN:
                         // none or out of range; -inf: p(x) = 0)
};

struct Plan {         // one request, after the acceptance scan
    int status;
    int A;            // accepted draft count
    int rp, rq;       // row of p (target) and q (draft, -1 for the bonus draw)
    float MCp, MCq, invSp, invSq, thrp, thrq;
    double u;         // correction or bonus uniform
};

struct __align__(8) TopkEntry {  // one kept top-k candidate
    float x;
    int idx;
};

struct ArgmaxPartial {
    float best;
    int idx;
    int nan;
    int pad;
};
static_assert(sizeof(ArgmaxPartial) == 16, "argmax partials are read as one 16-byte vector");

// ---------------------------------------------------------------- parameter blocks

// Streaming task geometry (persistent warps).  A task is a contiguous run of vectors of one row
// (or row pair): STEPS steps of 32 lanes x U vectors; lane l of step j reads vectors
// base + j*32*U + u*32 + l, so every load instruction of a warp covers 32 consecutive vectors.
constexpr int U1 = 8, ST1 = 4, TV1 = 32 * U1 * ST1;  // row statistics / argmax: 1024 vectors
constexpr int U2 = 4, ST2 = 4, TV2 = 32 * U2 * ST2;  // residual pass over a row pair: 512 vectors
constexpr int RCV = 8;  // residual pass over 16-byte vectors: vectors per row and thread of one CTA
constexpr int SEGV = 32;                             // vectors per residual segment
enum { RES_PLAIN = 0, RES_MASK = 1, RES_THR = 2 };   // residual pass variants
enum { MASK_NONE = 0, MASK_REGS = 1, MASK_RING = 2 };  // streaming kernel: where mask bits come from

struct SpecParams {
    const void* target;   // [B, gamma+1, V]
    const void* draft;    // [B, gamma, V]
    const int32_t* tokens;
    const float* uniforms;
    int B, gamma, V, R;   // R = 2*gamma+1 rows per request
    int dtype, vec;       // elements per vector load (8 bf16 / 4 fp32 / 1 unaligned)
    long long nvec;       // vectors per row
    float c;              // log2(e)/T
    double T;
    double invT;          // 1/T
    float invT_hi, invT_lo;  // 1/T as an unevaluated pair of floats
    int top_k;
    int pin_pairs;        // row pairs 0..pin_pairs-1 are read with L2 evict_last
    // softmax path: stats tasks (row, slice) and residual tasks (request, slice)
    int S1, S2, nseg;
    long long tasks1, tasks2;
    // top-k chunking and capacities
    int CT;               // 32 KB chunks per row
    int nsegr, sps;       // segments per row (<= 4) and chunks per segment
    int cap_s;            // capacity of one warp's candidate list for a segment (entries)
    int cap_k;            // per-row kept-list capacity
    // outputs
    int32_t* accepted_len;
    int32_t* out_tokens;
    int32_t* row_status;
    float* aux_lse_p;
    float* aux_lse_q;
    float* aux_accept;
    // workspace
    Partial* partials;    // [B*R*S1]
    RowStats* rstats;     // [B*R]
    Plan* plan;           // [B]
    float* segs;          // [B*nseg]
    unsigned* row_ctr;    // [B*R]
    unsigned* req_ctr;    // [B]
    unsigned* res_ctr;    // [B]
    unsigned* work;       // [2] task counters of the two streaming kernels
    TopkEntry* clist;     // [B*R*nsegr*cap_s] per segment: candidate groups (unordered): the
                          // group's maximum and the index of its first element
    uint4* cdata;         // [same] the candidate group's raw 16 bytes (8 bf16 or 4 fp32 logits)
    int* ccount;          // [B*R*nsegr] groups listed, or TK_NONFINITE / TK_OVERFLOW / TK_TIMEOUT
    float* cbound;        // [B*R*nsegr] the segment's final bound: >= k of its elements reach it
    TopkEntry* klist;     // [B*R*cap_k] per-row kept list, sorted by index
    unsigned* dense_ctr;  // [B]
    int* ndense;          // [B]
    // counters the first kernel clears itself (streaming paths; otherwise a memset does): words
    unsigned* ctr_clear;
    int ctr_words;
    // SMC-SD round (smc_verify): no acceptance test, every draft position is kept; uniforms are
    // [B, 2]: slot 0 draws the extension token from row gamma, slot 1 is the particle's ancestor draw
    int smc;
    const float* smc_logw_in;  // [B] log weight before the round
    float* smc_log_ratio;      // [B] or null: sum over the draft positions of log p - log q
    float* smc_logw;           // [B] logw_in + log ratio (the group step may reset it)
    // grammar mask (spec_verify_masked): [B, gamma+1, mwords] allowed-token bits, one 32-bit word
    // per 32 tokens (bit v % 32 of word v / 32); position i masks target row i and draft row i
    const uint32_t* mask;
    int mwords;
    float top_p;          // top-p processor (spec_verify_topp): < 1 keeps each row's nucleus
    int wait_limit;       // polls of a ring or segment wait before it gives up (ROW_TIMEOUT)
};

struct TreeParams {
    const void* logits;   // [B, N+1, V]
    const int32_t* parents;
    const int32_t* tokens;
    int B, N, V, R;       // R = N+1
    int dtype, vec;
    long long nvec;
    int S1;               // slices per row
    long long tasks;
    int max_out;
    int32_t* accepted_len;
    int32_t* out_tokens;
    int32_t* out_nodes;
    int32_t* row_status;
    ArgmaxPartial* partials;  // [B*R*S1]
    unsigned* req_ctr;        // [B]
    unsigned* work;           // [1]
    int32_t* amax;            // [B*R]
    int32_t* scratch;         // [B*N*2] depth / valid of each node
    int wait_limit;           // polls of a ring wait before it gives up (ROW_TIMEOUT)
};

// ---------------------------------------------------------------- small device helpers

// Pairs of fp32 in one 64-bit register, with the packed fp32 instructions of this GPU family: each
// half is computed exactly as the scalar instruction would (same rounding, no flush to zero).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// L2 cache policies for 16-byte streaming loads (L1 bypassed)
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_stream_v4_pol(const void* p, uint64_t pol)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ unsigned short ld_u16_pol(const void* p, uint64_t pol)
{
    unsigned short r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(r) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ld_u32_pol(const void* p, uint64_t pol)
{
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// packed bf16x2 maximum; NaN lanes are ignored unless both inputs are NaN
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// packed bf16x2 maximum that propagates NaN
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// fp32 maximum that propagates NaN
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// one logit as fp32 (scalar path)
__device__ __forceinline__ float load_logit(const void* row, int dtype, long long i)
{
    if (dtype == DT_BF16) {
        unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
        return __uint_as_float(((uint32_t)h) << 16);
    }
    return __ldg(reinterpret_cast<const float*>(row) + i);
}

__device__ __forceinline__ size_t esize(int dtype) { return dtype == DT_BF16 ? 2 : 4; }

// request b, row r (r <= gamma: target row r; r > gamma: draft row r - gamma - 1)
__device__ __forceinline__ const char* spec_row_ptr(const SpecParams& P, int b, int r)
{
    const size_t es = esize(P.dtype);
    if (r <= P.gamma)
        return reinterpret_cast<const char*>(P.target) +
               ((size_t)b * (P.gamma + 1) + r) * (size_t)P.V * es;
    return reinterpret_cast<const char*>(P.draft) +
           ((size_t)b * P.gamma + (r - P.gamma - 1)) * (size_t)P.V * es;
}

// Vector v of a row as fp32 values.  VEC = 8 (bf16, 16-byte aligned rows), 4 (fp32, aligned) or
// 1 (any layout).  Only called for in-range vectors.
template <int DT, int VEC>
__device__ __forceinline__ void load_vec(const char* row, long long v, float (&x)[VEC])
{
    if constexpr (VEC == 1) {
        x[0] = load_logit(row, DT, v);
    } else if constexpr (DT == DT_BF16) {
        static_assert(VEC == 8, "bf16 vectors hold 8 values");
        uint4 w = ld_stream_v4(row + v * 16);
        x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
        x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
    } else {
        static_assert(VEC == 4, "fp32 vectors hold 4 values");
        uint4 w = ld_stream_v4(row + v * 16);
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
    }
}

// Vector v of a row as fp32 values, loaded with an L2 cache policy.
template <int DT, int VEC>
__device__ __forceinline__ void load_vec_pol(const char* row, long long v, uint64_t pol, float (&x)[VEC])
{
    if constexpr (VEC == 1) {
        if constexpr (DT == DT_BF16) x[0] = __uint_as_float(((uint32_t)ld_u16_pol(row + v * 2, pol)) << 16);
        else x[0] = __uint_as_float(ld_u32_pol(row + v * 4, pol));
    } else if constexpr (DT == DT_BF16) {
        uint4 w = ld_stream_v4_pol(row + v * 16, pol);
        x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
        x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
    } else {
        uint4 w = ld_stream_v4_pol(row + v * 16, pol);
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
    }
}

__device__ __forceinline__ uint4 lds128(const uint4* p)
{
    uint4 r;
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a) : "memory");
    return r;
}

// ---------------------------------------------------------------- bulk copies (TMA engine)
//
// One thread arms an mbarrier with the byte count and issues cp.async.bulk global -> shared; the
// consumers poll the barrier's phase.  Every wait is bounded: after a limit of polls it gives up and
// reports failure, and the caller turns that into a status instead of hanging.  The ring and segment
// waits take the call's limit (the parameter block's wait_limit: MBAR_SPIN_LIMIT unless a test set
// a smaller one through spec_set_wait_limit); the final wait for the copies still in flight before
// a CTA leaves always takes MBAR_SPIN_LIMIT, so no CTA exits while a copy could still land.

constexpr int MBAR_SPIN_LIMIT = 1 << 22;

__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
// makes barrier initialisation visible to the async proxy before the first copy uses it
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// orders this CTA's generic-proxy shared-memory accesses before later async-proxy (bulk copy) ones
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to shared memory,
// completing on `bar`, with an L2 cache policy.  Called by one thread.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                          uint64_t pol)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol) : "memory");
}

// Two bulk copies completing on one barrier: `bytes` and `bytes2` (multiples of 16; all addresses
// 16-byte aligned) from global to shared memory.  Called by one thread.
__device__ __forceinline__ void bulk_load2(void* dst, const void* src, unsigned bytes, void* dst2,
                                           const void* src2, unsigned bytes2, uint64_t* bar,
                                           uint64_t pol, uint64_t pol2)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes + bytes2) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_addr(dst2)), "l"(src2), "r"(bytes2), "r"(smem_addr(bar)), "l"(pol2) : "memory");
}

// One arrival on `bar` (release: this thread's earlier shared-memory reads are ordered before it).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

// Bounded wait for the phase with parity `parity` of `bar` to complete: at most `limit` polls
// (none when limit <= 0); false if they ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int limit)
{
    const unsigned a = smem_addr(bar);
    for (int i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile("{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
                     : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

// Streaming kernels: persistent CTAs (two per SM) fetch 32 KB chunks of one row with bulk copies
// into a ring of STREAM_STAGES shared-memory stages; thread t reads vectors t + j*NT (j <
// STREAM_NV) of a stage into registers.
constexpr int STREAM_CHUNK_BYTES = 32768;
constexpr int STREAM_NV = STREAM_CHUNK_BYTES / (NT * 16);  // 16-byte vectors per thread (8)
constexpr int STREAM_STAGES = 3;
constexpr int STREAM_SMEM = STREAM_STAGES * STREAM_CHUNK_BYTES;
// a stage's grammar-mask bits when they travel with the chunk: one bit per element, at most a bf16
// chunk's (STREAM_CHUNK_BYTES / 2 elements)
constexpr int STREAM_MASK_BYTES = STREAM_CHUNK_BYTES / 16;
constexpr int STREAM_SMEM_MASKED = STREAM_SMEM + STREAM_STAGES * STREAM_MASK_BYTES;

// Warp-specialised streaming (the plain, tree and typical kernels) with NG consumer groups per
// CTA: group g (warps g * WARPS .. g * WARPS + WARPS - 1) is virtual CTA NG * blockIdx.x + g of
// NG * gridDim.x, takes chunks vb, vb + that stride, ... and reads its own STREAM_STAGES-stage ring
// (stages g * STREAM_STAGES ..).  With NG = 1 that is one ring per CTA and two CTAs per SM.  Two such
// CTAs on one SM do not run equally fast: on the typical stream, whose chunks cost the most
// arithmetic, the later CTA took about 15% longer per chunk, so the SMs' second CTAs finished last.
// With NG = 2 (one CTA per SM) one producer lane feeds the two rings in turn, one chunk each, so a
// group that falls behind holds the other back and the SM's chunks finish together.
template <int NG>
constexpr int stream_threads() { return NG * NT + 32; }  // the producer warp last

// A consumer thread's place: its group, virtual CTA, the virtual CTAs, its thread and warp in the group
template <int NG>
struct StreamGroup {
    int g, vb, stride, t, w;
    __device__ __forceinline__ StreamGroup()
    {
        g = NG > 1 ? (int)threadIdx.x / NT : 0;
        vb = NG * (int)blockIdx.x + g;
        stride = NG * (int)gridDim.x;
        t = (int)threadIdx.x - g * NT;
        w = t >> 5;
    }
};

// The producer lane.  issue(s, id) issues the copy of chunk id into stage s (of all the rings'
// NG * STREAM_STAGES), completing on full[s]; a stage is refilled once all WARPS warps of
// its group have arrived on empty[s].  A wait that runs out (after `limit` polls), or a consumer's
// (sfail), stops the issue; the copies in flight are then waited for with the full
// MBAR_SPIN_LIMIT, so the CTA never leaves while one could still land.
template <int NG, class Issue>
__device__ void ring_produce(uint64_t* full, uint64_t* empty, int* sfail, int nch, int limit, Issue issue)
{
    int stg[NG], id[NG];
    unsigned ph[NG];
    long long n[NG];
    const int stride = NG * (int)gridDim.x;
    for (int g = 0; g < NG; ++g) {
        stg[g] = 0;
        ph[g] = 0u;
        n[g] = 0;
        id[g] = NG * (int)blockIdx.x + g;
    }
    for (bool more = true; more;) {
        more = false;
        for (int g = 0; g < NG; ++g) {
            if (id[g] >= nch) continue;
            const int s = g * STREAM_STAGES + stg[g];
            if (*reinterpret_cast<volatile int*>(sfail) ||
                (n[g] >= STREAM_STAGES && !mbar_wait(&empty[s], ph[g] ^ 1u, limit))) {
                *reinterpret_cast<volatile int*>(sfail) = 1;
                more = false;
                break;
            }
            issue(s, id[g]);
            ++n[g];
            if (++stg[g] == STREAM_STAGES) {
                stg[g] = 0;
                ph[g] ^= 1u;
            }
            id[g] += stride;
            more = true;
        }
    }
    // the last fill of every stage: no later fill of that stage exists, so its phase is unambiguous
    for (int g = 0; g < NG; ++g)
        for (long long j = (n[g] > STREAM_STAGES ? n[g] - STREAM_STAGES : 0); j < n[g]; ++j)
            (void)mbar_wait(&full[g * STREAM_STAGES + j % STREAM_STAGES], (unsigned)(j / STREAM_STAGES) & 1u,
                            MBAR_SPIN_LIMIT);
}

// persistent grid of CTAs: resident CTAs per SM x SMs, at most one per task (the occupancy query
// runs once per kernel)
template <auto K>
inline unsigned cta_grid(long long tasks, int sms, size_t smem, int threads = NT)
{
    static int per_sm = 0;
    if (per_sm < 1) {
        int n = 0;
        if (smem > 48 * 1024) cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, threads, smem) != cudaSuccess || n < 1) n = 1;
        per_sm = n;
    }
    const long long cap = (long long)per_sm * sms;
    return (unsigned)(tasks < 1 ? 1 : (tasks < cap ? tasks : cap));
}

// Called at the start of a streaming kernel: its first CTA zeroes the call's completion counters,
// which no kernel touches before that grid has completed (the later kernels wait for it).
__device__ __forceinline__ void clear_counters(unsigned* ctr, int words)
{
    if (blockIdx.x == 0 && ctr)
        for (int i = threadIdx.x; i < words; i += blockDim.x) ctr[i] = 0u;
}

// Programmatic dependent launch: a kernel launched with launch_dependent may start while the
// previous kernel on the stream is still running; before it reads anything that kernel wrote it
// calls pdl_wait(), which returns once the previous grid has completed and its writes are visible
// (a no-op for an ordinary launch).  pdl_trigger() lets the next grid launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t st, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_dependent for a kernel of thread-block clusters of `cluster` CTAs along x
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                            size_t smem, unsigned cluster, cudaStream_t st,
                                            Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// raises a kernel's dynamic shared-memory limit to `smem` when above the default
template <auto K>
inline void set_smem_limit(size_t smem)
{
    static size_t done = 0;
    if (smem > 48 * 1024 && smem > done) {
        cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        done = smem;
    }
}

// One vector of a row kept as raw bits until it is used: 16 bytes (8 bf16 or 4 fp32) or a single
// element for the unaligned path.
template <int DT, int VEC>
struct RawVec {
    uint4 w;
    __device__ __forceinline__ void load(const char* row, long long v, uint64_t pol)
    {
        if constexpr (VEC == 1) {
            if constexpr (DT == DT_BF16) w.x = ((uint32_t)ld_u16_pol(row + v * 2, pol)) << 16;
            else w.x = ld_u32_pol(row + v * 4, pol);
        } else {
            w = ld_stream_v4_pol(row + v * 16, pol);
        }
    }
    __device__ __forceinline__ void fill_neg_inf()
    {
        const uint32_t p = (DT == DT_BF16 && VEC == 8) ? 0xff80ff80u : 0xff800000u;
        w = make_uint4(p, p, p, p);
    }
    __device__ __forceinline__ float get(int e) const
    {
        if constexpr (VEC == 1) {
            return __uint_as_float(w.x);
        } else if constexpr (DT == DT_BF16) {
            const uint32_t q = (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
            return (e & 1) ? bf16hi(q) : bf16lo(q);
        } else {
            return __uint_as_float(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
        }
    }
};

// ---------------------------------------------------------------- grammar mask
//
// "Exact speculative and assisted decoding for TinyRustLM", "Grammar and deterministic
// opportunities": a grammar mask replaces q by q_G(x) = q(x) 1[x in A_G] / sum over A_G, the same
// for p.  A token outside A_G is turned into a -inf logit the moment it is loaded, so every later
// step (maximum, sum, gathered token, residual, draw) sees only A_G and the renormalisation is the
// softmax's own.

// the mask words of request b's row r (target row r <= gamma, else draft row r - gamma - 1): both
// rows of position i share position i's valid set
__device__ __forceinline__ const uint32_t* spec_mask_row(const SpecParams& P, int b, int r)
{
    const int pos = (r <= P.gamma) ? r : r - P.gamma - 1;
    return P.mask + ((size_t)b * (P.gamma + 1) + pos) * (size_t)P.mwords;
}

// allowed bits of the VEC elements of vector v (VEC = 1, 4 or 8 divides 32): bit e = element e
template <int VEC>
__device__ __forceinline__ uint32_t allowed_bits(const uint32_t* mrow, long long v)
{
    const long long e0 = v * VEC;
    const uint32_t w = __ldg(mrow + (e0 >> 5));
    return (w >> (unsigned)(e0 & 31)) & ((VEC == 32) ? 0xffffffffu : ((1u << VEC) - 1u));
}

// one vector of raw logits with its disallowed elements replaced by -inf bit patterns (RawVec layout:
// VEC == 1 holds one fp32 pattern in .x, bf16 as its high half)
template <int DT, int VEC>
__device__ __forceinline__ void mask_raw(uint4& w, uint32_t bits)
{
    if constexpr (VEC == 1) {
        if (!(bits & 1u)) w.x = 0xff800000u;
    } else if constexpr (DT == DT_BF16) {
        // element 2k is the low half of word k, element 2k + 1 the high half.  The keep mask of word
        // k comes from one byte permute in sign-replicate mode: bit 2k moved to the top of byte 0
        // fills bytes 0-1, bit 2k + 1 moved to the top of the second operand's byte 0 fills bytes 2-3.
        auto sel = [bits](uint32_t x, int k) {
            uint32_t keep;
            asm("prmt.b32 %0, %1, %2, 0xCC88;" : "=r"(keep) : "r"(bits << (7 - 2 * k)), "r"(bits << (6 - 2 * k)));
            return (x & keep) | (0xff80ff80u & ~keep);
        };
        w.x = sel(w.x, 0);
        w.y = sel(w.y, 1);
        w.z = sel(w.z, 2);
        w.w = sel(w.w, 3);
    } else {
        if (!(bits & 1u)) w.x = 0xff800000u;
        if (!(bits & 2u)) w.y = 0xff800000u;
        if (!(bits & 4u)) w.z = 0xff800000u;
        if (!(bits & 8u)) w.w = 0xff800000u;
    }
}

// the same on values already converted to fp32
template <int VEC>
__device__ __forceinline__ void mask_vals(float (&x)[VEC], uint32_t bits)
{
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (!((bits >> e) & 1u)) x[e] = NEG_INF;
}

// the stored logit of token tok in request b's row r, -inf when the grammar mask removes it
__device__ __forceinline__ float masked_logit(const SpecParams& P, int b, int r, int dtype, int tok)
{
    if (P.mask && !((__ldg(spec_mask_row(P, b, r) + (tok >> 5)) >> (tok & 31)) & 1u)) return NEG_INF;
    return load_logit(spec_row_ptr(P, b, r), dtype, tok);
}

// warp-wide claim of the next task index from a global counter (lane 0 increments)
__device__ __forceinline__ long long claim_task(unsigned* ctr)
{
    unsigned t = 0;
    if ((threadIdx.x & 31) == 0) t = atomicAdd(ctr, 1u);
    return (long long)__shfl_sync(0xffffffffu, t, 0);
}

// Warp-level arrive: after this warp's global writes, lane 0 increments the counter; returns true
// in every lane of the warp that arrived last.  Never waits.
__device__ __forceinline__ bool warp_arrive_last(unsigned* ctr, unsigned expected)
{
    int last = 0;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        __threadfence();
        last = (atomicAdd(ctr, 1u) == expected - 1);
        if (last) __threadfence();
    }
    return __shfl_sync(0xffffffffu, last, 0) != 0;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Error-free transformation (Knuth's TwoSum) in fp32: a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// A value carried as an unevaluated pair hi + lo of floats (|lo| <= ulp(hi) / 2): about 48
// significant bits from fp32 operations only (the fp64 pipe is very slow on this part).
struct DFloat {
    float hi, lo;
};
__device__ __forceinline__ DFloat df_make(float hi, float lo)
{
    DFloat r;
    r.hi = __fadd_rn(hi, lo);
    r.lo = __fsub_rn(lo, __fsub_rn(r.hi, hi));  // Dekker's FastTwoSum (|hi| >= |lo|)
    return r;
}
__device__ __forceinline__ DFloat df_add(DFloat x, DFloat y)
{
    float s, e;
    two_sum(x.hi, y.hi, s, e);
    return df_make(s, __fadd_rn(e, __fadd_rn(x.lo, y.lo)));
}
// x * (c_hi + c_lo) for a constant given as a pair
__device__ __forceinline__ DFloat df_mul(DFloat x, float c_hi, float c_lo)
{
    const float p = __fmul_rn(x.hi, c_hi);
    const float e = fmaf(x.hi, c_hi, -p);  // the product's rounding error, exact
    return df_make(p, fmaf(x.hi, c_lo, fmaf(x.lo, c_hi, e)));
}
__device__ __forceinline__ double df_to_double(DFloat x) { return (double)x.hi + (double)x.lo; }

// Fixed-point masses: 2^40 w rounded toward zero for a mass w in [0, 1], from the float's bits
// with integer operations only (a conversion to a 64-bit integer is not a fast-pipe instruction).
// Sums of them are exact and independent of order, so a kept set's mass does not depend on
// scheduling.
constexpr double FIXED_ONE = 1099511627776.0;  // 2^40
__device__ __forceinline__ unsigned long long fixed_mass(float w)
{
    const uint32_t u = __float_as_uint(w);
    const int e = (int)(u >> 23);     // biased exponent; w >= 0
    if (e == 0 || e > 127) return 0ull;  // zero (the exponential flushes subnormals); NaN or inf
    const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
    const int sh = e - 127 - 23 + 40;  // 2^40 w = m 2^sh, sh <= 17
    return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

// a fixed-point sum as a pair of floats (exact in fp64 up to 2^53)
__device__ __forceinline__ DFloat fixed_to_df(unsigned long long f)
{
    const double d = (double)f * (1.0 / FIXED_ONE);
    const float hi = (float)d;
    return df_make(hi, (float)(d - (double)hi));
}

// Sum over the warp of pairs; every lane gets the same pair (the butterfly adds the same two
// operands in each pair of lanes, and the pair sum is symmetric).
__device__ __forceinline__ DFloat warp_sum_df(DFloat v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        DFloat w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = df_add(v, w);
    }
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// inclusive prefix sum across a warp
template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// block-wide maximum (all threads receive it)
__device__ __forceinline__ float block_max(float v, float* sh /* >= WARPS floats */)
{
    v = warp_max(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = sh[0];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) r = fmaxf(r, sh[w]);
    return r;
}

// block-wide sum: fp32 within warps, fp64 across warps in warp order (all threads receive it)
__device__ __forceinline__ double block_sum_f32(float v, double* sh /* >= WARPS doubles */)
{
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = (double)v;
    __syncthreads();
    double r = 0.0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) r += sh[w];
    return r;
}

__device__ __forceinline__ int block_sum_int(int v, int* sh)
{
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) r += sh[w];
    return r;
}

// block-wide exclusive prefix sum in fp64 (thread order); returns the exclusive prefix and
// writes the total to *total
__device__ __forceinline__ double block_excl_scan_f64(double v, double* sh, double* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const double incl = warp_incl_scan(v);
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    double before = 0.0, tot = 0.0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        if (w < warp) before += sh[w];
        tot += sh[w];
    }
    *total = tot;
    return before + (incl - v);
}

// Arrive on a completion counter after this CTA's global writes; returns true in every thread of
// the CTA that arrived last.  Never waits.  The counters are cleared by the host call before the
// first kernel of the call.
__device__ __forceinline__ bool arrive_last(unsigned* ctr, unsigned expected, int* sh_flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned prev = atomicAdd(ctr, 1u);
        int last = (prev == expected - 1);
        if (last) __threadfence();
        *sh_flag = last;
    }
    __syncthreads();
    return *sh_flag != 0;
}

// ---------------------------------------------------------------- outputs

// Writes a request's outputs: the accepted draft prefix, the drawn token, -1 padding.  Called by
// `n` cooperating threads with ranks 0..n-1.
__device__ __forceinline__ void emit_spec_n(const SpecParams& P, int b, int status, int A, int tok,
                                            int rank, int n)
{
    const int g = P.gamma;
    int32_t* out = P.out_tokens + (size_t)b * (g + 1);
    const int32_t* dt = P.tokens + (size_t)b * g;
    for (int i = rank; i <= g; i += n) {
        int v = -1;
        if (status == ROW_OK) v = (i < A) ? dt[i] : (i == A ? tok : -1);
        out[i] = v;
    }
    if (rank == 0) {
        P.accepted_len[b] = (status == ROW_OK) ? A : -1;
        if (P.row_status) P.row_status[b] = status;
    }
}
__device__ __forceinline__ void emit_spec(const SpecParams& P, int b, int status, int A, int tok)
{
    emit_spec_n(P, b, status, A, tok, threadIdx.x, NT);
}
__device__ __forceinline__ void emit_spec_warp(const SpecParams& P, int b, int status, int A, int tok)
{
    emit_spec_n(P, b, status, A, tok, threadIdx.x & 31, 32);
}

// ---------------------------------------------------------------- host launchers (one per .cu)

// Persistent grid for kernel K: enough CTAs for every task warp, at most the CTAs that fit on
// `sms` SMs at once.  The occupancy (and the dynamic shared-memory opt-in above 48 KB) is queried
// once per kernel.
template <auto K>
inline unsigned persistent_grid(long long tasks, int sms, int threads = NT, size_t smem = 0)
{
    static int per_sm = 0;
    if (per_sm < 1) {
        int n = 0;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, threads, smem) != cudaSuccess || n < 1) n = 1;
        per_sm = n;
    }
    const int wpc = threads / 32;
    const long long want = (tasks + wpc - 1) / wpc;
    const long long cap = (long long)per_sm * sms;
    return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

// Measurement aid (spec_set_kernel_events): events recorded on the call's stream around the
// call's dominant kernel, or none.
struct KernelEvents {
    cudaEvent_t start = nullptr, stop = nullptr;
};
extern KernelEvents g_kernel_events;
inline void mark_kernel_start(cudaStream_t st)
{
    if (g_kernel_events.start && g_kernel_events.stop) cudaEventRecord(g_kernel_events.start, st);
}
inline void mark_kernel_stop(cudaStream_t st)
{
    if (g_kernel_events.start && g_kernel_events.stop) cudaEventRecord(g_kernel_events.stop, st);
}

// spec_stats_kernel + spec_resample_kernel for the dtype / vector width in P
cudaError_t launch_softmax_path(const SpecParams& P, int sms, cudaStream_t st);
// the plain path's row statistics alone, and its correction draw with top-p thresholds
cudaError_t launch_softmax_stats(const SpecParams& P, int sms, cudaStream_t st);
cudaError_t launch_softmax_resample_thr(const SpecParams& P, int sms, cudaStream_t st);
// top-p: statistics, per-row threshold select and plan, thresholded draw
cudaError_t launch_topp_path(const SpecParams& P, int sms, cudaStream_t st);
// topk_stream_kernel + topk_finish_kernel + topk_dense_kernel
cudaError_t launch_topk_path(const SpecParams& P, int sms, cudaStream_t st);
// tree_argmax_kernel
cudaError_t launch_tree_path(const TreeParams& P, int sms, cudaStream_t st);

}  // namespace sv
