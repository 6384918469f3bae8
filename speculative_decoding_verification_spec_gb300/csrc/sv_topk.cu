// sv_topk.cu -- exact speculative sampling with a top-k processor on p and q.
//
// M7.1 section 0x03D: truncation keeps the method exact when p and q are the truncated,
// renormalised distributions and q is the one that sampled the draft.  A row keeps every token
// whose stored logit is >= the row's k-th largest stored logit (counted with multiplicity), so ties
// at the threshold are all kept.
//
// Kernel 1 (topk_stream_kernel) streams every logit row once.  Rows are cut into 32 KB chunks and
// runs of chunks (segments, at most 4 per row); persistent CTAs, one per SM, each run two consumer
// groups, and the groups take segments round-robin.  For 16-byte aligned rows a group's producer warp
// fetches its chunks with bulk copies (TMA engine) into a ring of TK_STAGES shared-memory stages, so
// the next chunks are in flight while one is filtered; a producer more than TK_LEAD chunks ahead of
// the other group's waits a little, so that the SM's two groups finish together.  Each
// consumer thread holds its 64 (bf16) or 32 (fp32) elements of a chunk in registers; the consumer
// warps run independently of one another and meet once per segment.  The k-th largest of the NT
// per-thread maxima of a segment's first chunk (NT disjoint groups, so at least k elements are >=
// it) bounds the segment's k-th largest value from below; a histogram of the candidates found so
// far tightens the bound as the segment proceeds.  Only elements >= the bound -- a few dozen per
// chunk at k = 50 -- join the warp's candidate list for the segment.  Every bound is <= the row's
// k-th largest value g, so the lists hold every element >= g.
//
// Kernel 2 (topk_finish_kernel), one warp per row, selects g exactly from the union of the row's
// candidate lists, keeps the entries >= g and forms the normaliser (M, and S as a fixed-point sum,
// which does not depend on the order the lists deliver the entries in).  After a CTA barrier one
// warp runs the request's acceptance scan and draws the correction or bonus token directly from the
// kept list of the p row, sorted by index first: the residual vanishes outside K_p, so no second
// pass over V is needed.
//
// Rows whose candidates overflow the capacities (massive ties, k > NT, ...) are marked dense; the
// finish CTA of their request then completes it exactly with full-row passes (topk_dense_request).
#include <cuda_bf16.h>

#include "sv_plan.cuh"

namespace sv {

constexpr int TK_NREG = STREAM_CHUNK_BYTES / (NT * 4);  // 32-bit words per thread (32)
constexpr int TK_NV = STREAM_NV;                        // 16-byte vectors per thread (8)
constexpr int TK_STAGES = STREAM_STAGES;                // bulk-copy ring depth
constexpr int TK_GROUPS = 2;               // kernel 1: consumer groups per CTA (one CTA per SM)
constexpr int TK_SMEM = TK_GROUPS * STREAM_SMEM;        // dynamic shared memory of kernel 1: a ring per group
// per-chunk candidate count codes
constexpr int TK_OVERFLOW = -1, TK_NONFINITE = -2, TK_TIMEOUT = -3;
constexpr int TK_LEAD = 2;                 // kernel 1: chunks one group's producer may run ahead of the other's
constexpr int TK_LEAD_POLLS = 1024;        // kernel 1: polls before a producer stops waiting for the other group
constexpr int TK_PRODUCER = TK_GROUPS * WARPS;  // kernel 1: the first producer warp (one per group)
constexpr int TK_SLOTS = 4;                // kernel 1: per-segment shared state, by segment mod 4
constexpr int TK_THREADS = TK_GROUPS * (NT + 32);  // kernel 1: per group WARPS consumer warps + a producer

// order-preserving 32-bit key of a float; -0 and +0 map to the same key
__device__ __forceinline__ uint32_t okey(float x)
{
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// one candidate entry through L2 (written by the previous kernel)
__device__ __forceinline__ TopkEntry ld_entry(const TopkEntry* p)
{
    const int2 v = __ldcg(reinterpret_cast<const int2*>(p));
    TopkEntry e;
    e.x = __int_as_float(v.x);
    e.idx = v.y;
    return e;
}


// The k-th largest key (largest P with count(key >= P) >= k) among n keys produced by key_at(i),
// by one warp: bitwise search from the top bit, counting with a warp reduction per bit.
// bf16-valued keys differ only in their top 16 bits.
template <int DT, class KeyAt>
__device__ uint32_t warp_kth_key(int n, int k, KeyAt key_at)
{
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        unsigned cnt = 0;
        for (int i = lane; i < n; i += 32) cnt += key_at(i) >= want;
        if ((int)__reduce_add_sync(0xffffffffu, cnt) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

// Warp-level bitonic sort of e[0..n) by index (ascending), padding to a power of two.
__device__ void warp_sort_by_index(TopkEntry* e, int n)
{
    const int lane = threadIdx.x & 31;
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = n + lane; i < m; i += 32) { e[i].idx = 0x7fffffff; e[i].x = NEG_INF; }
    __syncwarp();
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = lane; i < m; i += 32) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const TopkEntry a = e[i], b = e[j];
                    if ((a.idx > b.idx) == up) { e[i] = b; e[j] = a; }
                }
            }
            __syncwarp();
        }
    }
}

// One warp: the correction / bonus draw of request b, planned as pl, from the kept list of the p
// row (nk entries of the workspace, in the order the lists gave them); the residual is zero outside
// K_p.  Each entry's residual is formed (with the draft row's logit at its token), and the entries
// are sorted by index into se (room for 2 * cap_k entries), since the draw walks the tokens in
// index order.  Sums in pairs of floats.
template <int DT>
__device__ void topk_request_draw(const SpecParams& P, const Plan& pl, int nk, TopkEntry* se, int b)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    if (pl.status != ROW_OK) {
        emit_spec_warp(P, b, pl.status, 0, -1);
        return;
    }
    const TopkEntry* kl = P.klist + ((size_t)b * P.R + pl.rp) * P.cap_k;
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    auto residual = [&](float xp, float xq) {
        const float pp = __fmul_rn(ex2(fmaf(xp, P.c, -pl.MCp)), pl.invSp);
        if (!rowq) return pp;
        const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, P.c, -pl.MCq)), pl.invSq) : 0.f;
        return fmaxf(__fsub_rn(pp, qq), 0.f);
    };
    if (nk <= 64) {
        // entries lane and lane + 32 in registers with their residuals; each goes to its rank, the
        // number of smaller indices (the indices are distinct), counted by shuffles
        TopkEntry a, c;
        a.idx = c.idx = 0x7fffffff;
        a.x = c.x = 0.f;
        float qa = 0.f, qc = 0.f;
        if (lane < nk) a = ld_entry(kl + lane);
        if (lane + 32 < nk) c = ld_entry(kl + lane + 32);
        if (rowq) {
            if (lane < nk) qa = load_logit(rowq, DT, a.idx);
            if (lane + 32 < nk) qc = load_logit(rowq, DT, c.idx);
        }
        int ra = 0, rc = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const int ia = __shfl_sync(FULL, a.idx, j), ic = __shfl_sync(FULL, c.idx, j);
            ra += (ia < a.idx) + (ic < a.idx);
            rc += (ia < c.idx) + (ic < c.idx);
        }
        if (lane < nk) se[ra] = TopkEntry{residual(a.x, qa), a.idx};
        if (lane + 32 < nk) se[rc] = TopkEntry{residual(c.x, qc), c.idx};
    } else {
        for (int i = lane; i < nk; i += 32) se[i] = ld_entry(kl + i);
        __syncwarp();
        warp_sort_by_index(se, nk);
        // the draft row's logits at the sorted tokens, eight per lane in flight, then residuals
        for (int i0 = 0; i0 < nk; i0 += 32 * 8) {
            float xq[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int i = i0 + 32 * t + lane;
                xq[t] = (rowq && i < nk) ? load_logit(rowq, DT, se[i].idx) : 0.f;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int i = i0 + 32 * t + lane;
                if (i < nk) se[i].x = residual(se[i].x, xq[t]);
            }
        }
    }
    __syncwarp();
    // each lane owns a contiguous block of the sorted list
    const int per = (nk + 31) / 32;
    const int i0 = min(lane * per, nk), i1 = min(i0 + per, nk);
    DFloat mine = df_make(0.f, 0.f);
    for (int i = i0; i < i1; ++i) mine = df_add(mine, df_make(se[i].x, 0.f));
    // inclusive scan of the lane blocks' masses, in pairs of floats
    DFloat incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        DFloat n;
        n.hi = __shfl_up_sync(FULL, incl.hi, o);
        n.lo = __shfl_up_sync(FULL, incl.lo, o);
        if (lane >= o) incl = df_add(n, incl);
    }
    const double Z = df_to_double(DFloat{__shfl_sync(FULL, incl.hi, 31), __shfl_sync(FULL, incl.lo, 31)});
    int tok = -1;
    if (Z > 0.0 && isfinite(Z)) {
        const double t = pl.u * Z;
        const double inc = df_to_double(incl), m = df_to_double(mine), excl = inc - m;
        unsigned own = __ballot_sync(FULL, m > 0.0 && t < inc);
        if (!own) {
            const unsigned pos = __ballot_sync(FULL, m > 0.0);
            own = pos ? (1u << (31 - __clz(pos))) : 0u;
        }
        if (own) {
            const int owner = __ffs(own) - 1;
            if (lane == owner) {
                const float tr = (float)(t - excl);  // mass still to pass inside this lane's block
                float run = 0.f;
                int lastpos = -1;
                for (int i = i0; i < i1; ++i) {
                    const float ri = se[i].x;
                    if (ri > 0.f) lastpos = i;
                    run += ri;
                    if (tr < run && ri > 0.f) { tok = se[i].idx; break; }
                }
                if (tok < 0 && lastpos >= 0) tok = se[lastpos].idx;
            }
            tok = __shfl_sync(FULL, tok, owner);
        }
    }
    emit_spec_warp(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}

// element index (within the row) of register slot s of this thread: vector j = s / VEC, element
// e = s % VEC of it; vectors of a thread are NT apart
template <int VEC>
__device__ __forceinline__ int slot_elem(int cbase, int s, int t)
{
    if constexpr (VEC == 1) return cbase + s * NT + t;
    else return cbase + ((s / VEC) * NT + t) * VEC + (s % VEC);
}

// The k-th largest (with multiplicity) of the n keys key_at(0..n), by one warp: a radix select
// over 8-bit digits, each digit resolved by a 256-bin histogram in shared memory (hist: 256 ints of
// this warp) and a suffix sum over it.  The digits start at the highest bit in which the keys differ
// (the bits above are common to all of them), so values spread over a narrow range take one pass.
// Bits below 16 of bf16-valued keys never differ.
template <int DT, class KeyAt>
__device__ uint32_t warp_kth_key_hist(int n, int k, int* hist, KeyAt key_at)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = lane; i < n; i += 32) {
        const uint32_t kx = key_at(i);
        kmin = min(kmin, kx);
        kmax = max(kmax, kx);
    }
    kmin = __reduce_min_sync(FULL, kmin);
    kmax = __reduce_max_sync(FULL, kmax);
    const uint32_t diff = kmin ^ kmax;
    if (diff == 0u) return kmax;
    const int hd = 31 - __clz(diff);  // highest differing bit
    const uint32_t common = (hd == 31) ? 0u : ~((2u << hd) - 1u);
    uint32_t prefix = kmax & common, mask = common;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    int kk = k;  // rank sought among the keys that match the prefix
#pragma unroll 1
    for (int shift = hd - 7; shift + 8 > lo; shift -= 8) {
        const uint32_t dmask = shift >= 0 ? (255u << shift) : (255u >> -shift);
#pragma unroll
        for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0;
        __syncwarp();
        for (int i = lane; i < n; i += 32) {
            const uint32_t kx = key_at(i);
            if ((kx & mask) == prefix) {
                const uint32_t dg = shift >= 0 ? (kx >> shift) & 255u : (kx << -shift) & 255u;
                atomicAdd(&hist[dg], 1);
            }
        }
        __syncwarp();
        int h8[8], c8 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            h8[i] = hist[lane * 8 + i];
            c8 += h8[i];
        }
        int suf = c8;  // counts in this lane's bins and above
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_down_sync(FULL, suf, o);
            if (lane + o < 32) suf += v;
        }
        const unsigned reach = __ballot_sync(FULL, suf >= kk);
        const int ls = reach ? 31 - __clz(reach) : 0;
        int bin = 0, above = 0;
        if (lane == ls) {
            int acc = suf - c8;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (acc + h8[i] >= kk) {
                    bin = lane * 8 + i;
                    above = acc;
                    break;
                }
                acc += h8[i];
            }
        }
        bin = __shfl_sync(FULL, bin, ls);
        above = __shfl_sync(FULL, above, ls);
        kk -= above;
        prefix |= shift >= 0 ? ((uint32_t)bin << shift) : ((uint32_t)bin >> -shift);
        mask |= dmask;
        __syncwarp();
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

constexpr int TK_BINS = 256;  // histogram of candidate values above a segment's first bound
static_assert(TK_BINS == NT, "one bin per thread to clear");
constexpr int TK_CAND_MIN = 512;           // finish kernel: candidate elements of a row (at least)
// finish kernel: candidate capacity of a row, which also holds the kept list and the draw scratch
__device__ __host__ __forceinline__ int topk_cand_cap(int cap_k) { return cap_k > TK_CAND_MIN ? cap_k : TK_CAND_MIN; }

// Position in the segment sequence blockIdx.x, blockIdx.x + stride, ... with the segment's row and
// its index within the row kept up to date without divisions.
struct SegCursor {
    int sg, row_id, si, drow, dsi;
    __device__ __forceinline__ void init(int start, int stride, int nsegr)
    {
        sg = start;
        row_id = start / nsegr;
        si = start % nsegr;
        drow = stride / nsegr;
        dsi = stride % nsegr;
    }
    __device__ __forceinline__ void next(int stride, int nsegr)
    {
        sg += stride;
        row_id += drow;
        si += dsi;
        if (si >= nsegr) {
            si -= nsegr;
            ++row_id;
        }
    }
};

// The bound a segment's histogram gives (one warp): the lowest bin edge with at least k counted
// group maxima at or above it, or -inf if fewer than k were counted.  Bin b counts the maxima whose
// order-preserving key lies in [key0 + (b << 16), key0 + ((b + 1) << 16)), the last bin everything
// above.  Every counted maximum is a distinct element of the segment, so at least k of its elements
// reach the bound.
__device__ __forceinline__ float hist_bound(const int* h, int k, uint32_t key0)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    int c8 = 0;
    int hb[TK_BINS / 32];
#pragma unroll
    for (int i = 0; i < TK_BINS / 32; ++i) {
        hb[i] = h[lane * (TK_BINS / 32) + i];
        c8 += hb[i];
    }
    int suf = c8;  // counts in this lane's bins and above
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_down_sync(FULL, suf, o);
        if (lane + o < 32) suf += v;
    }
    const unsigned reach = __ballot_sync(FULL, suf >= k);
    if (!reach) return NEG_INF;
    const int ls = 31 - __clz(reach);  // highest lane whose suffix reaches k
    int bin = -1;
    if (lane == ls) {
        int acc = suf - c8;  // counts above this lane's bins
#pragma unroll
        for (int i = TK_BINS / 32 - 1; i >= 0; --i) {
            acc += hb[i];
            if (bin < 0 && acc >= k) bin = lane * (TK_BINS / 32) + i;
        }
    }
    bin = __shfl_sync(FULL, bin, ls);
    return key_value(key0 + ((uint32_t)bin << 16));
}

// The bound tau of a segment from its first chunk: the k-th largest of the NT thread maxima of the
// chunk (valid for k <= NT: NT disjoint groups, so at least k elements reach it), as an
// order-preserving key.  Group g is the set of elements consumer thread g holds -- vectors g + NT i
// of the chunk -- so the value is the one the consumer warps would select themselves.  Computed by
// one warp (the producer): lane l takes groups l + 32 j, from the stage (BULK) or from the row.
template <int DT, bool BULK>
__device__ uint32_t chunk_tau_key(const uint4* stage, const char* row, int cbase, int cend, int k)
{
    constexpr int VEC = BULK ? ((DT == DT_BF16) ? 8 : 4) : 1;
    constexpr int EPT = (DT == DT_BF16) ? 2 * TK_NREG : TK_NREG;
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    uint32_t keys[NT / 32];
#pragma unroll
    for (int j = 0; j < NT / 32; ++j) {
        const int g = lane + 32 * j;
        float tm = NEG_INF;
        if constexpr (BULK) {
            uint32_t pm = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
#pragma unroll
            for (int i = 0; i < TK_NV; ++i) {
                if (cbase + (g + NT * i) * VEC < cend) {
                    const uint4 q = lds128(stage + g + NT * i);
                    if constexpr (DT == DT_BF16) {
                        pm = bmax2_nan(pm, bmax2_nan(bmax2_nan(q.x, q.y), bmax2_nan(q.z, q.w)));
                    } else {
                        tm = fmax_nan(tm, fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                                                       fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w))));
                    }
                }
            }
            if constexpr (DT == DT_BF16) tm = fmax_nan(bf16lo(pm), bf16hi(pm));
        } else {
            for (int s = 0; s < EPT; ++s) {
                const int e = cbase + s * NT + g;
                if (e < cend) tm = fmax_nan(tm, load_logit(row, DT, e));
            }
        }
        keys[j] = okey(tm);
    }
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        unsigned cnt = 0;
#pragma unroll
        for (int j = 0; j < NT / 32; ++j) cnt += keys[j] >= want;
        if ((int)__reduce_add_sync(FULL, cnt) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

// Kernel 1: warp-specialised, with TK_GROUPS consumer groups of WARPS warps per CTA (one CTA per
// SM); group grp is virtual CTA TK_GROUPS * blockIdx.x + grp and has its own ring, producer warp
// (warp TK_PRODUCER + grp) and per-segment state.  Two groups, rather than two CTAs of one group per
// SM: two CTAs on one SM do not run equally fast (the later one took about 6% longer per chunk here),
// and the SMs' second CTAs set the end of the grid.  BULK: rows of 16-byte vectors fetched by bulk
// copies into the stage ring; otherwise the consumer warps load their elements straight into
// registers.  A group takes segments (runs of up to P.sps chunks of one row) round-robin; segment j of
// the group uses slot j % TK_SLOTS of its per-segment shared state (histogram, list length, flags, tau).
//
// Producer (warp TK_PRODUCER + grp): lane 0 issues one bulk copy per chunk once every consumer warp
// of the group has released the stage, and while it is more than TK_LEAD chunks ahead of the other
// group's producer it first waits (at most TK_LEAD_POLLS polls: a group that falls behind holds the
// other back, so both end together; the wait only paces, nothing depends on it).  Copies complete
// on mbarriers: an "empty" mbarrier per stage, which every consumer warp of the group has
// released; a "full" mbarrier completes when the bytes land.  The whole warp also keeps the books of
// the group's segments: before segment j starts it waits until segment j - TK_SLOTS is done by every
// consumer warp of the group (a "done" mbarrier per slot), publishes that segment -- its list length
// (or a status) and its final bound from the complete histogram -- and clears the slot; once the
// first chunk of segment j has landed it selects the segment's first bound tau from it and publishes
// it through a "tau" mbarrier.  So the consumer warps never wait for one another, and they are at
// most TK_SLOTS - 1 segments apart from their producer.
//
// Consumers (warps grp * WARPS ..): each waits on its chunk's full barrier, reads its 64 (bf16) or 32
// (fp32) elements into registers and releases the stage.  Elements sit in groups of 4 registers
// (one 16-byte vector); a group whose maximum reaches the current bound beta goes to the segment's
// list (positions reserved with one shared-memory atomic per warp and chunk), and its maximum is
// counted in a histogram above tau (bins 2^16 apart in the order-preserving key: one bf16 value per
// bin).  Every count is a distinct element of the segment, whichever chunks the other warps have
// reached, so the warps take turns turning the histogram into a tighter bound for the chunks still
// to come, published as one 64-bit word (segment, key).
template <int DT, bool BULK>
__global__ void __launch_bounds__(TK_THREADS, 1) topk_stream_kernel(SpecParams P)
{
    constexpr int NREG = TK_NREG;
    constexpr int EPT = (DT == DT_BF16) ? 2 * NREG : NREG;  // elements per thread
    constexpr int CHUNK = NT * EPT;                          // elements per chunk
    constexpr int VEC = BULK ? ((DT == DT_BF16) ? 8 : 4) : 1;
    constexpr int ES = (DT == DT_BF16) ? 2 : 4;
    constexpr int G = 4, NG = NREG / G;        // groups of 4 registers: one 16-byte vector each
    constexpr int EPG = (DT == DT_BF16) ? 2 * G : G;  // elements per group
    static_assert(NREG % G == 0, "register groups");
    static_assert((WARPS & (WARPS - 1)) == 0, "warps take turns by chunk index");
    // per consumer group (the first index); BULK: a ring of TK_STAGES x (NT * TK_NV) vectors each
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ int hist[TK_GROUPS][TK_SLOTS][TK_BINS];
    __shared__ int scount[TK_GROUPS][TK_SLOTS];        // groups listed in the segment
    __shared__ int sflag[TK_GROUPS][TK_SLOTS];         // 1: a NaN or +inf in the segment; 4: a wait ran out
    __shared__ uint32_t tau_key[TK_GROUPS][TK_SLOTS];  // the segment's tau, published by the producer
    __shared__ int seg_id[TK_GROUPS][TK_SLOTS];        // the segment in the slot (producer's books)
    __shared__ unsigned long long pub[TK_GROUPS];      // (segment << 32) | key of the latest running bound
    __shared__ int issued[TK_GROUPS];                  // BULK: chunks issued; 2^30 once all are
    __shared__ int sfail;                              // a wait ran out in this CTA: nothing more is read
    __shared__ __align__(8) uint64_t full[TK_GROUPS][TK_STAGES];
    __shared__ __align__(8) uint64_t empty[TK_GROUPS][TK_STAGES];
    __shared__ __align__(8) uint64_t tau_bar[TK_GROUPS][TK_SLOTS];
    __shared__ __align__(8) uint64_t done_bar[TK_GROUPS][TK_SLOTS];

    pdl_trigger();  // the finish kernel may be scheduled as SMs free up; it waits for this grid
    clear_counters(P.ctr_clear, P.ctr_words);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int nsegs = P.B * P.R * P.nsegr;
    const int G0 = TK_GROUPS * gridDim.x;  // virtual CTAs: group grp is TK_GROUPS * blockIdx.x + grp
    const int k = P.top_k;
    // the consumer group a warp serves (consumer warps first, then one producer warp per group), and
    // a consumer's thread and warp within its group
    const int grp = warp < TK_GROUPS * WARPS ? warp / WARPS : warp - TK_GROUPS * WARPS;
    const int ct = tid - grp * NT, cw = warp - grp * WARPS;

    for (int i = tid; i < TK_GROUPS * TK_SLOTS * TK_BINS; i += TK_THREADS) (&hist[0][0][0])[i] = 0;
    if (tid < TK_GROUPS * TK_SLOTS) {
        (&scount[0][0])[tid] = 0;
        (&sflag[0][0])[tid] = 0;
    }
    if (tid == 0) {
        for (int g = 0; g < TK_GROUPS; ++g) {
            pub[g] = ~0ull;  // segment field 0xffffffff: no bound yet
            issued[g] = 0;
            for (int s = 0; s < TK_STAGES; ++s) {
                mbar_init(&full[g][s], 1);
                mbar_init(&empty[g][s], WARPS);
            }
            for (int s = 0; s < TK_SLOTS; ++s) {
                mbar_init(&tau_bar[g][s], 1);
                mbar_init(&done_bar[g][s], WARPS);
            }
        }
        sfail = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer warp
    if (warp >= TK_PRODUCER) {  // the producer warp of group grp
        const uint64_t pol = policy_evict_first();
        // the list length (or status) and final bound of the segment in slot `slot`, done or not
        auto publish = [&](int slot, bool done) {
            const int psg = seg_id[grp][slot];
            const uint32_t key0 = tau_key[grp][slot];
            const float tau = (k <= NT) ? key_value(key0) : NEG_INF;
            float bnd = tau;
            if (done && k <= NT && tau != NEG_INF) bnd = fmaxf(bnd, hist_bound(hist[grp][slot], k, key0));
            if (lane == 0) {
                const int c = scount[grp][slot], f = sflag[grp][slot];
                P.ccount[psg] = (!done || (f & 4)) ? TK_TIMEOUT : (f & 1) ? TK_NONFINITE
                              : (k > NT || c > P.cap_s) ? TK_OVERFLOW : c;
                P.cbound[psg] = bnd;
            }
        };
        SegCursor pc;
        pc.init(TK_GROUPS * blockIdx.x + grp, G0, P.nsegr);
        int stg = 0;
        unsigned ph = 0;
        long long n = 0;  // copies issued
        bool ok = true;
        int m = 0;        // this CTA's segment counter
        for (; pc.sg < nsegs; pc.next(G0, P.nsegr), ++m) {
            const int slot = m % TK_SLOTS;
            // the slot's previous segment: done by every consumer warp, published, cleared
            if (m >= TK_SLOTS) {
                const bool done = __all_sync(FULL, mbar_wait(&done_bar[grp][slot], (unsigned)((m - TK_SLOTS) / TK_SLOTS) & 1u, P.wait_limit));
                publish(slot, done);
                if (!done) ok = false;
#pragma unroll
                for (int i = 0; i < TK_BINS / 32; ++i) hist[grp][slot][lane + 32 * i] = 0;
                if (lane == 0) {
                    scount[grp][slot] = 0;
                    sflag[grp][slot] = 0;
                }
            }
            if (lane == 0) seg_id[grp][slot] = pc.sg;
            const int nst = min(P.sps, P.CT - pc.si * P.sps);
            const char* row = spec_row_ptr(P, pc.row_id / P.R, pc.row_id % P.R);
            // tau from the segment's first chunk, selected once the next copy is on its way (or at
            // the segment's end), so that the ring keeps filling meanwhile
            int t_stg = -1;
            unsigned t_ph = 0;
            int t_cbase = 0, t_cend = 0;
            auto publish_tau = [&]() {
                uint32_t key = 0;
                if (k <= NT) {
                    if constexpr (BULK) {
                        if (t_stg >= 0 && __all_sync(FULL, mbar_wait(&full[grp][t_stg], t_ph, P.wait_limit))) {
                            key = chunk_tau_key<DT, true>(ring + (size_t)(grp * TK_STAGES + t_stg) * NT * TK_NV,
                                                          nullptr, t_cbase, t_cend, k);
                            fence_proxy_async_smem();  // these reads come before the stage's refill
                        } else {
                            ok = false;
                        }
                    } else {
                        key = chunk_tau_key<DT, false>(nullptr, row, t_cbase, t_cend, k);
                    }
                }
                __syncwarp();  // the slot is clear before the consumers see this segment
                if (lane == 0) {
                    tau_key[grp][slot] = key;
                    if (!ok) *reinterpret_cast<volatile int*>(&sfail) = 1;
                    mbar_arrive(&tau_bar[grp][slot]);
                }
            };
            for (int st = 0; st < nst; ++st) {
                const int cbase = (pc.si * P.sps + st) * CHUNK;
                const int cend = min(cbase + CHUNK, P.V);
                if constexpr (BULK) {
                    // lane 0: the stage's previous fill released by every consumer warp (bounded)
                    int go = 0;
                    if (lane == 0 && ok && !*reinterpret_cast<volatile int*>(&sfail)) {
                        // the other group no more than TK_LEAD chunks behind (a bounded wait; the two
                        // groups share the SM, and one left to run ahead would leave the other's chunks
                        // to the end)
                        for (int sp = 0; sp < min(P.wait_limit, TK_LEAD_POLLS) &&
                                         *reinterpret_cast<volatile int*>(&issued[grp ^ 1]) + TK_LEAD <= (int)n; ++sp)
                            __nanosleep(32);
                        if (n < TK_STAGES || mbar_wait(&empty[grp][stg], ph ^ 1u, P.wait_limit)) {
                            bulk_load(ring + (size_t)(grp * TK_STAGES + stg) * NT * TK_NV, row + (size_t)cbase * ES,
                                      (unsigned)(cend - cbase) * ES, &full[grp][stg], pol);
                            *reinterpret_cast<volatile int*>(&issued[grp]) = (int)n + 1;
                            go = 1;
                        } else {
                            *reinterpret_cast<volatile int*>(&sfail) = 1;
                        }
                    }
                    go = __shfl_sync(FULL, go, 0);
                    if (!go) ok = false;
                    if (go && st == 0) {
                        t_stg = stg;
                        t_ph = ph;
                    }
                    if (go) {
                        ++n;
                        if (++stg == TK_STAGES) {
                            stg = 0;
                            ph ^= 1u;
                        }
                    }
                }
                if (st == 0) {
                    t_cbase = cbase;
                    t_cend = cend;
                }
                if (st == 1) publish_tau();
            }
            if (nst == 1) publish_tau();
        }
        if (lane == 0) *reinterpret_cast<volatile int*>(&issued[grp]) = 1 << 30;  // holds the other back no more
        // the last segments: published once every consumer warp is done with them
        for (int j = (m > TK_SLOTS ? m - TK_SLOTS : 0); j < m; ++j) {
            const int slot = j % TK_SLOTS;
            const bool done = __all_sync(FULL, mbar_wait(&done_bar[grp][slot], (unsigned)(j / TK_SLOTS) & 1u, P.wait_limit));
            publish(slot, done);
        }
        // the CTA may not leave while a copy is in flight: wait (bounded) for the last fill of
        // every stage -- no later fill of that stage exists, so its phase is unambiguous
        if constexpr (BULK) {
            if (lane == 0)
                for (long long j = (n > TK_STAGES ? n - TK_STAGES : 0); j < n; ++j)
                    (void)mbar_wait(&full[grp][j % TK_STAGES], (unsigned)(j / TK_STAGES) & 1u, MBAR_SPIN_LIMIT);
        }
        return;
    }

    // ------------------------------------------------------------------ consumer warps
    int stg = 0;          // ring stage of the next chunk
    unsigned ph = 0;      // its fill parity
    int jseg = -1;        // this CTA's segment counter
    bool failed = false;  // a wait ran out: the remaining segments are marked, not read
    SegCursor cc;
    cc.init(TK_GROUPS * blockIdx.x + grp, G0, P.nsegr);
    for (; cc.sg < nsegs; cc.next(G0, P.nsegr)) {
        const int sg = cc.sg;
        ++jseg;
        const int slot = jseg % TK_SLOTS;
        const int nst = min(P.sps, P.CT - cc.si * P.sps);
        const char* row = BULK ? nullptr : spec_row_ptr(P, cc.row_id / P.R, cc.row_id % P.R);
        TopkEntry* slist = P.clist + (size_t)sg * P.cap_s;
        uint4* sdata = P.cdata + (size_t)sg * P.cap_s;
        int seg_bad = 0;             // this warp saw a NaN or +inf in the segment
        float tau_first = NEG_INF;   // the segment's first bound; histogram bins count from its key
        uint32_t key0 = 0;
        for (int st = 0; st < nst; ++st) {
            const int cbase = (cc.si * P.sps + st) * CHUNK;
            const int cend = min(cbase + CHUNK, P.V);
            const bool partial = cbase + CHUNK > cend;

            // ---- the chunk into registers (-inf padding past the row's end)
            uint32_t w[NREG];
            if (!failed && *reinterpret_cast<volatile int*>(&sfail)) failed = true;
            if constexpr (BULK) {
                bool ok = !failed && mbar_wait(&full[grp][stg], ph, P.wait_limit);
                const uint4* sb = ring + (size_t)(grp * TK_STAGES + stg) * NT * TK_NV + ct;
                if (ok && !partial) {
#pragma unroll
                    for (int j = 0; j < TK_NV; ++j) {
                        const uint4 q = lds128(sb + j * NT);
                        w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
                    }
                } else {
                    const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
#pragma unroll
                    for (int j = 0; j < TK_NV; ++j) {
                        uint4 q = make_uint4(pad, pad, pad, pad);
                        if (ok && cbase + (j * NT + ct) * VEC < cend) q = lds128(sb + j * NT);
                        w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
                    }
                }
                // release the stage once every lane has read it; a warp whose wait ran out never
                // releases it (its copy may still land), which stops the producer
                ok = __all_sync(FULL, ok);
                if (ok) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[grp][stg]);
                } else if (!failed) {
                    failed = true;
                    if (lane == 0) *reinterpret_cast<volatile int*>(&sfail) = 1;
                }
                if (++stg == TK_STAGES) {
                    stg = 0;
                    ph ^= 1u;
                }
            } else {
                if constexpr (DT == DT_BF16) {
                    const unsigned short* rp = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
                    for (int j = 0; j < NREG; ++j) {
                        const int e0 = slot_elem<1>(cbase, 2 * j, ct), e1 = slot_elem<1>(cbase, 2 * j + 1, ct);
                        const uint32_t lo = e0 < cend ? __ldg(rp + e0) : 0xff80u;
                        const uint32_t hi = e1 < cend ? __ldg(rp + e1) : 0xff80u;
                        w[j] = lo | (hi << 16);
                    }
                } else {
                    const float* rp = reinterpret_cast<const float*>(row);
#pragma unroll
                    for (int j = 0; j < NREG; ++j) {
                        const int e0 = slot_elem<1>(cbase, j, ct);
                        w[j] = e0 < cend ? __float_as_uint(__ldg(rp + e0)) : 0xff800000u;
                    }
                }
            }

            // ---- group maxima and the thread maximum, NaN-propagating
            uint32_t gm[NG];
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                uint32_t m = w[g * G];
#pragma unroll
                for (int j = 1; j < G; ++j) {
                    if constexpr (DT == DT_BF16) m = bmax2_nan(m, w[g * G + j]);
                    else m = __float_as_uint(fmax_nan(__uint_as_float(m), __uint_as_float(w[g * G + j])));
                }
                gm[g] = m;
            }
            float tm;
            if constexpr (DT == DT_BF16) {
                uint32_t pm = gm[0];
#pragma unroll
                for (int g = 1; g < NG; ++g) pm = bmax2_nan(pm, gm[g]);
                tm = fmax_nan(bf16lo(pm), bf16hi(pm));
            } else {
                tm = __uint_as_float(gm[0]);
#pragma unroll
                for (int g = 1; g < NG; ++g) tm = fmax_nan(tm, __uint_as_float(gm[g]));
            }
            const bool bad_now = __any_sync(FULL, tm != tm || tm == __int_as_float(0x7f800000));

            // ---- a segment's first chunk: tau from the producer (bounded wait); only after this
            // does the warp touch the segment's slot, which the producer has cleared by then
            if (st == 0) {
                if (!failed) {
                    const bool got = __all_sync(FULL, mbar_wait(&tau_bar[grp][slot], (unsigned)(jseg / TK_SLOTS) & 1u, P.wait_limit));
                    if (!got) {
                        failed = true;
                        if (lane == 0) *reinterpret_cast<volatile int*>(&sfail) = 1;
                    }
                }
                if (!failed && k <= NT) {
                    key0 = tau_key[grp][slot];
                    tau_first = key_value(key0);
                }
            }
            if (!failed) {
                if (bad_now && !seg_bad) {
                    seg_bad = 1;
                    if (lane == 0) atomicOr(&sflag[grp][slot], 1);
                }
                float beta = tau_first;
                {
                    const unsigned long long pb = *reinterpret_cast<volatile unsigned long long*>(&pub[grp]);
                    if ((int)(pb >> 32) == sg) beta = fmaxf(beta, key_value((uint32_t)pb));
                }

                // ---- the warps take turns: a tighter bound from the histogram (counts of every
                // warp so far), for the chunks still to come
                if (cw == (st & (WARPS - 1)) && !seg_bad && k <= NT && st + 1 < nst && tau_first != NEG_INF) {
                    const float nb = hist_bound(hist[grp][slot], k, key0);
                    if (lane == 0 && nb > beta)
                        *reinterpret_cast<volatile unsigned long long*>(&pub[grp]) =
                            ((unsigned long long)(unsigned)sg << 32) | okey(nb);
                }

                // ---- this warp's groups whose maximum reaches beta go to the segment's list: the
                // maximum and the first element's index, and the group's 16 raw bytes; the maximum
                // is counted in the histogram
                if (!seg_bad && k <= NT) {
                    // bf16: compare against beta rounded down to bf16, so no element >= beta is missed
                    const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_rd(beta));
                    unsigned pass = 0;
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        bool ge;
                        if constexpr (DT == DT_BF16) ge = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&gm[g]), t2) != 0u;
                        else ge = __uint_as_float(gm[g]) >= beta;
                        pass |= (unsigned)ge << g;
                    }
                    if (partial && pass) {  // groups that start past the row's end hold padding only
#pragma unroll
                        for (int g = 0; g < NG; ++g)
                            if (slot_elem<VEC>(cbase, EPG * g, ct) >= cend) pass &= ~(1u << g);
                    }
                    const int mine = __popc(pass);
                    if (__any_sync(FULL, mine)) {
                        const int incl = warp_incl_scan(mine);
                        int pos = 0;
                        if (lane == 31) pos = atomicAdd(&scount[grp][slot], incl);
                        pos = __shfl_sync(FULL, pos, 31) + incl - mine;
                        int* h = hist[grp][slot];
                        const bool count = tau_first != NEG_INF;
#pragma unroll
                        for (int g = 0; g < NG; ++g) {
                            if (pass & (1u << g)) {
                                TopkEntry en;
                                if constexpr (DT == DT_BF16) en.x = fmaxf(bf16lo(gm[g]), bf16hi(gm[g]));
                                else en.x = __uint_as_float(gm[g]);
                                en.idx = slot_elem<VEC>(cbase, EPG * g, ct);
                                if (pos < P.cap_s) {
                                    slist[pos] = en;
                                    sdata[pos] = make_uint4(w[G * g], w[G * g + 1], w[G * g + 2], w[G * g + 3]);
                                }
                                ++pos;
                                if (count) {
                                    const uint32_t kx = okey(en.x);
                                    if (kx >= key0) atomicAdd(&h[min((int)((kx - key0) >> 16), TK_BINS - 1)], 1);
                                }
                            }
                        }
                    }
                }
            } else if (lane == 0) {
                atomicOr(&sflag[grp][slot], 4);
            }
            // ---- the segment's last chunk: this warp is done with the segment
            if (st + 1 == nst) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&done_bar[grp][slot]);
            }
        }
    }
}

// Kernel 2, one warp per row: exact threshold g from the row's candidate groups (nsegr segment
// lists of kernel 1, up to 1024 groups in all), the kept list (in list order), and the
// normaliser over it.  Each segment's final bound reaches at most g (at least k of the row's
// elements reach it), so only the listed groups whose maximum reaches the largest of them, beta,
// can hold an element >= g; their elements >= beta are the candidates from which g is selected
// exactly.  u holds topk_cand_cap(cap_k) entries, kept cap_k.
template <int DT>
__device__ RowStats topk_row_finish(const SpecParams& P, TopkEntry* u, TopkEntry* kept, int row_id)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    RowStats st;
    st.M = NEG_INF; st.MC = NEG_INF; st.S = 0.0; st.thr = NEG_INF;
    st.status = ROW_OK; st.klist_n = -1; st.dense = 0;
    st.lse = __int_as_float(0x7fc00000);
    st.invS = 0.f;
    st.lx_hi = __int_as_float(0x7fc00000);
    st.lx_lo = 0.f;
    const int nl = P.nsegr;  // lists of the row, <= 4
    const size_t sg0 = (size_t)row_id * nl;
    // the token this row scores (target row i and draft row i score draft token i; the last target
    // row scores none) and its logit, fetched now so that they arrive while the lists are read
    const int b = row_id / P.R, r = row_id - b * P.R, g = P.gamma;
    const int pos = (r < g) ? r : (r > g) ? r - g - 1 : -1;
    const int tok = (pos >= 0) ? __ldg(P.tokens + (size_t)b * g + pos) : -1;
    const bool tok_ok = tok >= 0 && tok < P.V;
    const float xtok = tok_ok ? load_logit(spec_row_ptr(P, b, r), DT, tok) : 0.f;
    pdl_trigger();
    pdl_wait();  // the candidate lists of the streaming kernel

    int n = 0;
    float bd = NEG_INF;
    if (lane < nl) {
        n = __ldcg(P.ccount + sg0 + lane);
        bd = __ldcg(P.cbound + sg0 + lane);
    }
    int flag = 0;
    if (n == TK_NONFINITE) flag |= 1;
    else if (n == TK_TIMEOUT) flag |= 4;
    else if (n < 0) flag |= 2;
    flag = (int)__reduce_or_sync(FULL, (unsigned)flag);
    if (flag & 4) { st.status = ROW_TIMEOUT; return st; }
    if (flag & 1) { st.status = ROW_NONFINITE; return st; }
    if (flag & 2) { st.dense = 1; return st; }
    n = max(0, min(n, P.cap_s));
    const int incl = warp_incl_scan(n);
    const int total = __shfl_sync(FULL, incl, 31);
    const float beta = warp_max(bd);
    // list starts in the packed order (lists 1..3; nl <= 4)
    const int ls1 = __shfl_sync(FULL, incl, 0), ls2 = __shfl_sync(FULL, incl, 1), ls3 = __shfl_sync(FULL, incl, 2);

    // the groups whose maximum reaches beta: (first element's index, slot), compacted into kept;
    // entries in batches of 6 per lane, every load of a batch issued before any is used
    const TopkEntry* lists = P.clist + sg0 * P.cap_s;
    const uint4* gdata = P.cdata + sg0 * P.cap_s;
    constexpr int EB = 6;
    int ng = 0;
    for (int p0 = 0; p0 < total; p0 += 32 * EB) {
        TopkEntry e[EB];
        int slot[EB];
#pragma unroll
        for (int t = 0; t < EB; ++t) {
            const int p = p0 + 32 * t + lane;
            e[t].x = NEG_INF;
            e[t].idx = 0;
            slot[t] = -1;
            if (p < total) {
                const int l = (nl > 1 && p >= ls1) + (nl > 2 && p >= ls2) + (nl > 3 && p >= ls3);
                const int start = (l == 0) ? 0 : (l == 1) ? ls1 : (l == 2) ? ls2 : ls3;
                slot[t] = l * P.cap_s + (p - start);
                e[t] = ld_entry(lists + slot[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < EB; ++t) {
            if (p0 + 32 * t >= total) break;  // the same for every lane
            const bool keep = slot[t] >= 0 && e[t].x >= beta;
            const unsigned bal = __ballot_sync(FULL, keep);
            const int q = ng + __popc(bal & ((1u << lane) - 1u));
            if (keep && q < P.cap_k) {
                TopkEntry ge;
                ge.x = __int_as_float(slot[t]);
                ge.idx = e[t].idx;
                kept[q] = ge;
            }
            ng += __popc(bal);
        }
    }
    __syncwarp();
    if (ng > P.cap_k) { st.dense = 1; return st; }
    // their elements >= beta inside the row are the candidates, packed into u (32 x GB groups at a
    // time, every load of a batch issued before any is used)
    constexpr int EPG = (DT == DT_BF16) ? 8 : 4;  // elements per group (one 16-byte vector)
    const int estride = (P.vec > 1) ? 1 : NT;     // index step between a group's elements
    const int cand = topk_cand_cap(P.cap_k);
    const uint32_t bkey = okey(beta);
    int ne = 0;
    constexpr int GB = 4;
    for (int r0 = 0; r0 < ng; r0 += 32 * GB) {
        uint4 d[GB];
        int base[GB];
#pragma unroll
        for (int t = 0; t < GB; ++t) {
            const int i = r0 + 32 * t + lane;
            base[t] = P.V;  // nothing inside the row
            if (i < ng) {
                const TopkEntry ge = kept[i];
                d[t] = __ldcg(gdata + __float_as_int(ge.x));
                base[t] = ge.idx;
            }
        }
#pragma unroll
        for (int t = 0; t < GB; ++t) {
            if (r0 + 32 * t >= ng) break;  // the same for every lane
            const uint32_t wd[4] = {d[t].x, d[t].y, d[t].z, d[t].w};
            float xe[EPG];
            unsigned m = 0;
#pragma unroll
            for (int e = 0; e < EPG; ++e) {
                if constexpr (DT == DT_BF16) xe[e] = (e & 1) ? bf16hi(wd[e >> 1]) : bf16lo(wd[e >> 1]);
                else xe[e] = __uint_as_float(wd[e]);
                if (base[t] + e * estride < P.V && okey(xe[e]) >= bkey) m |= 1u << e;
            }
            const int c = __popc(m);
            const int ci = warp_incl_scan(c);
            int p = ne + ci - c;
            ne += __shfl_sync(FULL, ci, 31);
#pragma unroll
            for (int e = 0; e < EPG; ++e) {
                if (m & (1u << e)) {
                    if (p < cand) {
                        TopkEntry en;
                        en.x = xe[e];
                        en.idx = base[t] + e * estride;
                        u[p] = en;
                    }
                    ++p;
                }
            }
        }
    }
    __syncwarp();
    if (ne > cand) { st.dense = 1; return st; }
    // g: the exact k-th largest candidate (kept serves as the histogram)
    const int k = P.top_k;
    uint32_t gkey = okey(NEG_INF);
    if (ne >= k)
        gkey = warp_kth_key_hist<DT>(ne, k, reinterpret_cast<int*>(kept),
                                     [&](int i) { return okey(u[i].x); });
    __syncwarp();
    // the candidates >= g, in candidate order
    int nk = 0;
    for (int i0 = 0; i0 < ne; i0 += 32) {
        const int i = i0 + lane;
        TopkEntry en;
        en.x = NEG_INF;
        en.idx = 0;
        if (i < ne) en = u[i];
        const bool keep = i < ne && okey(en.x) >= gkey;
        const unsigned bal = __ballot_sync(FULL, keep);
        const int q = nk + __popc(bal & ((1u << lane) - 1u));
        if (keep && q < P.cap_k) kept[q] = en;
        nk += __popc(bal);
    }
    __syncwarp();
    if (nk > P.cap_k) { st.dense = 1; return st; }
    // the normaliser over the kept entries: their maximum, and their mass in fixed point (an
    // integer sum, exact whatever the order the lists delivered them in); the kept list is stored
    // in that order and sorted by index only where a draw uses it
    float mx = NEG_INF;
    for (int i = lane; i < nk; i += 32) mx = fmaxf(mx, kept[i].x);
    const float M = warp_max(mx);
    const float MC = __fmul_rn(M, P.c);
    unsigned long long fs = 0ull;
    if (M != NEG_INF)
        for (int i = lane; i < nk; i += 32) fs += fixed_mass(ex2(fmaf(kept[i].x, P.c, -MC)));
    const DFloat S = fixed_to_df(warp_sum(fs));
    TopkEntry* kl = P.klist + (size_t)row_id * P.cap_k;
    for (int i = lane; i < nk; i += 32) kl[i] = kept[i];
    st.M = M;
    st.MC = MC;
    st.S = (double)S.hi;
    st.thr = key_value(gkey);
    st.klist_n = nk;
    st.status = (M != NEG_INF && isfinite(M)) ? ROW_OK : ROW_NONFINITE;
    if (st.status == ROW_OK && lane == 0)  // only lane 0's RowStats is stored
        row_norm(st, M, MC, S, P, tok_ok, xtok, st.thr);
    return st;
}

// Kernel 2: one CTA per request, one warp per row (nw = min(R, FIN_MAX_WARPS) warps, rows w, w +
// nw, ...): each warp finishes its row into shared memory; after one CTA barrier warp 0 runs the
// acceptance scan over them and draws from the kept list of the p row.  A request with a dense row
// is completed by the whole CTA with full-row passes instead.
template <int DT>
__device__ __noinline__ void topk_dense_request(const SpecParams& P, int b);

constexpr int FIN_MAX_WARPS = 16;
constexpr size_t FIN_MAX_SMEM = 200 * 1024;  // dynamic shared memory of one finish CTA, at most
template <int DT>
__global__ void __launch_bounds__(FIN_MAX_WARPS * 32, 2) topk_finish_kernel(SpecParams P)
{
    extern __shared__ __align__(16) TopkEntry fin[];  // per warp: u[cand], kept[cap_k]
    __shared__ RowStats srs[32];
    __shared__ int sdense;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int b = blockIdx.x, R = P.R;
    const int cand = topk_cand_cap(P.cap_k);
    TopkEntry* u = fin + (size_t)warp * (cand + P.cap_k);
    TopkEntry* kept = u + cand;
    if (tid == 0) sdense = 0;
    __syncthreads();
    for (int r = warp; r < R; r += nw) {
        const RowStats st = topk_row_finish<DT>(P, u, kept, b * R + r);
        if (lane == 0) {
            P.rstats[(size_t)b * R + r] = st;
            if (r < 32) srs[r] = st;
            else __threadfence();  // read back from global memory below
            if (st.dense) atomicAdd(&sdense, 1);
        }
        __syncwarp();  // u and kept serve the next row
    }
    __syncthreads();
    if (sdense > 0) {  // the whole CTA finishes the request exactly (rare)
        topk_dense_request<DT>(P, b);
        return;
    }
    if (warp != 0) return;
    Plan pl;
    int nk;
    if (R <= 32) {
        RowStats rs = blank_rowstats();
        if (lane < R) rs = srs[lane];
        pl = plan_from_lanes(P, b, rs);
        nk = __shfl_sync(0xffffffffu, rs.klist_n, pl.rp);
    } else {
        pl = compute_plan_warp<DT, true>(P, b, true);
        nk = __ldcg(&P.rstats[(size_t)b * R + pl.rp].klist_n);
    }
    topk_request_draw<DT>(P, pl, nk, u, b);
}

// ---------------------------------------------------------------- exact fallback for dense rows

template <int DT>
__device__ __forceinline__ double topk_residual_at(const char* rowp, const char* rowq, long long v,
                                                   const Plan& pl, float c)
{
    const float xp = load_logit(rowp, DT, v);
    float pp = (xp >= pl.thrp) ? __fmul_rn(ex2(fmaf(xp, c, -pl.MCp)), pl.invSp) : 0.f;
    if (!rowq) return (double)pp;
    const float xq = load_logit(rowq, DT, v);
    const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, c, -pl.MCq)), pl.invSq) : 0.f;
    return (double)fmaxf(__fsub_rn(pp, qq), 0.f);
}

// Block-wide reductions over the CTA's blockDim.x threads (a whole number of warps, at most 32):
// warp partials in shared memory, combined in warp order.  Every thread receives the result.
template <class T, class Op>
__device__ __forceinline__ T cta_reduce(T v, T* sh /* >= 32 */, Op op)
{
    const int nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    T r = sh[0];
    for (int w = 1; w < nw; ++w) r = op(r, sh[w]);
    return r;
}

// sum over the CTA: fp32 within warps, fp64 across warps in warp order
__device__ __forceinline__ double cta_sum_f32(float v, double* sh /* >= 32 */)
{
    const int nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = (double)v;
    __syncthreads();
    double r = 0.0;
    for (int w = 0; w < nw; ++w) r += sh[w];
    return r;
}

// exclusive prefix sum in fp64 over the CTA (thread order); the total goes to *total
__device__ __forceinline__ double cta_excl_scan_f64(double v, double* sh, double* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const double incl = warp_incl_scan(v);
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    double before = 0.0, tot = 0.0;
    for (int w = 0; w < nw; ++w) {
        if (w < warp) before += sh[w];
        tot += sh[w];
    }
    *total = tot;
    return before + (incl - v);
}

// The exact fallback for a request with a dense row (candidates that overflowed the lists: mass
// ties, k > NT, ...), run by the whole finish CTA: each dense row's threshold by a bitwise search
// over full-row counts and its normaliser by full-row passes; then the acceptance scan and the
// correction / bonus draw by two passes of the residual over V (fp64 sums, tile by tile).
template <int DT>
__device__ __noinline__ void topk_dense_request(const SpecParams& P, int b)
{
    __shared__ int sh_i[32];
    __shared__ float sh_f[32];
    __shared__ double sh_d[32];
    __shared__ int sh_tok;
    __shared__ Plan sh_plan;
    const int tid = threadIdx.x, nth = blockDim.x;
    const auto add_i = [](int x, int y) { return x + y; };
    const auto add_d = [](double x, double y) { return x + y; };
    const auto max_f = [](float x, float y) { return fmaxf(x, y); };
    const int V = P.V, k = P.top_k;
    for (int r = 0; r < P.R; ++r) {
        const int row_id = b * P.R + r;
        if (!__ldcg(&P.rstats[row_id].dense)) continue;  // the same for every thread
        const char* row = spec_row_ptr(P, b, r);
        // exact k-th largest key by bitwise search over full-row counts
        uint32_t prefix = 0;
        constexpr int lo = (DT == DT_BF16) ? 16 : 0;
        for (int bit = 31; bit >= lo; --bit) {
            const uint32_t want = prefix | (1u << bit);
            int cnt = 0;
            for (int v = tid; v < V; v += nth) cnt += okey(load_logit(row, DT, v)) >= want;
            if (cta_reduce(cnt, sh_i, add_i) >= k) prefix = want;
        }
        if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
        const float g = key_value(prefix);
        float mx = NEG_INF;
        for (int v = tid; v < V; v += nth) {
            const float x = load_logit(row, DT, v);
            if (x >= g) mx = fmaxf(mx, x);
        }
        const float M = cta_reduce(mx, sh_f, max_f);
        const float MC = __fmul_rn(M, P.c);
        float s = 0.f;
        if (M != NEG_INF)
            for (int v = tid; v < V; v += nth) {
                const float x = load_logit(row, DT, v);
                if (x >= g) s += ex2(fmaf(x, P.c, -MC));
            }
        const double S = cta_sum_f32(s, sh_d);
        if (tid == 0) {
            RowStats st = blank_rowstats();
            st.M = M; st.MC = MC; st.S = S; st.thr = g;
            st.status = (M != NEG_INF && isfinite(M) && S > 0.0) ? ROW_OK : ROW_NONFINITE;
            st.klist_n = -1;
            st.dense = 1;
            P.rstats[row_id] = st;
        }
        __syncthreads();
    }
    if (tid < 32) {
        const Plan p0 = compute_plan_warp<DT>(P, b, true);
        if (tid == 0) sh_plan = p0;
    }
    __syncthreads();
    const Plan pl = sh_plan;
    if (pl.status != ROW_OK) {
        if (tid < 32) emit_spec_n(P, b, pl.status, 0, -1, tid, 32);
        return;
    }
    const char* rowp = spec_row_ptr(P, b, pl.rp);
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    // pass 1: total residual mass, tile by tile in index order (fp64)
    double Z = 0.0;
    for (int t0 = 0; t0 < V; t0 += nth) {
        const int v = t0 + tid;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        Z += cta_reduce(rv, sh_d, add_d);
    }
    if (!(Z > 0.0) || !isfinite(Z)) {
        if (tid < 32) emit_spec_n(P, b, ROW_DEGENERATE, 0, -1, tid, 32);
        return;
    }
    // pass 2: the tile where the running mass passes u*Z, then the element inside it
    const double t = pl.u * Z;
    double run = 0.0;
    int tok = -1;
    for (int t0 = 0; t0 < V; t0 += nth) {
        const int v = t0 + tid;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        const double ts = cta_reduce(rv, sh_d, add_d);
        if (t < run + ts) {  // uniform across the CTA
            double tot;
            const double excl = cta_excl_scan_f64(rv, sh_d, &tot);
            if (tid == 0) sh_tok = 0x7fffffff;
            __syncthreads();
            if (rv > 0.0 && t < run + excl + rv) atomicMin(&sh_tok, v);
            __syncthreads();
            tok = sh_tok;
            if (tok == 0x7fffffff) {  // rounding: last positive entry of the tile
                __syncthreads();
                if (tid == 0) sh_tok = -1;
                __syncthreads();
                if (rv > 0.0) atomicMax(&sh_tok, v);
                __syncthreads();
                tok = sh_tok;
            }
            break;
        }
        run += ts;
    }
    if (tok < 0) {  // rounding ran past the end: last token with positive mass
        __syncthreads();
        if (tid == 0) sh_tok = -1;
        __syncthreads();
        for (int v = tid; v < V; v += nth)
            if (topk_residual_at<DT>(rowp, rowq, v, pl, P.c) > 0.0) atomicMax(&sh_tok, v);
        __syncthreads();
        tok = sh_tok;
    }
    if (tid < 32) emit_spec_n(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok, tid, 32);
}

template <int DT>
static void launch_topk(const SpecParams& P, int sms, cudaStream_t st)
{
    // one CTA per SM at most, TK_GROUPS segment sequences per CTA
    const long long nsegs = ((long long)P.B * P.R * P.nsegr + TK_GROUPS - 1) / TK_GROUPS;
    mark_kernel_start(st);
    if (P.vec > 1) {
        constexpr auto K1 = topk_stream_kernel<DT, true>;
        K1<<<cta_grid<K1>(nsegs, sms, TK_SMEM, TK_THREADS), TK_THREADS, TK_SMEM, st>>>(P);
    } else {
        constexpr auto K1 = topk_stream_kernel<DT, false>;
        K1<<<cta_grid<K1>(nsegs, sms, 0, TK_THREADS), TK_THREADS, 0, st>>>(P);
    }
    mark_kernel_stop(st);
    // one warp per row, as many as the shared memory of one CTA holds (the rest loop over rows)
    const size_t per_warp = (size_t)(topk_cand_cap(P.cap_k) + P.cap_k) * sizeof(TopkEntry);
    const int fw = std::max(1, std::min(std::min(P.R, FIN_MAX_WARPS), (int)(FIN_MAX_SMEM / per_warp)));
    const size_t fsm = (size_t)fw * per_warp;
    set_smem_limit<topk_finish_kernel<DT>>(fsm);
    launch_dependent(topk_finish_kernel<DT>, (unsigned)P.B, (unsigned)(32 * fw), fsm, st, P);
}

cudaError_t launch_topk_path(const SpecParams& P, int sms, cudaStream_t st)
{
    if (P.dtype == DT_BF16) launch_topk<DT_BF16>(P, sms, st);
    else launch_topk<DT_F32>(P, sms, st);
    return cudaGetLastError();
}

}  // namespace sv
