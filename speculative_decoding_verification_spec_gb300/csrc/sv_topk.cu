// sv_topk.cu -- exact speculative sampling with a top-k processor on p and q.
//
// M7.1 section 0x03D: truncation keeps the method exact when p and q are the truncated,
// renormalised distributions and q is the one that sampled the draft.  A row keeps every token
// whose stored logit is >= the row's k-th largest stored logit (counted with multiplicity), so ties
// at the threshold are all kept.
//
// Kernel 1 (topk_stream_kernel) streams every logit row once.  Rows are cut into 32 KB chunks and
// runs of chunks (segments, at most 4 per row); persistent CTAs take segments round-robin and, for
// 16-byte aligned rows, fetch their chunks with bulk copies (TMA engine) into a ring of TK_STAGES
// shared-memory stages, so the next chunks are in flight while one is filtered.  Each thread holds
// its 64 (bf16) or 32 (fp32) elements of a chunk in registers.  The k-th largest of the NT
// per-thread maxima (NT disjoint groups, so at least k chunk elements are >= it) bounds the chunk's
// k-th largest value from below; every warp selects it from shared memory by itself, so no warp
// waits for another.  With the bound carried over from the segment's earlier chunks it forms beta,
// and only elements >= beta -- a few dozen per chunk at k = 50 -- join the segment's candidate set
// in shared memory.  When the set grows large, and at the end of the segment, one warp cuts it to
// the entries >= its exact k-th largest value, which becomes the new bound; the segment's list is
// what remains.  Every bound is <= the row's k-th largest value g, so the lists hold every
// element >= g.
//
// Kernel 2 (topk_finish_kernel), one CTA per request: one warp per row selects g exactly from the
// union of the row's segment lists, keeps the entries >= g sorted by index and forms the
// normaliser (M, S).  Then one warp runs the acceptance scan and draws the correction or bonus
// token directly from the kept list of the p row: the residual vanishes outside K_p, so no second
// pass over V is needed.
//
// Rows whose candidates overflow the capacities (massive ties, k > NT, ...) are marked dense and
// finished exactly by kernel 3 (topk_dense_kernel) with full-row passes.
#include <cuda_bf16.h>

#include "sv_plan.cuh"

namespace sv {

constexpr int TK_CHUNK_BYTES = 32768;                 // bytes of one row per chunk
constexpr int TK_NREG = TK_CHUNK_BYTES / (NT * 4);    // 32-bit words per thread (32)
constexpr int TK_NV = TK_NREG / 4;                    // 16-byte vectors per thread (8)
constexpr int TK_STAGES = 3;                          // bulk-copy ring depth
constexpr int TK_SMEM = TK_STAGES * TK_CHUNK_BYTES;   // dynamic shared memory of kernel 1
// per-chunk candidate count codes
constexpr int TK_OVERFLOW = -1, TK_NONFINITE = -2, TK_TIMEOUT = -3;

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

__device__ __forceinline__ float fmax_nan_f(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
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

// w[base + j] for a run-time j in [0, 8) and a compile-time base, by a select tree (no local memory)
template <int N>
__device__ __forceinline__ uint32_t select8(const uint32_t (&w)[N], int base, int j)
{
    const uint32_t a0 = (j & 1) ? w[base + 1] : w[base];
    const uint32_t a1 = (j & 1) ? w[base + 3] : w[base + 2];
    const uint32_t a2 = (j & 1) ? w[base + 5] : w[base + 4];
    const uint32_t a3 = (j & 1) ? w[base + 7] : w[base + 6];
    const uint32_t c0 = (j & 2) ? a1 : a0;
    const uint32_t c1 = (j & 2) ? a3 : a2;
    return (j & 4) ? c1 : c0;
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

// One warp: acceptance scan of request b and the correction / bonus draw from the kept list of
// the p row (index order); the residual is zero outside K_p.
template <int DT>
__device__ void topk_request_epilogue(const SpecParams& P, double* rr, int b)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const Plan pl = compute_plan_warp<DT>(P, b, true);
    if (pl.status != ROW_OK) {
        emit_spec_warp(P, b, pl.status, 0, -1);
        return;
    }
    const RowStats sp = ld_rowstats(P.rstats + (size_t)b * P.R + pl.rp);
    const int nk = sp.klist_n;
    const TopkEntry* kl = P.klist + ((size_t)b * P.R + pl.rp) * P.cap_k;
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    // each lane owns a contiguous block of the kept list
    const int per = (nk + 31) / 32;
    const int i0 = min(lane * per, nk), i1 = min(i0 + per, nk);
    double mine = 0.0;
    for (int i = i0; i < i1; ++i) {
        const float xp = __ldcg(&kl[i].x);
        const int v = __ldcg(&kl[i].idx);
        const float pp = __fmul_rn(ex2(fmaf(xp, P.c, -pl.MCp)), pl.invSp);
        float res = pp;
        if (rowq) {
            const float xq = load_logit(rowq, DT, v);
            const float qq = (xq >= pl.thrq) ? __fmul_rn(ex2(fmaf(xq, P.c, -pl.MCq)), pl.invSq) : 0.f;
            res = fmaxf(__fsub_rn(pp, qq), 0.f);
        }
        rr[i] = (double)res;
        mine += (double)res;
    }
    const double incl = warp_incl_scan(mine);
    const double Z = __shfl_sync(FULL, incl, 31);
    int tok = -1;
    if (Z > 0.0 && isfinite(Z)) {
        const double t = pl.u * Z, excl = incl - mine;
        unsigned own = __ballot_sync(FULL, mine > 0.0 && t < excl + mine);
        if (!own) {
            const unsigned pos = __ballot_sync(FULL, mine > 0.0);
            own = pos ? (1u << (31 - __clz(pos))) : 0u;
        }
        if (own) {
            const int owner = __ffs(own) - 1;
            if (lane == owner) {
                double run = excl;
                int lastpos = -1;
                for (int i = i0; i < i1; ++i) {
                    if (rr[i] > 0.0) lastpos = i;
                    run += rr[i];
                    if (t < run && rr[i] > 0.0) { tok = __ldcg(&kl[i].idx); break; }
                }
                if (tok < 0 && lastpos >= 0) tok = __ldcg(&kl[lastpos].idx);
            }
            tok = __shfl_sync(FULL, tok, owner);
        }
    }
    emit_spec_warp(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}


// element index (within the row) of register slot s of this thread: vector j = s / VEC, element
// e = s % VEC of it; vectors of a thread are NT apart
template <int VEC>
__device__ __forceinline__ int slot_elem(int cbase, int s)
{
    if constexpr (VEC == 1) return cbase + s * NT + (int)threadIdx.x;
    else return cbase + ((s / VEC) * NT + (int)threadIdx.x) * VEC + (s % VEC);
}

// Bits of a group's passing-slot mask (as built in topk_stream_kernel) whose elements lie before
// cend.  Group g holds registers 8g..8g+7 of the thread: for bf16 bit j is the low half of register
// 8g+j and bit 16+j its high half; for fp32 bit j is register 8g+j.
template <int DT, int VEC>
__device__ __forceinline__ uint32_t valid_bits(int cbase, int cend, int g)
{
    uint32_t m = 0;
    constexpr int PER = (DT == DT_BF16) ? 2 : 1;  // elements per register
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int h = 0; h < PER; ++h)
            if (slot_elem<VEC>(cbase, PER * (8 * g + j) + h) < cend) m |= 1u << (j + 16 * h);
    return m;
}

// k-th largest key (as warp_kth_key) of e[0..n), n <= 32 * KPL, with the keys held in registers.
template <int DT, int KPL>
__device__ uint32_t warp_kth_key_regs(const TopkEntry* e, int n, int k)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[KPL];
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
        const int i = lane + 32 * j;
        key[j] = i < n ? okey(e[i].x) : 0u;  // 0: below every key a value can have
    }
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        unsigned cnt = 0;
#pragma unroll
        for (int j = 0; j < KPL; ++j) cnt += key[j] >= want;
        if ((int)__reduce_add_sync(0xffffffffu, cnt) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    return prefix;
}

constexpr int TK_CAPC = 1024;  // on-chip candidate set of the segment being streamed

// Kernel 1.  BULK: rows of 16-byte vectors fetched by bulk copies into the stage ring; otherwise
// element loads straight into registers.  A CTA takes segments (runs of up to P.sps chunks of one
// row) round-robin and streams them chunk by chunk.
template <int DT, bool BULK>
__global__ void __launch_bounds__(NT, 2) topk_stream_kernel(SpecParams P)
{
    constexpr int NREG = TK_NREG;
    constexpr int EPT = (DT == DT_BF16) ? 2 * NREG : NREG;  // elements per thread
    constexpr int CHUNK = NT * EPT;                          // elements per chunk
    constexpr int VEC = BULK ? ((DT == DT_BF16) ? 8 : 4) : 1;
    constexpr int ES = (DT == DT_BF16) ? 2 : 4;
    constexpr int G = 8, NG = NREG / G;
    static_assert(NREG % G == 0, "register groups");
    extern __shared__ __align__(128) uint4 ring[];  // BULK: TK_STAGES x (NT * TK_NV) vectors
    __shared__ float tmax[NT];
    __shared__ TopkEntry cset[TK_CAPC];
    __shared__ int ncset;     // candidates in cset (may exceed TK_CAPC: then the segment overflowed)
    __shared__ float sbeta;   // running lower bound of the segment's k-th largest value
    __shared__ int sover;     // the segment's candidates overflowed
    __shared__ int sbad[2];   // a NaN or +inf was seen in the chunk (double-buffered by parity)
    __shared__ __align__(8) uint64_t full[TK_STAGES];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const long long nsegs = (long long)P.B * P.R * P.nsegr;
    const long long G0 = gridDim.x;
    const int k = P.top_k;
    const uint64_t pol = policy_evict_first();

    auto seg_stages = [&](long long sg) -> int {
        const int si = (int)(sg % P.nsegr);
        return min(P.sps, P.CT - si * P.sps);
    };
    // row and element range of chunk `st` of segment `sg`
    auto chunk_of = [&](long long sg, int st, int& row_id, int& cbase, int& cend) {
        row_id = (int)(sg / P.nsegr);
        const int c = (int)(sg % P.nsegr) * P.sps + st;
        cbase = c * CHUNK;
        cend = min(cbase + CHUNK, P.V);
    };

    // producer cursor (thread 0): the next (segment, chunk) to fetch, in this CTA's consumption order
    long long pseg = blockIdx.x;
    int pst = 0;
    long long nissued = 0;
    auto issue_next = [&](int s) {
        if (pseg >= nsegs) return;
        int row_id, cbase, cend;
        chunk_of(pseg, pst, row_id, cbase, cend);
        const char* src = spec_row_ptr(P, row_id / P.R, row_id % P.R) + (size_t)cbase * ES;
        bulk_load(ring + (size_t)s * NT * TK_NV, src, (unsigned)(cend - cbase) * ES, &full[s], pol);
        ++nissued;
        if (++pst == seg_stages(pseg)) {
            pst = 0;
            pseg += G0;
        }
    };

    if (tid == 0) {
        ncset = 0;
        sbeta = NEG_INF;
        sover = 0;
        sbad[0] = 0;
        sbad[1] = 0;
        if constexpr (BULK) {
            for (int s = 0; s < TK_STAGES; ++s) mbar_init(&full[s], 1);
            fence_mbar_init();
            for (int s = 0; s < TK_STAGES; ++s) issue_next(s);
        }
    }
    __syncthreads();

    bool failed = false;  // a bulk-copy wait ran out: the remaining segments are reported, not read
    long long fail_it = 0;
    long long it = 0;
    for (long long sg = blockIdx.x; sg < nsegs; sg += G0) {
        const int nst = seg_stages(sg);
        int seg_bad = 0;
        for (int st = 0; st < nst; ++st, ++it) {
            int row_id, cbase, cend;
            chunk_of(sg, st, row_id, cbase, cend);
            const bool partial = cbase + CHUNK > cend;

            // ---- the chunk into registers (-inf padding past the row's end)
            uint32_t w[NREG];
            bool ok = !failed;
            if constexpr (BULK) {
                const int s = (int)(it % TK_STAGES);
                if (ok) ok = mbar_wait(&full[s], (unsigned)(it / TK_STAGES) & 1u);
                const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
                const uint4* sb = ring + (size_t)s * NT * TK_NV;
#pragma unroll
                for (int j = 0; j < TK_NV; ++j) {
                    uint4 q = make_uint4(pad, pad, pad, pad);
                    if (ok && (!partial || cbase + (j * NT + tid) * VEC < cend)) q = lds128(sb + j * NT + tid);
                    w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
                }
            } else {
                const char* row = spec_row_ptr(P, row_id / P.R, row_id % P.R);
                if constexpr (DT == DT_BF16) {
                    const unsigned short* rp = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
                    for (int j = 0; j < NREG; ++j) {
                        const int e0 = slot_elem<1>(cbase, 2 * j), e1 = slot_elem<1>(cbase, 2 * j + 1);
                        const uint32_t lo = e0 < cend ? __ldg(rp + e0) : 0xff80u;
                        const uint32_t hi = e1 < cend ? __ldg(rp + e1) : 0xff80u;
                        w[j] = lo | (hi << 16);
                    }
                } else {
                    const float* rp = reinterpret_cast<const float*>(row);
#pragma unroll
                    for (int j = 0; j < NREG; ++j) {
                        const int e0 = slot_elem<1>(cbase, j);
                        w[j] = e0 < cend ? __float_as_uint(__ldg(rp + e0)) : 0xff800000u;
                    }
                }
            }

            // ---- group maxima (G registers each) and the thread maximum, NaN-propagating
            uint32_t gm[NG];
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                uint32_t m = w[g * G];
#pragma unroll
                for (int j = 1; j < G; ++j) {
                    if constexpr (DT == DT_BF16) m = bmax2_nan(m, w[g * G + j]);
                    else m = __float_as_uint(fmax_nan_f(__uint_as_float(m), __uint_as_float(w[g * G + j])));
                }
                gm[g] = m;
            }
            float tm;
            if constexpr (DT == DT_BF16) {
                uint32_t pm = gm[0];
#pragma unroll
                for (int g = 1; g < NG; ++g) pm = bmax2_nan(pm, gm[g]);
                tm = fmax_nan_f(bf16lo(pm), bf16hi(pm));
            } else {
                tm = __uint_as_float(gm[0]);
#pragma unroll
                for (int g = 1; g < NG; ++g) tm = fmax_nan_f(tm, __uint_as_float(gm[g]));
            }
            tmax[tid] = tm;
            if (tm != tm || tm == __int_as_float(0x7f800000)) sbad[it & 1] = 1;
            if (tid == 0) sbad[(it + 1) & 1] = 0;  // the next chunk's flag
            // every thread has read its part of the stage, every thread maximum is published, and
            // warp 0 has finished with the previous chunk's candidate set
            const int anyfail = __syncthreads_or(!ok);
            if (anyfail && !failed) {
                failed = true;
                fail_it = it;
            }
            if constexpr (BULK) {
                if (tid == 0 && !failed) {
                    fence_proxy_async_smem();
                    issue_next((int)(it % TK_STAGES));
                }
            }
            if (failed) {
                if (tid == 0 && st + 1 == nst) P.ccount[sg] = TK_TIMEOUT;
                continue;
            }

            // ---- the bound for this chunk.  On a segment's first chunk (or while no finite bound
            // exists) every warp selects tau = the k-th largest thread maximum (valid for k <= NT)
            // by itself; later chunks reuse the segment's running bound, which is already tighter.
            const int bad = sbad[it & 1];
            seg_bad |= bad;
            float beta = (st == 0) ? NEG_INF : sbeta;
            if (!bad && k <= NT && beta == NEG_INF) {
                uint32_t keys[NT / 32];
#pragma unroll
                for (int i = 0; i < NT / 32; ++i) keys[i] = okey(tmax[lane + 32 * i]);
                uint32_t prefix = 0;
                constexpr int lo = (DT == DT_BF16) ? 16 : 0;
                for (int bit = 31; bit >= lo; --bit) {
                    const uint32_t want = prefix | (1u << bit);
                    unsigned cnt = 0;
#pragma unroll
                    for (int i = 0; i < NT / 32; ++i) cnt += keys[i] >= want;
                    if ((int)__reduce_add_sync(FULL, cnt) >= k) prefix = want;
                }
                if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
                // tau and the carried bound are both <= the segment's k-th largest value, hence
                // <= the row's
                beta = key_value(prefix);
            }

            // ---- every element >= beta joins the candidate set.  A group whose maximum reaches
            // beta yields a bitmask of its passing slots (slots past the row's end masked off);
            // each warp reserves room for all of its candidates with one shared-memory atomic and
            // every thread then writes its own at consecutive positions.
            if (!seg_bad && !sover && k <= NT) {
                uint32_t bits[NG];
                int mine = 0;
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    uint32_t bt = 0;
                    if constexpr (DT == DT_BF16) {
                        const __nv_bfloat162 t2 = __floats2bfloat162_rn(beta, beta);
                        if (__hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&gm[g]), t2)) {
#pragma unroll
                            for (int j = 0; j < G; ++j) {
                                const uint32_t wd = w[g * G + j];
                                bt |= (__hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&wd), t2) & 0x00010001u) << j;
                            }
                        }
                    } else {
                        if (__uint_as_float(gm[g]) >= beta) {
#pragma unroll
                            for (int j = 0; j < G; ++j) bt |= (uint32_t)(__uint_as_float(w[g * G + j]) >= beta) << j;
                        }
                    }
                    if (partial && bt) bt &= valid_bits<DT, VEC>(cbase, cend, g);
                    bits[g] = bt;
                    mine += __popc(bt);
                }
                const int incl = warp_incl_scan(mine);
                const int wtot = __shfl_sync(FULL, incl, 31);
                if (wtot > 0) {
                    int base = 0;
                    if (lane == 31) base = atomicAdd(&ncset, wtot);
                    int pos = __shfl_sync(FULL, base, 31) + incl - mine;
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        uint32_t bt = bits[g];
                        while (bt) {
                            const int bp = __ffs(bt) - 1;
                            bt &= bt - 1;
                            const int j = bp & 15, half = bp >> 4;  // register j of the group, bf16 half
                            const uint32_t wd = select8(w, g * G, j);
                            TopkEntry en;
                            if constexpr (DT == DT_BF16) {
                                en.x = half ? bf16hi(wd) : bf16lo(wd);
                                en.idx = slot_elem<VEC>(cbase, 2 * (g * G + j) + half);
                            } else {
                                en.x = __uint_as_float(wd);
                                en.idx = slot_elem<VEC>(cbase, g * G + j);
                            }
                            if (pos < TK_CAPC) cset[pos] = en;
                            ++pos;
                        }
                    }
                }
            }
            __syncthreads();  // every candidate of the chunk is in the set

            // ---- warp 0: tighten the set to its exact k-th largest when it grows large or the
            // segment ends; at the end, publish the segment's list.  The other warps go on with
            // the next chunk meanwhile.
            if (warp == 0) {
                const bool last = st + 1 == nst;
                int n = ncset;
                const int over = sover || k > NT || n > TK_CAPC;
                float nb = beta;
                if (!seg_bad && !over && (last || n > max(3 * k, 128) || n > TK_CAPC / 2)) {
                    uint32_t gk = okey(NEG_INF);
                    if (n >= k) {
                        if (n <= 32 * 8) gk = warp_kth_key_regs<DT, 8>(cset, n, k);
                        else if (n <= 32 * 16) gk = warp_kth_key_regs<DT, 16>(cset, n, k);
                        else gk = warp_kth_key<DT>(n, k, [&](int i) { return okey(cset[i].x); });
                    }
                    int m = 0;
                    for (int i0 = 0; i0 < n; i0 += 32) {
                        const int i = i0 + lane;
                        TopkEntry e;
                        bool keep = false;
                        if (i < n) {
                            e = cset[i];
                            keep = okey(e.x) >= gk;
                        }
                        const unsigned bal = __ballot_sync(FULL, keep);
                        __syncwarp();
                        if (keep) cset[m + __popc(bal & ((1u << lane) - 1u))] = e;
                        m += __popc(bal);
                        __syncwarp();
                    }
                    n = m;
                    nb = fmaxf(nb, key_value(gk));
                }
                if (last) {
                    const int code = seg_bad ? TK_NONFINITE : (over || n > P.cap_s) ? TK_OVERFLOW : n;
                    if (code > 0) {
                        TopkEntry* dst = P.clist + (size_t)sg * P.cap_s;
                        for (int i = lane; i < n; i += 32) dst[i] = cset[i];
                    }
                    if (lane == 0) {
                        P.ccount[sg] = code;
                        ncset = 0;
                        sbeta = NEG_INF;
                        sover = 0;
                    }
                } else if (lane == 0) {
                    ncset = n;
                    sbeta = nb;
                    sover = over;
                }
                __syncwarp();
            }
        }
    }
    // after a failed wait, let the copies still in flight land before the CTA leaves (bounded)
    if constexpr (BULK) {
        if (failed && tid == 0)
            for (long long j = fail_it; j < nissued && j < fail_it + TK_STAGES; ++j)
                (void)mbar_wait(&full[j % TK_STAGES], (unsigned)(j / TK_STAGES) & 1u);
    }
}

// Kernel 2, one warp per row: exact threshold g over the union of the row's segment lists, the
// kept list sorted by index, and the normaliser over it.  u holds nsegr * cap_s entries, kept
// cap_k.
template <int DT>
__device__ RowStats topk_row_finish(const SpecParams& P, TopkEntry* u, TopkEntry* kept, int row_id)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    RowStats st;
    st.M = NEG_INF; st.MC = NEG_INF; st.S = 0.0; st.thr = NEG_INF;
    st.status = ROW_OK; st.klist_n = -1; st.dense = 0;
    const int ns = P.nsegr;  // <= 4
    const int* cnt = P.ccount + (size_t)row_id * ns;
    const TopkEntry* lists = P.clist + (size_t)row_id * ns * P.cap_s;

    int n = (lane < ns) ? min(__ldcg(cnt + lane), P.cap_s) : 0;
    int flag = 0;
    if (n == TK_NONFINITE) flag |= 1;
    else if (n == TK_TIMEOUT) flag |= 4;
    else if (n < 0) flag |= 2;
    flag = (int)__reduce_or_sync(FULL, (unsigned)flag);
    if (flag & 4) { st.status = ROW_TIMEOUT; return st; }
    if (flag & 1) { st.status = ROW_NONFINITE; return st; }
    if (flag & 2) { st.dense = 1; return st; }
    // offsets of the segment lists in the union
    const int incl = warp_incl_scan(n);
    const int o1 = __shfl_sync(FULL, incl, 0), o2 = __shfl_sync(FULL, incl, 1),
              o3 = __shfl_sync(FULL, incl, 2), total = __shfl_sync(FULL, incl, 31);
    for (int f0 = 0; f0 < total; f0 += 32 * 8) {
        TopkEntry e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int f = f0 + 32 * j + lane;
            if (f < total) {
                const int sgi = (f >= o1) + (ns > 2 && f >= o2) + (ns > 3 && f >= o3);
                const int off = sgi == 0 ? 0 : sgi == 1 ? o1 : sgi == 2 ? o2 : o3;
                const TopkEntry* src = lists + (size_t)sgi * P.cap_s + (f - off);
                e[j].x = __ldcg(&src->x);
                e[j].idx = __ldcg(&src->idx);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int f = f0 + 32 * j + lane;
            if (f < total) u[f] = e[j];
        }
    }
    __syncwarp();

    const int k = P.top_k;
    const uint32_t gkey = (total >= k) ? warp_kth_key<DT>(total, k, [&](int i) { return okey(u[i].x); })
                                       : okey(NEG_INF);
    // stable ballot compaction of the entries >= g
    int nk = 0;
    for (int i0 = 0; i0 < total; i0 += 32) {
        const int i = i0 + lane;
        const bool keep = i < total && okey(u[i].x) >= gkey;
        const unsigned bal = __ballot_sync(FULL, keep);
        const int pos = nk + __popc(bal & ((1u << lane) - 1u));
        if (keep && pos < P.cap_k) kept[pos] = u[i];
        nk += __popc(bal);
    }
    __syncwarp();
    if (nk > P.cap_k) { st.dense = 1; return st; }
    warp_sort_by_index(kept, nk);
    float mx = NEG_INF;
    for (int i = lane; i < nk; i += 32) mx = fmaxf(mx, kept[i].x);
    const float M = warp_max(mx);
    const float MC = M * P.c;
    double acc = 0.0;
    if (M != NEG_INF)
        for (int i = lane; i < nk; i += 32) acc += (double)ex2(fmaf(kept[i].x, P.c, -MC));
    const double S = warp_sum(acc);
    TopkEntry* kl = P.klist + (size_t)row_id * P.cap_k;
    for (int i = lane; i < nk; i += 32) kl[i] = kept[i];
    st.M = M;
    st.MC = MC;
    st.S = S;
    st.thr = key_value(gkey);
    st.klist_n = nk;
    st.status = (M != NEG_INF && isfinite(M)) ? ROW_OK : ROW_NONFINITE;
    return st;
}

// Kernel 2: one CTA per request.  Warps take the request's rows; then one warp scans and draws.
template <int DT>
__global__ void __launch_bounds__(NT) topk_finish_kernel(SpecParams P)
{
    extern __shared__ __align__(16) TopkEntry fin[];  // per warp: u[nsegr*cap_s], kept[cap_k]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x;
    const int per = P.nsegr * P.cap_s + P.cap_k;
    TopkEntry* u = fin + (size_t)warp * per;
    TopkEntry* kept = u + P.nsegr * P.cap_s;
    for (int r = warp; r < P.R; r += WARPS) {
        const int row_id = b * P.R + r;
        const RowStats st = topk_row_finish<DT>(P, u, kept, row_id);
        if (lane == 0) P.rstats[row_id] = st;
    }
    __syncthreads();
    if (warp != 0) return;
    int nd = 0;
    for (int rr = lane; rr < P.R; rr += 32) nd += __ldcg(&P.rstats[(size_t)b * P.R + rr].dense);
    nd = __reduce_add_sync(0xffffffffu, nd);
    if (nd > 0) {  // finished by topk_dense_kernel
        if (lane == 0) P.ndense[b] = nd;
        return;
    }
    topk_request_epilogue<DT>(P, reinterpret_cast<double*>(fin), b);
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

__device__ __forceinline__ double block_sum_f64(double v, double* sh)
{
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = 0.0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) r += sh[w];
    return r;
}

template <int DT>
__global__ void __launch_bounds__(NT) topk_dense_kernel(SpecParams P)
{
    __shared__ int sh_red[WARPS];
    __shared__ double sh_d[WARPS];
    __shared__ float sh_f[WARPS];
    __shared__ int sh_flag, sh_tok;

    const int row_id = blockIdx.x;
    const int b = row_id / P.R, r = row_id % P.R;
    if (!__ldcg(&P.rstats[row_id].dense)) return;
    const char* row = spec_row_ptr(P, b, r);
    const int V = P.V, k = P.top_k;

    // exact k-th largest key by bitwise search over full-row counts
    uint32_t prefix = 0;
    constexpr int lo = (DT == DT_BF16) ? 16 : 0;
    for (int bit = 31; bit >= lo; --bit) {
        const uint32_t want = prefix | (1u << bit);
        int cnt = 0;
        for (int v = threadIdx.x; v < V; v += NT) cnt += okey(load_logit(row, DT, v)) >= want;
        if (block_sum_int(cnt, sh_red) >= k) prefix = want;
    }
    if (DT == DT_BF16 && prefix < 0x80000000u) prefix |= 0xffffu;
    const float g = key_value(prefix);
    float mx = NEG_INF;
    for (int v = threadIdx.x; v < V; v += NT) {
        const float x = load_logit(row, DT, v);
        if (x >= g) mx = fmaxf(mx, x);
    }
    const float M = block_max(mx, sh_f);
    const float MC = M * P.c;
    float s = 0.f;
    if (M != NEG_INF)
        for (int v = threadIdx.x; v < V; v += NT) {
            const float x = load_logit(row, DT, v);
            if (x >= g) s += ex2(fmaf(x, P.c, -MC));
        }
    const double S = block_sum_f32(s, sh_d);
    if (threadIdx.x == 0) {
        RowStats st;
        st.M = M; st.MC = MC; st.S = S; st.thr = g;
        st.status = (M != NEG_INF && isfinite(M) && S > 0.0) ? ROW_OK : ROW_NONFINITE;
        st.klist_n = -1;
        st.dense = 1;
        P.rstats[row_id] = st;
    }
    const unsigned nd = (unsigned)__ldcg(&P.ndense[b]);
    if (!arrive_last(&P.dense_ctr[b], nd, &sh_flag)) return;
    if (threadIdx.x == 0) P.ndense[b] = 0;

    __shared__ Plan sh_plan;
    if (threadIdx.x < 32) {
        const Plan p0 = compute_plan_warp<DT>(P, b, true);
        if (threadIdx.x == 0) sh_plan = p0;
    }
    __syncthreads();
    const Plan pl = sh_plan;
    if (pl.status != ROW_OK) {
        emit_spec(P, b, pl.status, 0, -1);
        return;
    }
    const char* rowp = spec_row_ptr(P, b, pl.rp);
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    // pass 1: total residual mass, tile by tile in index order (fp64)
    double Z = 0.0;
    for (int t0 = 0; t0 < V; t0 += NT) {
        const int v = t0 + threadIdx.x;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        Z += block_sum_f64(rv, sh_d);
    }
    if (!(Z > 0.0) || !isfinite(Z)) {
        emit_spec(P, b, ROW_DEGENERATE, 0, -1);
        return;
    }
    // pass 2: the tile where the running mass passes u*Z, then the element inside it
    const double t = pl.u * Z;
    double run = 0.0;
    int tok = -1;
    for (int t0 = 0; t0 < V; t0 += NT) {
        const int v = t0 + threadIdx.x;
        const double rv = v < V ? topk_residual_at<DT>(rowp, rowq, v, pl, P.c) : 0.0;
        const double ts = block_sum_f64(rv, sh_d);
        if (t < run + ts) {  // uniform across the CTA
            double tot;
            const double excl = block_excl_scan_f64(rv, sh_d, &tot);
            if (threadIdx.x == 0) sh_tok = 0x7fffffff;
            __syncthreads();
            if (rv > 0.0 && t < run + excl + rv) atomicMin(&sh_tok, v);
            __syncthreads();
            tok = sh_tok;
            if (tok == 0x7fffffff) {  // rounding: last positive entry of the tile
                __syncthreads();
                if (threadIdx.x == 0) sh_tok = -1;
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
        if (threadIdx.x == 0) sh_tok = -1;
        __syncthreads();
        for (int v = threadIdx.x; v < V; v += NT)
            if (topk_residual_at<DT>(rowp, rowq, v, pl, P.c) > 0.0) atomicMax(&sh_tok, v);
        __syncthreads();
        tok = sh_tok;
    }
    emit_spec(P, b, tok >= 0 ? ROW_OK : ROW_DEGENERATE, pl.A, tok);
}


// persistent grid of CTAs: resident CTAs per SM x SMs, at most one per task
template <auto K>
static unsigned cta_grid(long long tasks, int sms, size_t smem)
{
    static int per_sm = 0;
    if (per_sm < 1) {
        int n = 0;
        if (smem > 48 * 1024) cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, NT, smem) != cudaSuccess || n < 1) n = 1;
        per_sm = n;
    }
    const long long cap = (long long)per_sm * sms;
    return (unsigned)(tasks < 1 ? 1 : (tasks < cap ? tasks : cap));
}

template <auto K>
static void set_smem_limit(size_t smem)
{
    static size_t done = 0;
    if (smem > 48 * 1024 && smem > done) {
        cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        done = smem;
    }
}

template <int DT>
static void launch_topk(const SpecParams& P, int sms, cudaStream_t st)
{
    const long long nsegs = (long long)P.B * P.R * P.nsegr;
    if (P.vec > 1) {
        constexpr auto K1 = topk_stream_kernel<DT, true>;
        K1<<<cta_grid<K1>(nsegs, sms, TK_SMEM), NT, TK_SMEM, st>>>(P);
    } else {
        constexpr auto K1 = topk_stream_kernel<DT, false>;
        K1<<<cta_grid<K1>(nsegs, sms, 0), NT, 0, st>>>(P);
    }
    const size_t fsm = (size_t)WARPS * (P.nsegr * P.cap_s + P.cap_k) * sizeof(TopkEntry);
    set_smem_limit<topk_finish_kernel<DT>>(fsm);
    topk_finish_kernel<DT><<<(unsigned)P.B, NT, fsm, st>>>(P);
    topk_dense_kernel<DT><<<(unsigned)((long long)P.B * P.R), NT, 0, st>>>(P);
}

cudaError_t launch_topk_path(const SpecParams& P, int sms, cudaStream_t st)
{
    if (P.dtype == DT_BF16) launch_topk<DT_BF16>(P, sms, st);
    else launch_topk<DT_F32>(P, sms, st);
    return cudaGetLastError();
}

}  // namespace sv
