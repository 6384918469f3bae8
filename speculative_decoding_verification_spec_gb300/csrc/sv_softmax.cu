// sv_softmax.cu -- exact speculative sampling without top-k: one-pass row normalisers and the
// residual / bonus inverse-CDF draw.
//
// Kernel 1 (row statistics).  Rows of 16-byte vectors: spec_stream_kernel, persistent CTAs that
// fetch 32 KB chunks with bulk copies into a shared-memory ring and write one (max, sum of
// 2^(x c - max c)) partial per (chunk, warp) -- the (m, l) pairs of M7.1 section 0x04J; then
// spec_rowplan_kernel merges each row's partials (pairs of floats, chunk order) with one warp per
// row, and the last warp of a request runs the acceptance scan (sv_plan.cuh).  Rows that are not
// 16-byte aligned use persistent warps with plain loads and do the same merge through completion
// counters.
//
// Kernel 2 (residual draw): r = max(p - q, 0) (M7.1 section 0x03C; p alone for the bonus, 0x03H)
// over the selected row pair, summed per segment of 32 vectors; the last CTA of a request scans the
// segment sums in index order (lane totals in fp64), finds the segment where the running mass
// passes u * Z, and resolves the token inside it.
//
// Rows of the two row pairs most likely to be corrected (pairs 0 and 1) are read with the L2
// evict_normal policy and all other rows evict_first, so that kernel 2 tends to find them in L2.
#include "sv_draw.cuh"

namespace sv {

// ---------------------------------------------------------------- kernel 1: row statistics

// Online softmax statistics of one task: lane accumulators (m, mc, s), mc = fp32(m*c),
// s = sum 2^(fma(x, c, -mc)).
template <int DT, int VEC>
__device__ __forceinline__ void task_softmax_stats(const char* row, const uint32_t* mrow, long long t0,
                                                   long long t1, float c, uint64_t pol, float& m,
                                                   float& mc, float& s)
{
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int step = 0; step < ST1; ++step) {
        const long long base = t0 + (long long)step * 32 * U1 + lane;
        if (t0 + (long long)step * 32 * U1 >= t1) break;
        if constexpr (DT == DT_BF16 && VEC == 8) {
            uint4 w[U1];
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                const long long v = base + u * 32;
                if (v < t1) {
                    w[u] = ld_stream_v4_pol(row + v * 16, pol);
                    if (mrow) mask_raw<DT, 8>(w[u], allowed_bits<8>(mrow, v));
                } else {
                    w[u] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                }
            }
            uint32_t pm = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
            for (int u = 1; u < U1; ++u)
                pm = bmax2(pm, bmax2(bmax2(w[u].x, w[u].y), bmax2(w[u].z, w[u].w)));
            const float bm = fmaxf(bf16lo(pm), bf16hi(pm));
            if (bm > m) {
                const float mcn = __fmul_rn(bm, c);
                s *= ex2(mc - mcn);
                m = bm;
                mc = mcn;
            }
            if (mc != NEG_INF) {
                float acc[U1];
#pragma unroll
                for (int u = 0; u < U1; ++u) {
                    const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                    float e[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        e[2 * k] = ex2(fmaf(bf16lo(q[k]), c, -mc));
                        e[2 * k + 1] = ex2(fmaf(bf16hi(q[k]), c, -mc));
                    }
                    acc[u] = tree_sum(e);
                }
                s += tree_sum(acc);
            }
        } else {
            float x[U1][VEC];
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                const long long v = base + u * 32;
                if (v < t1) {
                    load_vec_pol<DT, VEC>(row, v, pol, x[u]);
                    if (mrow) mask_vals<VEC>(x[u], allowed_bits<VEC>(mrow, v));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) x[u][e] = NEG_INF;
                }
            }
            float bm = NEG_INF;
#pragma unroll
            for (int u = 0; u < U1; ++u)
#pragma unroll
                for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, x[u][e]);
            if (bm > m) {
                const float mcn = __fmul_rn(bm, c);
                s *= ex2(mc - mcn);
                m = bm;
                mc = mcn;
            }
            if (mc != NEG_INF) {
                float acc[U1];
#pragma unroll
                for (int u = 0; u < U1; ++u) {
                    float e[VEC];
#pragma unroll
                    for (int k = 0; k < VEC; ++k) e[k] = ex2(fmaf(x[u][k], c, -mc));
                    acc[u] = tree_sum(e);
                }
                s += tree_sum(acc);
            }
        }
    }
}

__device__ __forceinline__ Partial ld_partial(const Partial* p)
{
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
    Partial r;
    r.M = v.x;
    r.MC = v.y;
    r.S = v.z;
    r.pad = 0.f;
    return r;
}

// task t -> (request b, row r, slice s); request-major, rows in index order
__device__ __forceinline__ void decode_stats_task(const SpecParams& P, long long t, int& b, int& r,
                                                  int& s)
{
    s = (int)(t % P.S1);
    const long long rr = t / P.S1;
    r = (int)(rr % P.R);
    b = (int)(rr / P.R);
}


template <int DT>
__device__ void row_merge_and_plan(const SpecParams& P, int b, int row_id, int nparts);

// End of a stats task: warp merge of the lane accumulators, the slice partial, and -- for the warp
// that completes a row / a request -- the row merge and the acceptance scan.
template <int DT>
__device__ __forceinline__ void stats_finalize(const SpecParams& P, int b, int r, int s, float m,
                                               float mc, float acc)
{
    const int lane = threadIdx.x & 31;
    const float M = warp_max(m);
    const float MC = __fmul_rn(M, P.c);
    const float sc = (mc == NEG_INF) ? 0.f : acc * ex2(mc - MC);
    const float S = warp_sum(sc);
    const int row_id = b * P.R + r;
    if (lane == 0) {
        Partial pt;
        pt.M = M;
        pt.MC = MC;
        pt.S = S;
        pt.pad = 0.f;
        P.partials[(size_t)row_id * P.S1 + s] = pt;
    }
    if (warp_arrive_last(&P.row_ctr[row_id], (unsigned)P.S1)) row_merge_and_plan<DT>(P, b, row_id, P.S1);
}

// Called by the warp that completed row `row_id`: merge its `nparts` partials in order into
// RowStats; the warp that completes the last row of request b then runs the acceptance scan.
template <int DT>
__device__ void row_merge_and_plan(const SpecParams& P, int b, int row_id, int nparts)
{
    const int lane = threadIdx.x & 31;
    const Partial* pp = P.partials + (size_t)row_id * nparts;
    float Mr = NEG_INF;
    for (int k = lane; k < nparts; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
    Mr = warp_max(Mr);
    const float MCr = __fmul_rn(Mr, P.c);
    double Sr = 0.0;
    for (int k = lane; k < nparts; k += 32) {
        const Partial q = ld_partial(pp + k);
        if (q.S != 0.0) Sr += q.S * exp2((double)q.MC - (double)MCr);
    }
    Sr = warp_sum(Sr);
    if (lane == 0) {
        RowStats st;
        st.M = Mr;
        st.MC = MCr;
        st.S = Sr;
        st.thr = NEG_INF;
        st.klist_n = -1;
        st.dense = 0;
        const bool ok = isfinite(Sr) && Sr > 0.0 && Mr != NEG_INF && isfinite(Mr);
        st.status = ok ? ROW_OK : ROW_NONFINITE;
        P.rstats[row_id] = st;
    }
    if (warp_arrive_last(&P.req_ctr[b], (unsigned)P.R)) {
        const Plan pl = compute_plan_warp<DT>(P, b, false);
        if (lane == 0) P.plan[b] = pl;
    }
}

// Online update of the lane accumulators with one step of 16-byte vectors (raw bits).
template <int DT, int NU>
__device__ __forceinline__ void stats_step(const uint4 (&w)[NU], float c, float& m, float& mc,
                                           float& s)
{
    float bm;
    if constexpr (DT == DT_BF16) {
        uint32_t pm = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
        for (int u = 1; u < NU; ++u) pm = bmax2(pm, bmax2(bmax2(w[u].x, w[u].y), bmax2(w[u].z, w[u].w)));
        bm = fmaxf(bf16lo(pm), bf16hi(pm));
    } else {
        bm = NEG_INF;
#pragma unroll
        for (int u = 0; u < NU; ++u)
            bm = fmaxf(fmaxf(bm, fmaxf(__uint_as_float(w[u].x), __uint_as_float(w[u].y))),
                       fmaxf(__uint_as_float(w[u].z), __uint_as_float(w[u].w)));
    }
    if (bm > m) {
        const float mcn = __fmul_rn(bm, c);
        s *= ex2(mc - mcn);
        m = bm;
        mc = mcn;
    }
    if (mc == NEG_INF) return;
    float acc[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        if constexpr (DT == DT_BF16) {
            float e[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                e[2 * k] = ex2(fmaf(bf16lo(q[k]), c, -mc));
                e[2 * k + 1] = ex2(fmaf(bf16hi(q[k]), c, -mc));
            }
            acc[u] = tree_sum(e);
        } else {
            float e[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) e[k] = ex2(fmaf(__uint_as_float(q[k]), c, -mc));
            acc[u] = tree_sum(e);
        }
    }
    s += tree_sum(acc);
}

// Scalar-path kernel (rows not 16-byte aligned): plain loads, one task per warp at a time.
template <int DT, int VEC>
__global__ void __launch_bounds__(NT) spec_stats_kernel(SpecParams P)
{
    const uint64_t pol_first = policy_evict_first(), pol_keep = policy_evict_normal();
    long long t = claim_task(&P.work[0]);
    while (t < P.tasks1) {
        const long long next = claim_task(&P.work[0]);  // claimed early: hides the atomic latency
        int b, r, s;
        decode_stats_task(P, t, b, r, s);
        const char* row = spec_row_ptr(P, b, r);
        const long long t0 = (long long)s * TV1;
        const long long t1 = min(t0 + TV1, P.nvec);
        float m = NEG_INF, mc = NEG_INF, acc = 0.f;
        task_softmax_stats<DT, VEC>(row, P.mask ? spec_mask_row(P, b, r) : nullptr, t0, t1, P.c,
                                    pinned_row(P, r) ? pol_keep : pol_first, m, mc, acc);
        stats_finalize<DT>(P, b, r, s, m, mc, acc);
        t = next;
    }
}

// consumer groups per CTA of the streaming kernel (see ring_produce): one, with two CTAs per SM;
// two groups in one CTA per SM were slower here (plain rows by 1%, masked rows by 3%)
constexpr int SPEC_GROUPS = 1;

// Streaming kernel for rows of 16-byte vectors: persistent CTAs take 32 KB chunks round-robin,
// fetched by bulk copies (TMA engine) into a ring of STREAM_STAGES shared-memory stages, so the
// next chunks are in flight while one is reduced.  Each warp reduces its part of a chunk -- the
// maximum first, then the sum of 2^(x c - MC) with MC = fp32(M c) -- and writes one partial per
// (chunk, warp).  Warp-specialised: a producer warp fills the ring (ring_produce) and the consumer
// warps release each stage on its "empty" mbarrier, so they never wait for one another.
// NaN or +inf anywhere makes the partial's sum NaN, so the row merge reports the row non-finite.
// MASK (a grammar mask): the mask bits of the thread's vectors are applied to the raw vectors as
// they leave shared memory.  MASK_RING: the producer copies a chunk's mask bits (one bit per
// element) into the stage beside its logits, with a second bulk copy completing on the same barrier
// (mask rows of a multiple of 16 bytes, 16-byte aligned).  MASK_REGS otherwise: each thread loads
// its bits two chunks ahead into one of two register sets used in turn, so their latency hides
// behind the chunks in between.
template <int DT, int MASK>
__global__ void __launch_bounds__(stream_threads<SPEC_GROUPS>(), 2 / SPEC_GROUPS) spec_stream_kernel(SpecParams P)
{
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    constexpr int ES = (DT == DT_BF16) ? 2 : 4;
    constexpr int CHUNK = NT * STREAM_NV * VEC;  // elements per chunk
    // SPEC_GROUPS x STREAM_STAGES stages of NT * STREAM_NV vectors; MASK_RING: then as many
    // stages of STREAM_MASK_BYTES of mask bits
    extern __shared__ __align__(128) uint4 ring[];
    uint32_t* mring = reinterpret_cast<uint32_t*>(ring + (size_t)SPEC_GROUPS * STREAM_STAGES * NT * STREAM_NV);
    __shared__ __align__(8) uint64_t full[SPEC_GROUPS * STREAM_STAGES];
    __shared__ __align__(8) uint64_t empty[SPEC_GROUPS * STREAM_STAGES];
    __shared__ int sfail;  // a wait ran out in this CTA: nothing more is read

    pdl_trigger();  // the row-merge kernel may be scheduled as SMs free up; it waits for this grid
    clear_counters(P.ctr_clear, P.ctr_words);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int nch = P.B * P.R * P.S1;  // < 2^31 (checked on the host)
    const float c = P.c;
    if (tid == 0) {
        sfail = 0;
        for (int s = 0; s < SPEC_GROUPS * STREAM_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == SPEC_GROUPS * WARPS) {  // the producer: the rows of the likely correction pairs stay in L2
        if (lane == 0)
            ring_produce<SPEC_GROUPS>(full, empty, &sfail, nch, P.wait_limit, [&](int s, int id) {
                const int row_id = id / P.S1, ci = id - row_id * P.S1;
                const int b = row_id / P.R, r = row_id - b * P.R;
                const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, P.V);
                const uint64_t pol = pinned_row(P, r) ? policy_evict_normal() : policy_evict_first();
                if constexpr (MASK == MASK_RING) {
                    // with the chunk's mask words, rounded up to 16 bytes: inside the row, whose
                    // words are a multiple of four
                    const unsigned mbytes = (unsigned)((((cend - cbase + 31) >> 5) + 3) & ~3) * 4u;
                    bulk_load2(ring + (size_t)s * NT * STREAM_NV, spec_row_ptr(P, b, r) + (size_t)cbase * ES,
                               (unsigned)(cend - cbase) * ES, mring + (size_t)s * (STREAM_MASK_BYTES / 4),
                               spec_mask_row(P, b, r) + (size_t)ci * (CHUNK / 32), mbytes, &full[s], pol,
                               policy_evict_first());
                } else {
                    bulk_load(ring + (size_t)s * NT * STREAM_NV, spec_row_ptr(P, b, r) + (size_t)cbase * ES,
                              (unsigned)(cend - cbase) * ES, &full[s], pol);
                }
            });
        return;
    }
    const StreamGroup<SPEC_GROUPS> sg;
    uint64_t* gfull = full + sg.g * STREAM_STAGES;
    uint64_t* gempty = empty + sg.g * STREAM_STAGES;
    const uint4* gring = ring + (size_t)sg.g * STREAM_STAGES * NT * STREAM_NV;
    const uint32_t* gmring = mring + (size_t)sg.g * STREAM_STAGES * (STREAM_MASK_BYTES / 4);
    const int tid_g = sg.t;  // thread within the group

    bool failed = false;  // a wait ran out: the remaining chunks are reported, not read
    int stg = 0;          // it % STREAM_STAGES
    unsigned phase = 0;   // (it / STREAM_STAGES) & 1
    // chunk id = row_id * S1 + ci, advanced by the stride without a division per chunk
    int row_id = sg.vb / P.S1, ci = sg.vb - row_id * P.S1;
    const int drow = sg.stride / P.S1, dci = sg.stride - drow * P.S1;
    // the mask bits of chunk (rid, cix) for this thread's vectors: vector j * NT + tid_g of the
    // chunk sits in word (j * NT + tid_g) * VEC / 32 of the chunk's CHUNK / 32 words, at a fixed shift
    auto load_mask = [&](int rid, int cix, uint32_t (&out)[STREAM_NV]) {
        const int b = rid / P.R;
        const uint32_t* mw = spec_mask_row(P, b, rid - b * P.R) + (size_t)cix * (CHUNK / 32) + (tid_g * VEC) / 32;
        const unsigned sh = (unsigned)(tid_g * VEC) & 31u;
        const int left = P.V - cix * CHUNK - tid_g * VEC;  // elements from this thread's first vector on
#pragma unroll
        for (int j = 0; j < STREAM_NV; ++j) {
            uint32_t wv = 0u;
            if (j * NT * VEC < left)
                asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(wv) : "l"(mw + j * (NT * VEC / 32)));
            out[j] = (wv >> sh) & ((1u << VEC) - 1u);
        }
    };
    auto advance = [&](int& r, int& c) {
        r += drow;
        c += dci;
        if (c >= P.S1) {
            c -= P.S1;
            ++r;
        }
    };
    int pr = row_id, pc = ci;  // MASK: the chunk whose bits are loaded next
    // one chunk; with MASK, mreg holds its bits (loaded two chunks earlier) and is refilled
    auto process = [&](int id, uint32_t (&mreg)[STREAM_NV]) {
        if (id != sg.vb) {
            advance(row_id, ci);
            if (++stg == STREAM_STAGES) {
                stg = 0;
                phase ^= 1u;
            }
        }
        const int cbase = ci * CHUNK, cend = min(cbase + CHUNK, P.V);
        const bool partial = cbase + CHUNK > cend;
        const int s = stg;
        if (!failed && *reinterpret_cast<volatile int*>(&sfail)) failed = true;
        bool ok = !failed && mbar_wait(&gfull[s], phase, P.wait_limit);
        uint4 w[STREAM_NV];
        const uint32_t pad = (DT == DT_BF16) ? 0xff80ff80u : 0xff800000u;
        const uint4* sb = gring + (size_t)s * NT * STREAM_NV + tid_g;
        if (ok && !partial) {
#pragma unroll
            for (int j = 0; j < STREAM_NV; ++j) w[j] = lds128(sb + j * NT);
        } else {
#pragma unroll
            for (int j = 0; j < STREAM_NV; ++j) {
                w[j] = make_uint4(pad, pad, pad, pad);
                if (ok && cbase + (j * NT + tid_g) * VEC < cend) w[j] = lds128(sb + j * NT);
            }
        }
        // MASK: vector j of every lane of the warp fully masked (bit j) is skipped below: its
        // elements would only add 2^-inf = 0
        unsigned skipm = 0u;
        if constexpr (MASK != MASK_NONE) {
            uint32_t bits[STREAM_NV];
            if constexpr (MASK == MASK_REGS) {
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) bits[j] = mreg[j];
                // this register set is free again: the bits of the chunk two ahead
                if ((long long)id + 2 * sg.stride < nch) load_mask(pr, pc, mreg);
                advance(pr, pc);
            } else {
                // vector j * NT + tid_g of the chunk: word (j * NT + tid_g) * VEC / 32 of the stage's bits
                const uint32_t* mw = gmring + (size_t)s * (STREAM_MASK_BYTES / 4);
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) {
                    const int e0 = (j * NT + tid_g) * VEC;
                    bits[j] = (ok && (!partial || cbase + e0 < cend))
                                  ? (mw[e0 >> 5] >> (e0 & 31)) & ((1u << VEC) - 1u) : 0u;
                }
            }
#pragma unroll
            for (int j = 0; j < STREAM_NV; ++j) {
                if (__all_sync(FULL, bits[j] == 0u)) {
                    skipm |= 1u << j;
                    w[j] = make_uint4(pad, pad, pad, pad);
                } else {
                    mask_raw<DT, VEC>(w[j], bits[j]);
                }
            }
        }
        // release the stage once every lane has read it; a warp whose wait ran out never releases
        // it (its copy may still land), which stops the producer
        ok = __all_sync(FULL, ok);
        if (ok) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&gempty[s]);
        } else if (!failed) {
            failed = true;
            if (lane == 0) *reinterpret_cast<volatile int*>(&sfail) = 1;
        }
        Partial pt;
        pt.pad = 0.f;
        if (failed) {
            pt.M = __int_as_float(0x7fc00000);  // the chunk was not read: S < 0 marks a timeout
            pt.MC = pt.M;
            pt.S = -1.f;
        } else {
            // maximum of the thread's elements, then of the warp
            float m;
            if constexpr (DT == DT_BF16) {
                uint32_t pm = w[0].x;
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) {
                    pm = bmax2(pm, w[j].x); pm = bmax2(pm, w[j].y);
                    pm = bmax2(pm, w[j].z); pm = bmax2(pm, w[j].w);
                }
                m = fmaxf(bf16lo(pm), bf16hi(pm));
            } else {
                m = NEG_INF;
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j)
                    m = fmaxf(fmaxf(m, __uint_as_float(w[j].x)), fmaxf(fmaxf(__uint_as_float(w[j].y),
                            __uint_as_float(w[j].z)), __uint_as_float(w[j].w)));
            }
            const float M = warp_max(m);
            const float MC = __fmul_rn(M, c);
            // sum of 2^(x c - MC) in four fp32 accumulators, combined in a fixed order: a0 and a1
            // take the low and high elements of words x and z, a2 and a3 those of y and w, two at a
            // time with the packed fp32 instructions (each half rounds as the scalar one would)
            unsigned long long a01 = 0ull, a23 = 0ull;
            if (M != NEG_INF) {
                const unsigned long long c2 = f2_pack(c, c), nmc2 = f2_pack(-MC, -MC);
                auto acc2 = [&](unsigned long long& a, float lo, float hi) {
                    float ylo, yhi;
                    f2_unpack(f2_fma(f2_pack(lo, hi), c2, nmc2), ylo, yhi);
                    a = f2_add(a, f2_pack(ex2(ylo), ex2(yhi)));
                };
#pragma unroll
                for (int j = 0; j < STREAM_NV; ++j) {
                    if (MASK != MASK_NONE && ((skipm >> j) & 1u)) continue;  // the same in every lane
                    if constexpr (DT == DT_BF16) {
                        acc2(a01, bf16lo(w[j].x), bf16hi(w[j].x));
                        acc2(a23, bf16lo(w[j].y), bf16hi(w[j].y));
                        acc2(a01, bf16lo(w[j].z), bf16hi(w[j].z));
                        acc2(a23, bf16lo(w[j].w), bf16hi(w[j].w));
                    } else {
                        acc2(a01, __uint_as_float(w[j].x), __uint_as_float(w[j].y));
                        acc2(a23, __uint_as_float(w[j].z), __uint_as_float(w[j].w));
                    }
                }
            }
            float a0, a1, a2, a3;
            f2_unpack(a01, a0, a1);
            f2_unpack(a23, a2, a3);
            pt.M = M;
            pt.MC = MC;
            pt.S = warp_sum((a0 + a1) + (a2 + a3));
        }
        if (lane == 0) P.partials[((size_t)row_id * P.S1 + ci) * WARPS + sg.w] = pt;
    };
    if constexpr (MASK == MASK_REGS) {
        // two register sets in turn, so that no register move waits for a load still in flight
        uint32_t mA[STREAM_NV], mB[STREAM_NV];
        if (sg.vb < nch) load_mask(pr, pc, mA);
        advance(pr, pc);
        if ((long long)sg.vb + sg.stride < nch) load_mask(pr, pc, mB);
        advance(pr, pc);
        for (int id = sg.vb; id < nch; id += 2 * sg.stride) {
            process(id, mA);
            if ((long long)id + sg.stride < nch) process(id + sg.stride, mB);
        }
    } else {
        uint32_t none[STREAM_NV];
        for (int id = sg.vb; id < nch; id += sg.stride) process(id, none);
    }
}

// Row merge and plan, one CTA per request of nw = min(R, PLAN_WARPS) warps (8 when R > 32).  Warp
// w merges rows w, w + nw, ... (two at a time, the partial loads of both in flight together): each
// row's S1 x WARPS partials in order into RowStats, with the lse, 1/S and log2 p(x) of the token the
// row scores, kept in shared memory.  After one CTA barrier warp 0 runs the acceptance scan over
// them and writes the plan.
constexpr int PLAN_WARPS = 16;
template <int DT>
__global__ void __launch_bounds__(PLAN_WARPS * 32) spec_rowplan_kernel(SpecParams P)
{
    __shared__ RowStats srs[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int b = blockIdx.x, g = P.gamma, R = P.R;
    const unsigned FULL = 0xffffffffu;
    const int nparts = P.S1 * WARPS;

    // the token row r scores and its logit (inputs: fetched before waiting for the partials)
    auto token_logit = [&](int r, bool& ok) -> float {
        const int pos = (r < g) ? r : (r > g) ? r - g - 1 : -1;
        const int tok = (r < R && pos >= 0) ? __ldg(P.tokens + (size_t)b * g + pos) : -1;
        ok = tok >= 0 && tok < P.V;
        return ok ? masked_logit(P, b, r, DT, tok) : 0.f;
    };
    // lane 0: the row's statistics from its merged maximum and sum
    auto row_stats = [&](float Mr, DFloat Sr, int tmo, bool tok_ok, float xtok) {
        const float MCr = __fmul_rn(Mr, P.c);
        RowStats st = blank_rowstats();
        st.M = Mr;
        st.MC = MCr;
        st.S = (double)Sr.hi;
        const bool ok = !tmo && isfinite(Sr.hi) && Sr.hi > 0.f && Mr != NEG_INF && isfinite(Mr);
        st.status = tmo ? ROW_TIMEOUT : ok ? ROW_OK : ROW_NONFINITE;
        st.lse = __int_as_float(0x7fc00000);
        st.lx_hi = __int_as_float(0x7fc00000);
        st.lx_lo = 0.f;
        if (ok) row_norm(st, Mr, MCr, Sr, P, tok_ok, xtok, NEG_INF);
        return st;
    };
    auto publish_row = [&](int r, const RowStats& st) {
        if (lane == 0) {
            P.rstats[(size_t)b * R + r] = st;
            if (r < 32) srs[r] = st;
            else __threadfence();  // read back by warp 0 from global memory
        }
    };

    // rows r0 = warp + 2 nw j and r1 = r0 + nw, prefetched before the wait
    for (int r0 = warp; r0 < R; r0 += 2 * nw) {
        const int r1 = r0 + nw;
        bool ok0, ok1;
        const float x0 = token_logit(r0, ok0);
        const float x1 = token_logit(r1, ok1);
        if (r0 == warp) {
            pdl_trigger();
            pdl_wait();  // the partials of the streaming kernel
        }
        if (nparts <= 64) {
            // both rows' partials in flight at once: two per lane and row
            Partial q[2][2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int rr = h ? r1 : r0, k = lane + 32 * t;
                    q[h][t].M = NEG_INF;
                    q[h][t].MC = NEG_INF;
                    q[h][t].S = 0.f;
                    if (rr < R && k < nparts) q[h][t] = ld_partial(P.partials + ((size_t)b * R + rr) * nparts + k);
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = h ? r1 : r0;
                if (rr >= R) break;  // the same for the whole warp
                const float Mr = warp_max(fmaxf(q[h][0].M, q[h][1].M));
                const float MCr = __fmul_rn(Mr, P.c);
                // the chunk sums rescaled to MCr, added as pairs of floats
                DFloat Sr = df_make(0.f, 0.f);
                int tmo = 0;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (q[h][t].S < 0.f) tmo = 1;  // a chunk the streaming kernel could not read
                    if (q[h][t].S != 0.f) Sr = df_add(Sr, df_make(__fmul_rn(q[h][t].S, ex2(q[h][t].MC - MCr)), 0.f));  // NaN and inf propagate
                }
                Sr = warp_sum_df(Sr);
                tmo = __any_sync(FULL, tmo);
                publish_row(rr, row_stats(Mr, Sr, tmo, h ? ok1 : ok0, h ? x1 : x0));
            }
        } else {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int rr = h ? r1 : r0;
                if (rr >= R) break;
                const Partial* pp = P.partials + ((size_t)b * R + rr) * nparts;
                float Mr = NEG_INF;
                for (int k = lane; k < nparts; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
                Mr = warp_max(Mr);
                const float MCr = __fmul_rn(Mr, P.c);
                DFloat Sr = df_make(0.f, 0.f);
                int tmo = 0;
                for (int k = lane; k < nparts; k += 32) {
                    const Partial q = ld_partial(pp + k);
                    if (q.S < 0.f) tmo = 1;
                    if (q.S != 0.f) Sr = df_add(Sr, df_make(__fmul_rn(q.S, ex2(q.MC - MCr)), 0.f));
                }
                Sr = warp_sum_df(Sr);
                tmo = __any_sync(FULL, tmo);
                publish_row(rr, row_stats(Mr, Sr, tmo, h ? ok1 : ok0, h ? x1 : x0));
            }
        }
    }
    if (warp >= R) {  // a warp without rows still lets the next grid launch and waits like the rest
        pdl_trigger();
        pdl_wait();
    }
    __syncthreads();
    if (warp != 0) return;
    Plan pl;
    if (R <= 32) {
        RowStats rs = blank_rowstats();
        if (lane < R) rs = srs[lane];
        pl = plan_from_lanes(P, b, rs);
    } else {
        __threadfence_block();
        pl = compute_plan_warp<DT, true>(P, b, false);
    }
    if (lane == 0) P.plan[b] = pl;
}

// ---------------------------------------------------------------- kernel 2: residual draw
// (apply_thresholds, residual_from, resolve_in_segment, draw_from_segments: sv_draw.cuh)

template <int DT, int VEC>
__global__ void __launch_bounds__(NT) spec_resample_kernel(SpecParams P)
{
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    long long t = claim_task(&P.work[1]);
    while (t < P.tasks2) {
        const long long next = claim_task(&P.work[1]);
        const int b = (int)(t / P.S2), s = (int)(t % P.S2);
        const Plan pl = ld_plan(P.plan + b);
        const char* rowp = spec_row_ptr(P, b, pl.rp);
        const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
        const uint32_t* mrow = P.mask ? spec_mask_row(P, b, pl.rp) : nullptr;
        if (pl.status == ROW_OK) {
            const long long t0 = (long long)s * TV2;
            const long long t1 = min(t0 + TV2, P.nvec);
            float* segs = P.segs + (size_t)b * P.nseg;
#pragma unroll 1
            for (int step = 0; step < ST2; ++step) {
                const long long sb = t0 + (long long)step * 32 * U2;
                if (sb >= t1) break;
                RawVec<DT, VEC> xp[U2], xq[U2];
#pragma unroll
                for (int u = 0; u < U2; ++u) {
                    const long long v = sb + u * 32 + lane;
                    xp[u].fill_neg_inf();
                    xq[u].fill_neg_inf();
                    if (v < t1) {
                        xp[u].load(rowp, v, pol);
                        if (rowq) xq[u].load(rowq, v, pol);
                        if (mrow) {
                            const uint32_t bits = allowed_bits<VEC>(mrow, v);
                            mask_raw<DT, VEC>(xp[u].w, bits);
                            mask_raw<DT, VEC>(xq[u].w, bits);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U2; ++u) {
                    const long long v = sb + u * 32 + lane;
                    float ls = 0.f;
                    if (v < t1) {
                        float a[VEC], q[VEC], r[VEC];
#pragma unroll
                        for (int e = 0; e < VEC; ++e) { a[e] = xp[u].get(e); q[e] = xq[u].get(e); }
                        apply_thresholds<VEC>(a, q, rowq != nullptr, pl);
                        residual_from<VEC>(a, q, rowq != nullptr, pl, P.c, r);
                        ls = tree_sum(r);
                    }
                    const float ws = warp_sum(ls);
                    if (lane == 0 && sb + u * 32 < t1) segs[(sb + u * 32) / SEGV] = ws;
                }
            }
        }
        if (warp_arrive_last(&P.res_ctr[b], (unsigned)P.S2)) {
            int st = pl.status, tok = -1;
            if (st == ROW_OK) {
                tok = draw_from_segments<DT, VEC>(P, b, pl, rowp, rowq);
                if (tok < 0) st = ROW_DEGENERATE;
            }
            emit_spec_warp(P, b, st, pl.A, tok);
        }
        t = next;
    }
}

// Chunk kernel for 16-byte vectors: one CTA per (request, chunk of RCHUNK contiguous vectors of the
// selected row pair).  Thread t loads vectors t + i*NT (i < RCV) of both rows, U2 of each at a time
// into registers.  Each warp's 32 vectors of one i form one segment; the last CTA of a request draws
// the token.
constexpr int RCHUNK = NT * RCV;

// MODE: RES_PLAIN, RES_MASK (grammar mask applied to both rows) or RES_THR (top-p thresholds)
template <int DT, int MODE>
__global__ void __launch_bounds__(NT) spec_resample_chunk_kernel(SpecParams P)
{
    constexpr int VEC = (DT == DT_BF16) ? 8 : 4;
    __shared__ int sh_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / P.S2, c = blockIdx.x % P.S2;
    pdl_wait();  // the plan of the row-merge kernel
    const Plan pl = ld_plan(P.plan + b);
    const char* rowp = spec_row_ptr(P, b, pl.rp);
    const char* rowq = pl.rq >= 0 ? spec_row_ptr(P, b, pl.rq) : nullptr;
    const int c0 = c * RCHUNK;
    const int c1 = (int)min((long long)c0 + RCHUNK, P.nvec);
    if (pl.status == ROW_OK) {
        const uint64_t pol = policy_evict_first();
        float* segs = P.segs + (size_t)b * P.nseg;
#pragma unroll
        for (int it = 0; it < RCV / U2; ++it) {
            RawVec<DT, VEC> a[U2], q[U2];
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int v = c0 + (it * U2 + u) * NT + tid;
                a[u].w = make_uint4(0, 0, 0, 0);
                q[u].w = make_uint4(0, 0, 0, 0);
                if (v < c1) {
                    a[u].load(rowp, v, pol);
                    if (rowq) q[u].load(rowq, v, pol);
                    if constexpr (MODE == RES_MASK) {
                        const uint32_t bits = allowed_bits<VEC>(spec_mask_row(P, b, pl.rp), v);
                        mask_raw<DT, VEC>(a[u].w, bits);
                        mask_raw<DT, VEC>(q[u].w, bits);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U2; ++u) {
                const int seg0 = c0 + (it * U2 + u) * NT + warp * 32;
                const int v = seg0 + lane;
                float ls = 0.f;
                if (v < c1) {
                    float xp[VEC], xq[VEC], rv[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) { xp[e] = a[u].get(e); xq[e] = q[u].get(e); }
                    if constexpr (MODE == RES_THR) apply_thresholds<VEC>(xp, xq, rowq != nullptr, pl);
                    residual_from<VEC>(xp, xq, rowq != nullptr, pl, P.c, rv);
                    ls = tree_sum(rv);
                }
                const float ws = warp_sum(ls);
                if (lane == 0 && seg0 < c1) segs[seg0 / SEGV] = ws;
            }
        }
    }
    if (!arrive_last(&P.res_ctr[b], (unsigned)P.S2, &sh_flag)) return;
    if (warp == 0) {
        int st = pl.status, tok = -1;
        if (st == ROW_OK) {
            tok = draw_from_segments<DT, VEC>(P, b, pl, rowp, rowq);
            if (tok < 0) st = ROW_DEGENERATE;
        }
        emit_spec_warp(P, b, st, pl.A, tok);
    }
}

template <int DT, int VEC>
static void launch_softmax_plain(const SpecParams& P, int sms, cudaStream_t st)
{
    mark_kernel_start(st);
    spec_stats_kernel<DT, VEC><<<persistent_grid<spec_stats_kernel<DT, VEC>>(P.tasks1, sms), NT, 0, st>>>(P);
    mark_kernel_stop(st);
    spec_resample_kernel<DT, VEC><<<persistent_grid<spec_resample_kernel<DT, VEC>>(P.tasks2, sms), NT, 0, st>>>(P);
}

// the streaming kernel's grid: as many CTAs as fit, at most one per SPEC_GROUPS chunks
template <auto K>
static unsigned stream_grid(const SpecParams& P, int sms, int smem)
{
    return cta_grid<K>(((long long)P.B * P.R * P.S1 + SPEC_GROUPS - 1) / SPEC_GROUPS, sms, smem,
                       stream_threads<SPEC_GROUPS>());
}

template <int DT, int MASK>
static void launch_softmax_chunk(const SpecParams& P, int sms, cudaStream_t st)
{
    constexpr auto K1 = spec_stream_kernel<DT, MASK>;
    constexpr int smem = SPEC_GROUPS * (MASK == MASK_RING ? STREAM_SMEM_MASKED : STREAM_SMEM);
    mark_kernel_start(st);
    K1<<<stream_grid<K1>(P, sms, smem), stream_threads<SPEC_GROUPS>(), smem, st>>>(P);
    mark_kernel_stop(st);
    const int pw = (P.R <= 32) ? std::min(P.R, PLAN_WARPS) : WARPS;
    launch_dependent(spec_rowplan_kernel<DT>, (unsigned)P.B, (unsigned)(32 * pw), 0, st, P);
    launch_dependent(spec_resample_chunk_kernel<DT, MASK != MASK_NONE ? RES_MASK : RES_PLAIN>,
                     (unsigned)((long long)P.B * P.S2), NT, 0, st, P);
}

// Kernel 1 alone (the row statistics): the top-p path's first step.  The scalar variant also forms a
// plan, which the top-p kernels replace.
cudaError_t launch_softmax_stats(const SpecParams& P, int sms, cudaStream_t st)
{
    mark_kernel_start(st);
    if (P.vec > 1) {
        if (P.dtype == DT_BF16) {
            constexpr auto K1 = spec_stream_kernel<DT_BF16, MASK_NONE>;
            K1<<<stream_grid<K1>(P, sms, SPEC_GROUPS * STREAM_SMEM), stream_threads<SPEC_GROUPS>(),
                 SPEC_GROUPS * STREAM_SMEM, st>>>(P);
        } else {
            constexpr auto K1 = spec_stream_kernel<DT_F32, MASK_NONE>;
            K1<<<stream_grid<K1>(P, sms, SPEC_GROUPS * STREAM_SMEM), stream_threads<SPEC_GROUPS>(),
                 SPEC_GROUPS * STREAM_SMEM, st>>>(P);
        }
    } else if (P.dtype == DT_BF16) {
        spec_stats_kernel<DT_BF16, 1><<<persistent_grid<spec_stats_kernel<DT_BF16, 1>>(P.tasks1, sms), NT, 0, st>>>(P);
    } else {
        spec_stats_kernel<DT_F32, 1><<<persistent_grid<spec_stats_kernel<DT_F32, 1>>(P.tasks1, sms), NT, 0, st>>>(P);
    }
    mark_kernel_stop(st);
    return cudaGetLastError();
}

// Kernel 2 with the plan's top-p thresholds: the correction or bonus draw of the top-p path.
cudaError_t launch_softmax_resample_thr(const SpecParams& P, int sms, cudaStream_t st)
{
    if (P.vec > 1) {
        if (P.dtype == DT_BF16)
            return launch_dependent(spec_resample_chunk_kernel<DT_BF16, RES_THR>,
                                    (unsigned)((long long)P.B * P.S2), NT, 0, st, P);
        return launch_dependent(spec_resample_chunk_kernel<DT_F32, RES_THR>,
                                (unsigned)((long long)P.B * P.S2), NT, 0, st, P);
    }
    if (P.dtype == DT_BF16)
        spec_resample_kernel<DT_BF16, 1><<<persistent_grid<spec_resample_kernel<DT_BF16, 1>>(P.tasks2, sms), NT, 0, st>>>(P);
    else
        spec_resample_kernel<DT_F32, 1><<<persistent_grid<spec_resample_kernel<DT_F32, 1>>(P.tasks2, sms), NT, 0, st>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_softmax_path(const SpecParams& P, int sms, cudaStream_t st)
{
    const bool mask = P.mask != nullptr;
    // the mask bits can travel with the chunks when every mask row is a whole number of 16 bytes
    const bool ring_mask = mask && P.mwords % 4 == 0 && (reinterpret_cast<uintptr_t>(P.mask) & 15) == 0;
    if (P.dtype == DT_BF16 && P.vec == 8) {
        if (mask && ring_mask) launch_softmax_chunk<DT_BF16, MASK_RING>(P, sms, st);
        else if (mask) launch_softmax_chunk<DT_BF16, MASK_REGS>(P, sms, st);
        else launch_softmax_chunk<DT_BF16, MASK_NONE>(P, sms, st);
    } else if (P.dtype == DT_BF16) {
        launch_softmax_plain<DT_BF16, 1>(P, sms, st);
    } else if (P.vec == 4) {
        if (mask && ring_mask) launch_softmax_chunk<DT_F32, MASK_RING>(P, sms, st);
        else if (mask) launch_softmax_chunk<DT_F32, MASK_REGS>(P, sms, st);
        else launch_softmax_chunk<DT_F32, MASK_NONE>(P, sms, st);
    } else {
        launch_softmax_plain<DT_F32, 1>(P, sms, st);
    }
    return cudaGetLastError();
}

}  // namespace sv
