// sv_topp.cu -- exact speculative sampling with a top-p (nucleus) processor on p and q.
//
// "Exact speculative and assisted decoding for TinyRustLM": top-p is one of the declared processors
// that both distributions pass through before the ratio is formed; M7.1 section 0x03D: truncation
// keeps the round exact when q is the truncated distribution that sampled the draft.  A row keeps
// the tokens of largest probability, whole groups of equal stored logit at a time, until the kept
// mass (after temperature) first reaches top_p: the kept set is {v : x_v >= g}, and p is
// renormalised over it.
//
// Kernel 1: the plain path's row statistics (M, MC, S per chunk and warp).
// Kernel 2 (topp_row_kernel), one CTA per row: the row's M, MC and full mass S from kernel 1's
// partials, then the threshold g.  Masses are w = 2^y, y = x c - MC, and a kept set's mass is summed
// in fixed point (2^40 w rounded toward zero, integer sums: exact and order-free, so g does not
// depend on scheduling).
//   Fast path, one pass over the row that only compares: a vector whose largest stored logit reaches
//   the cut xcut = (MC - TOPP_CUT) / c (mass about 2^-14 of the row maximum's) is staged whole in its
//   warp's ring, and each time 32 are staged the warp takes them one per lane (so the element-wise
//   work runs on full warps).  The candidates are the elements at or above the cut.
//   - bf16 rows whose candidates take at most TOPP_BINS distinct stored values (the usual case):
//     a count per value, bin kM - key for the order key of the value and kM of the maximum.  A bin
//     is one value, so its mass is its count times that value's fixed-point mass; a scan from the
//     top finds the bin where the mass first reaches top_p * S, and that value is g.
//   - otherwise a candidate list in shared memory; the candidates' fixed-point masses fill
//     TOPP_BINS bins over y, the scan finds the crossing bin, and each of its candidates counts the
//     mass of larger and of equal logits in the bin, which places its group of equal logits: the
//     group that takes the kept mass to the target sets g.
//   Either way the kept mass is the sum through g's group.
//   Fallback (a candidate list that overflows, a crossing below the cut, a crowded crossing bin):
//   a mass-weighted radix select over the order-preserving key of the stored logits, four bits per
//   pass over the row, each pass adding the fixed-point masses of the elements that match the digits
//   chosen so far to the thread's own bin of its next digit.
// The row's lse, 1/S and log2 p(x) of the token it scores are then formed as on the plain path; the
// last CTA of a request runs the acceptance scan.
// Kernel 3: the plain path's residual pass with each row's threshold applied.
#include <type_traits>

#include "sv_plan.cuh"

namespace sv {

// Monotone key of a float (x < y iff key(x) < key(y)); -0 is folded into +0 first, since the two
// compare equal.
__device__ __forceinline__ uint32_t order_key(float x)
{
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// fast path geometry: candidates have y >= -TOPP_CUT (mass at least 2^-14 of the row maximum's);
// TOPP_BINS bins of width TOPP_CUT / TOPP_BINS over (-TOPP_CUT, 0] (anything lower in the last); the
// crossing bin is resolved when it holds at most TOPP_SORT candidates.  The candidate list takes TOPP_LIST bytes: stored bf16 bit
// patterns (2 bytes) or fp32 values (4 bytes).
constexpr float TOPP_CUT = 14.f;
constexpr int TOPP_LIST = 24576;
constexpr int TOPP_BINS = 2048;  // 16 KB of 64-bit masses
constexpr int TOPP_SORT = 512;  // (value, mass) pairs of the crossing bin, in the bins' space
constexpr int TOPP_RING = 64;   // staged 16-byte vectors per warp during the pass, in the bins' space
constexpr size_t TOPP_SMEM = TOPP_LIST + TOPP_BINS * sizeof(unsigned long long);
static_assert(16 * NT * sizeof(unsigned long long) <= TOPP_SMEM, "the radix bins share the space");
static_assert(WARPS * TOPP_RING * 16 <= TOPP_BINS * sizeof(unsigned long long), "the rings fit in the bins' space");
static_assert(TOPP_SORT * 2 * sizeof(unsigned long long) <= TOPP_BINS * sizeof(unsigned long long),
              "the crossing bin's pairs fit in the bins' space");

// order key of a bf16 bit pattern (16 bits; -0 folded into +0) and its inverse
__device__ __forceinline__ uint32_t key16(uint32_t h)
{
    return h == 0x8000u ? 0x8000u : (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
}
__device__ __forceinline__ float key16_float(uint32_t k)
{
    return __uint_as_float(((k & 0x8000u) ? (k ^ 0x8000u) : (~k & 0xffffu)) << 16);
}
// the bit pattern of the smallest bf16 value at or above the finite or infinite float f
__device__ __forceinline__ uint32_t bf16_ceil_bits(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u >> 16) + (((u & 0xffffu) != 0u && !(u & 0x80000000u)) ? 1u : 0u);
}

__device__ __forceinline__ int topp_bin(float y)
{
    const int k = (int)(-y * (TOPP_BINS / TOPP_CUT));
    return k < 0 ? 0 : (k >= TOPP_BINS ? TOPP_BINS - 1 : k);
}

// block-wide inclusive scan of 64-bit integers (thread order); returns the inclusive prefix
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    __syncthreads();
    if (lane == 31) sh[warp] = v;
    __syncthreads();
    unsigned long long before = 0ull;
    for (int w = 0; w < warp; ++w) before += sh[w];
    return before + v;
}

template <int DT, int VEC>
__global__ void __launch_bounds__(NT, 5) topp_row_kernel(SpecParams P)
{
    constexpr int KB = (DT == DT_BF16) ? 16 : 32;  // key bits that carry information
    using Cand = typename std::conditional<DT == DT_BF16, unsigned short, float>::type;
    constexpr int TOPP_CAP = TOPP_LIST / (int)sizeof(Cand);
    extern __shared__ __align__(16) unsigned long long dsm[];
    unsigned long long* hist = dsm;                         // radix fallback: digit-major, one column per thread
    Cand* cand = reinterpret_cast<Cand*>(dsm);              // fast path: candidates' stored logits
    unsigned long long* bins = dsm + TOPP_LIST / 8;         // fast path: fixed-point mass per bin
    auto cval = [&](int i) -> float {
        if constexpr (DT == DT_BF16) return __uint_as_float(((uint32_t)cand[i]) << 16);
        else return cand[i];
    };
    __shared__ unsigned long long tot[16];
    __shared__ unsigned long long wsum[WARPS];
    __shared__ int sh_n, sh_nk, sh_fast, sh_kb;
    __shared__ unsigned long long sh_above_kb;
    __shared__ float sh_thr;
    __shared__ float sh_M;
    __shared__ DFloat sh_S;
    __shared__ int sh_st;
    __shared__ uint32_t sh_prefix;
    __shared__ unsigned long long sh_above, sh_kept;
    __shared__ double sh_target;
    __shared__ int sh_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned FULL = 0xffffffffu;
    const int row_id = blockIdx.x, b = row_id / P.R, r = row_id - b * P.R, g = P.gamma;
    const char* row = spec_row_ptr(P, b, r);

    // the token this row scores and its logit: inputs, read before waiting for kernel 1
    const int pos = (r < g) ? r : (r > g) ? r - g - 1 : -1;
    const int tok = (pos >= 0) ? __ldg(P.tokens + (size_t)b * g + pos) : -1;
    const bool tok_ok = tok >= 0 && tok < P.V;
    const float xtok = tok_ok ? load_logit(row, DT, tok) : 0.f;
    pdl_wait();  // the partials of kernel 1

    // ---- the row's maximum and full mass (warp 0), as on the plain path
    if (warp == 0) {
        const int np = P.vec > 1 ? P.S1 * WARPS : P.S1;
        const Partial* pp = P.partials + (size_t)row_id * np;
        float Mr = NEG_INF;
        for (int k = lane; k < np; k += 32) Mr = fmaxf(Mr, __ldcg(&pp[k].M));
        Mr = warp_max(Mr);
        const float MCr = __fmul_rn(Mr, P.c);
        DFloat S = df_make(0.f, 0.f);
        int tmo = 0;
        for (int k = lane; k < np; k += 32) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(pp + k));
            if (q.z < 0.f) tmo = 1;
            if (q.z != 0.f) S = df_add(S, df_make(__fmul_rn(q.z, ex2(q.y - MCr)), 0.f));
        }
        S = warp_sum_df(S);
        tmo = __any_sync(FULL, tmo);
        if (lane == 0) {
            const bool ok = !tmo && isfinite(S.hi) && S.hi > 0.f && Mr != NEG_INF && isfinite(Mr);
            sh_M = Mr;
            sh_S = S;
            sh_st = tmo ? ROW_TIMEOUT : ok ? ROW_OK : ROW_NONFINITE;
            sh_prefix = 0;
            sh_above = 0;
        }
    }
    __syncthreads();
    const float M = sh_M, MC = __fmul_rn(M, P.c);
    float thr = NEG_INF;
    DFloat S = sh_S;

    // ---- the nucleus threshold, fast path: one pass, a candidate list and mass bins
    bool fast = false;
    const bool select = sh_st == ROW_OK && P.top_p < 1.0f;
    // the cut on the stored logit: x >= xcut is (up to rounding) y >= -TOPP_CUT; whatever the
    // rounding, the candidates are every element at or above one value, which is all the select
    // needs (it checks that the crossing lies among them)
    const float xcut = __fdiv_rn(MC - TOPP_CUT, P.c);
    // bf16 rows whose candidates take at most TOPP_BINS distinct stored values (order keys kc to
    // kM): a bin per value, counted during the pass (in the list's space), and no list
    bool exact = false;
    uint32_t kM = 0u;
    if constexpr (DT == DT_BF16) {
        kM = key16(__float_as_uint(M) >> 16);
        const uint32_t kc = key16(bf16_ceil_bits(xcut));
        exact = select && kc <= kM && kM - kc < (uint32_t)TOPP_BINS;
    }
    if (select) {
        uint32_t* cnt = reinterpret_cast<uint32_t*>(dsm);
        if (exact)
            for (int k = tid; k < TOPP_BINS; k += NT) cnt[k] = 0u;
        if (tid == 0) sh_n = 0;
        __syncthreads();
        // A vector that holds a candidate is staged whole in its warp's ring (the bins' space, free
        // until the pass ends); each time 32 are staged the warp takes them one per lane, so the
        // element-wise work runs on full warps instead of on the few lanes that found one.
        uint4* ring = reinterpret_cast<uint4*>(bins) + warp * TOPP_RING;
        int head = 0, tail = 0;  // warp-uniform positions in the ring
        auto take = [&](bool valid, uint4 w) {
            RawVec<DT, VEC> rv;
            rv.w = w;
            unsigned cm = 0u;
#pragma unroll
            for (int e = 0; e < VEC; ++e) cm |= (valid && rv.get(e) >= xcut ? 1u : 0u) << e;
            if constexpr (DT == DT_BF16) {
                if (exact) {  // a candidate's key lies in [kc, kM]: its bin is kM - key
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if ((cm >> e) & 1u) {
                            const uint32_t wd = VEC == 1 ? w.x : (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
                            const uint32_t h = (VEC == 1 || (e & 1)) ? (wd >> 16) : (wd & 0xffffu);
                            atomicAdd(&cnt[kM - key16(h)], 1u);
                        }
                    }
                    return;
                }
            }
            const int k = __popc(cm);
            int incl = k;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            int base = 0;
            if (lane == 31 && incl > 0) base = atomicAdd(&sh_n, incl);
            int at = __shfl_sync(FULL, base, 31) + incl - k;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if ((cm >> e) & 1u) {
                    if (at < TOPP_CAP) {
                        if constexpr (VEC == 1) {
                            if constexpr (DT == DT_BF16) cand[at] = (unsigned short)(w.x >> 16);
                            else cand[at] = __uint_as_float(w.x);
                        } else {
                            const uint32_t wd = (DT == DT_BF16 ? (e >> 1) : e) == 0 ? w.x
                                              : (DT == DT_BF16 ? (e >> 1) : e) == 1 ? w.y
                                              : (DT == DT_BF16 ? (e >> 1) : e) == 2 ? w.z : w.w;
                            if constexpr (DT == DT_BF16) cand[at] = (unsigned short)((e & 1) ? (wd >> 16) : (wd & 0xffffu));
                            else cand[at] = __uint_as_float(wd);
                        }
                    }
                    ++at;
                }
            }
        };
        const unsigned below_me = (1u << lane) - 1u;
        constexpr int UL = 4;  // vectors per thread in flight
        constexpr int STEP = NT * UL;  // vectors per iteration of the CTA
        const int vend = (int)P.nvec;  // a row has fewer than 2^31 vectors
        for (int v0 = 0; v0 < vend; v0 += STEP) {
            RawVec<DT, VEC> rv[UL];
#pragma unroll
            for (int u = 0; u < UL; ++u) {
                const int v = v0 + u * NT + tid;
                if (v < vend) rv[u].load(row, v, policy_evict_first());
                else rv[u].fill_neg_inf();
            }
#pragma unroll
            for (int u = 0; u < UL; ++u) {
                // the vector's maximum against the cut (NaN never reaches here: the row is finite)
                float vm;
                if constexpr (VEC == 1) {
                    vm = rv[u].get(0);
                } else if constexpr (DT == DT_BF16) {
                    const uint32_t pm = bmax2(bmax2(rv[u].w.x, rv[u].w.y), bmax2(rv[u].w.z, rv[u].w.w));
                    vm = fmaxf(bf16lo(pm), bf16hi(pm));
                } else {
                    vm = fmaxf(fmaxf(rv[u].get(0), rv[u].get(1)), fmaxf(rv[u].get(2), rv[u].get(3)));
                }
                const bool hot = vm >= xcut;
                const unsigned hm = __ballot_sync(FULL, hot);
                if (hm) {
                    if (hot) ring[(tail + __popc(hm & below_me)) & (TOPP_RING - 1)] = rv[u].w;
                    tail += __popc(hm);
                    if (tail - head >= 32) {
                        __syncwarp();
                        take(true, ring[(head + lane) & (TOPP_RING - 1)]);
                        head += 32;
                        __syncwarp();
                    }
                }
            }
        }
        // what is left in the ring (fewer than 32)
        __syncwarp();
        if (tail > head) take(head + lane < tail, ring[(head + lane) & (TOPP_RING - 1)]);
        __syncthreads();
        // exact: bin k holds the count of value key16_float(kM - k) times that value's mass
        for (int k = tid; k < TOPP_BINS; k += NT) {
            unsigned long long m = 0ull;
            if (exact) {
                const uint32_t ck = cnt[k];
                if (ck) m = (unsigned long long)ck * fixed_mass(ex2(fmaf(key16_float(kM - (uint32_t)k), P.c, -MC)));
            }
            bins[k] = m;
        }
        __syncthreads();
        const int n = sh_n;
        if (n <= TOPP_CAP) {
            // fixed-point masses of the candidates into the bins
            for (int i = tid; i < n; i += NT) {
                const float y = fmaf(cval(i), P.c, -MC);
                atomicAdd(&bins[topp_bin(y)], fixed_mass(ex2(y)));
            }
            __syncthreads();
            // the row's total mass (every element; the stream's pairs of floats) in 2^-40 units
            const double target = (double)P.top_p * (df_to_double(S) * FIXED_ONE);
            // the crossing bin: thread t holds bins [8t, 8t + 8)
            constexpr int BPT = TOPP_BINS / NT;
            unsigned long long loc[BPT], s = 0ull;
#pragma unroll
            for (int j = 0; j < BPT; ++j) {
                loc[j] = bins[tid * BPT + j];
                s += loc[j];
            }
            const unsigned long long incl = block_scan_u64(s, wsum);
            if (tid == 0) sh_kb = -1;
            __syncthreads();
            const unsigned long long run0 = incl - s;
            if ((double)incl >= target && (double)run0 < target) {
                // the first of this thread's bins whose mass, with all above it, reaches the target
                // (unrolled without an early exit, so that loc stays in registers)
                int jc = -1;
                unsigned long long acc = run0, above = 0ull;
#pragma unroll
                for (int j = 0; j < BPT; ++j) {
                    if (jc < 0 && (double)(acc + loc[j]) >= target) {
                        jc = j;
                        above = acc;
                    }
                    acc += loc[j];
                }
                const int kbin = tid * BPT + jc;  // jc >= 0: the thread's total reaches the target
                sh_kb = kbin;
                sh_above_kb = above;
                if (exact) {  // the bin is one value: the threshold group itself
                    sh_thr = key16_float(kM - (uint32_t)kbin);
                    sh_kept = above + bins[kbin];
                }
            }
            __syncthreads();
            const int kb = sh_kb;
            if (exact) {
                fast = kb >= 0;
            } else if (kb >= 0) {
                // the crossing bin's candidates as (value, mass) pairs in the bins' space
                unsigned long long* pairs = bins;
                if (tid == 0) sh_nk = 0;
                __syncthreads();
                for (int i = tid; i < n; i += NT) {
                    const float xi = cval(i);
                    const float y = fmaf(xi, P.c, -MC);
                    if (topp_bin(y) == kb) {
                        const int at = atomicAdd(&sh_nk, 1);
                        if (at < TOPP_SORT) {
                            pairs[2 * at] = (unsigned long long)order_key(xi);
                            pairs[2 * at + 1] = fixed_mass(ex2(y));
                        }
                    }
                }
                __syncthreads();
                const int nk = sh_nk;
                if (nk <= TOPP_SORT) {
                    // each pair finds its group's place by counting: the mass above the group (larger
                    // keys) and the group's own (equal keys); the one group that takes the kept mass
                    // from below the target to at least it sets the threshold (its members all write
                    // the same values)
                    if (tid == 0) sh_fast = 0;
                    __syncthreads();
                    for (int i = tid; i < nk; i += NT) {
                        const unsigned long long key = pairs[2 * i];
                        unsigned long long gt = 0ull, eq = 0ull;
                        for (int j = 0; j < nk; ++j) {
                            const unsigned long long kj = pairs[2 * j], mj = pairs[2 * j + 1];
                            gt += kj > key ? mj : 0ull;
                            eq += kj == key ? mj : 0ull;
                        }
                        const unsigned long long before = sh_above_kb + gt, through = before + eq;
                        if ((double)before < target && (double)through >= target) {
                            sh_thr = key_float((uint32_t)key);
                            sh_kept = through;
                            sh_fast = 1;
                        }
                    }
                    __syncthreads();
                    fast = sh_fast != 0;
                }
            }
        }
        __syncthreads();
    }
    if (fast) {
        thr = sh_thr;
        S = fixed_to_df(sh_kept);
    }

    // ---- the nucleus threshold, fallback: a radix select on the key, weighted by fixed-point mass
    if (!fast && sh_st == ROW_OK && P.top_p < 1.0f) {
        if (tid == 0) {
            sh_prefix = 0;
            sh_above = 0;
        }
        __syncthreads();
        for (int lvl = 0; lvl < KB / 4; ++lvl) {
            const int shift = 32 - 4 * (lvl + 1);  // this level's digit of the 32-bit key
            const uint32_t prefix = sh_prefix;
#pragma unroll
            for (int d = 0; d < 16; ++d) hist[d * NT + tid] = 0ull;
            // consecutive elements of a thread mostly share a digit: their masses are added in a
            // register and reach the thread's bin when the digit changes
            unsigned long long run = 0ull;
            int cur = 0;
            for (long long v = tid; v < P.nvec; v += NT) {
                float x[VEC];
                load_vec<DT, VEC>(row, v, x);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const uint32_t key = order_key(x[e]);
                    if (lvl == 0 || (key >> (shift + 4)) == prefix) {
                        const int d = (int)((key >> shift) & 15u);
                        const unsigned long long fx = fixed_mass(ex2(fmaf(x[e], P.c, -MC)));
                        if (d != cur) {
                            hist[cur * NT + tid] += run;
                            cur = d;
                            run = fx;
                        } else {
                            run += fx;
                        }
                    }
                }
            }
            hist[cur * NT + tid] += run;
            __syncthreads();
            // digit totals: warp w adds the columns of digits 2w and 2w + 1
            for (int d = 2 * warp; d < 2 * warp + 2; ++d) {
                unsigned long long s = 0ull;
                for (int t = lane; t < NT; t += 32) s += hist[d * NT + t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
                if (lane == 0) tot[d] = s;
            }
            __syncthreads();
            if (tid == 0) {
                if (lvl == 0) {
                    unsigned long long all = 0ull;
                    for (int d = 0; d < 16; ++d) all += tot[d];
                    sh_target = (double)P.top_p * (double)all;
                }
                // the largest digit whose mass, with everything above it, reaches the target
                unsigned long long above = sh_above;
                int dsel = 0;
                for (int d = 15; d >= 0; --d) {
                    if ((double)(above + tot[d]) >= sh_target || d == 0) {
                        dsel = d;
                        break;
                    }
                    above += tot[d];
                }
                sh_above = above;
                sh_kept = above + tot[dsel];
                sh_prefix = (prefix << 4) | (uint32_t)dsel;
            }
            __syncthreads();
        }
        // the threshold's full key: for bf16 the low 16 bits of a key are all 0 (x >= 0) or all 1
        uint32_t gk = sh_prefix << (32 - KB);
        if (KB < 32 && !(gk & 0x80000000u)) gk |= (1u << (32 - KB)) - 1u;
        thr = key_float(gk);
        // the kept mass as a pair of floats (2^-40 units, exact in fp64 up to 2^53)
        S = fixed_to_df(sh_kept);
    }

    // ---- the row's statistics, as the plain path's row plan forms them
    if (tid == 0) {
        RowStats st = blank_rowstats();
        st.M = M;
        st.MC = MC;
        st.S = (double)S.hi;
        st.status = sh_st;
        st.lse = __int_as_float(0x7fc00000);
        st.lx_hi = __int_as_float(0x7fc00000);
        st.lx_lo = 0.f;
        if (sh_st == ROW_OK) {
            row_norm(st, M, MC, S, P, tok_ok, xtok, thr);
            st.thr = thr;
        }
        P.rstats[row_id] = st;
    }
    // ---- the last row of the request: the acceptance scan
    if (!arrive_last(&P.dense_ctr[b], (unsigned)P.R, &sh_flag)) return;
    if (warp == 0) {
        const Plan pl = compute_plan_warp<DT, true>(P, b, true);
        if (lane == 0) P.plan[b] = pl;
    }
}

cudaError_t launch_topp_path(const SpecParams& P, int sms, cudaStream_t st)
{
    cudaError_t e = launch_softmax_stats(P, sms, st);
    if (e != cudaSuccess) return e;
    const unsigned rows = (unsigned)((long long)P.B * P.R);
    set_smem_limit<topp_row_kernel<DT_BF16, 8>>(TOPP_SMEM);
    set_smem_limit<topp_row_kernel<DT_BF16, 1>>(TOPP_SMEM);
    set_smem_limit<topp_row_kernel<DT_F32, 4>>(TOPP_SMEM);
    set_smem_limit<topp_row_kernel<DT_F32, 1>>(TOPP_SMEM);
    if (P.dtype == DT_BF16)
        e = P.vec > 1 ? launch_dependent(topp_row_kernel<DT_BF16, 8>, rows, NT, TOPP_SMEM, st, P)
                      : launch_dependent(topp_row_kernel<DT_BF16, 1>, rows, NT, TOPP_SMEM, st, P);
    else
        e = P.vec > 1 ? launch_dependent(topp_row_kernel<DT_F32, 4>, rows, NT, TOPP_SMEM, st, P)
                      : launch_dependent(topp_row_kernel<DT_F32, 1>, rows, NT, TOPP_SMEM, st, P);
    if (e != cudaSuccess) return e;
    return launch_softmax_resample_thr(P, sms, st);
}

}  // namespace sv
