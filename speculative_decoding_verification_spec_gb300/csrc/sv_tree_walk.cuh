// sv_tree_walk.cuh -- the walk over a candidate tree shared by greedy tree verify (sv_tree.cu) and
// typical-acceptance tree verify (sv_typical.cu).
//
// Module 16 "Verify the Tree": a node is valid when it passes its own test against its predictor
// row and its parent is valid; the deepest valid node is accepted with its root path, and one more
// token follows the path.  M7.7 section 0x07E: a depth-1 node is scored by the frontier row (row 0),
// any other node by its parent's row (parent + 1).  The tests differ: greedy compares the token
// with the predictor row's argmax, typical acceptance compares its probability with an entropy
// threshold.
#pragma once

#include "sv_common.cuh"

namespace sv {

struct TreeWalk {
    int st;     // ROW_OK or the request's status
    int depth;  // depth of the accepted node (0: none)
    int node;   // the accepted node, -1 when none is valid
};

// One warp: validates the request's tree, finds every node's validity and depth, picks the deepest
// valid node (lowest index on ties).  par / tok are the request's parent and token arrays (par
// null: a chain, node i's parent is i - 1), depth / valid N-int scratch (global or shared memory).
// match(i, p) is node i's own test given its parent p (p = -1 at depth 1); it is only asked for
// trees whose parents and tokens are in range.
//   bad: 0, 1 (a row is non-finite) or 2 (a row could not be read);
//   late: a status that ranks after the parent and token checks (0 when none).
// Every lane returns the same result; OVERFLOW when the path and one more token exceed max_out.
//
// Nodes are taken 32 at a time in index order, one per lane.  A node whose parent lies in an
// earlier group reads the parent's final validity and depth; within a group the values move from
// parent to child by ballot / shuffle until nothing changes (parents precede children, so this
// settles after as many rounds as the group's longest chain).
template <class Match>
__device__ __forceinline__ TreeWalk tree_walk(int N, int V, int max_out, int bad, int late,
                                              const int32_t* par, const int32_t* tok, Match match,
                                              int32_t* depth, int32_t* valid)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    int st = (bad == 2) ? ROW_TIMEOUT : bad ? ROW_NONFINITE : ROW_OK;
    if (st == ROW_OK) {
        int badp = 0, badt = 0;
        for (int i = lane; i < N; i += 32) {
            const int p = par ? par[i] : i - 1;
            if (p < -1 || p >= i) badp = 1;
            const int tk = tok[i];
            if (tk < 0 || tk >= V) badt = 1;
        }
        badp = __any_sync(FULL, badp);
        badt = __any_sync(FULL, badt);
        st = badp ? ROW_BAD_PARENT : (badt ? ROW_BAD_TOKEN : late ? late : ROW_OK);
    }
    int bestd = 0, bestn = -1;
    if (st == ROW_OK) {
        for (int i0 = 0; i0 < N; i0 += 32) {
            const int i = i0 + lane;
            const bool in = i < N;
            const int p = !in ? -1 : par ? par[i] : i - 1;
            const bool local = p >= i0;  // the parent is in this group
            const int m = in && match(i, p);
            int v = 0, dd = 0;
            if (in && !local) {
                v = m && (p < 0 || valid[p]);
                dd = p < 0 ? 1 : depth[p] + 1;
            }
            for (int round = 0; round < 32; ++round) {
                const unsigned vm = __ballot_sync(FULL, v);
                const int pd = __shfl_sync(FULL, dd, local ? p - i0 : lane);
                int nv = v, nd = dd;
                if (in && local) {
                    nv = m && ((vm >> (p - i0)) & 1u);
                    nd = pd > 0 ? pd + 1 : 0;
                }
                if (!__any_sync(FULL, nv != v || nd != dd)) break;
                v = nv;
                dd = nd;
            }
            if (in) {
                valid[i] = v;
                depth[i] = dd;
                if (v && dd > bestd) { bestd = dd; bestn = i; }
            }
            __syncwarp();
        }
        // deepest valid node, lowest index on ties
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const int od = __shfl_xor_sync(FULL, bestd, o);
            const int on = __shfl_xor_sync(FULL, bestn, o);
            if (od > bestd || (od == bestd && on >= 0 && (bestn < 0 || on < bestn))) {
                bestd = od;
                bestn = on;
            }
        }
        if (bestd + 1 > max_out) st = ROW_OVERFLOW;
    }
    TreeWalk w;
    w.st = st;
    w.depth = bestd;
    w.node = bestn;
    return w;
}

// One warp: the outputs of request b from its walk: accepted_len, row_status, the path's tokens
// (and node ids) followed by final_tok, then -1; a request whose status is not OK emits -1 only.
__device__ __forceinline__ void tree_emit(const TreeParams& P, int b, const TreeWalk& w,
                                          const int32_t* par, const int32_t* tok, int final_tok)
{
    const int lane = threadIdx.x & 31;
    const int mo = P.max_out;
    int32_t* out = P.out_tokens + (size_t)b * mo;
    int32_t* onodes = P.out_nodes ? P.out_nodes + (size_t)b * (mo - 1) : nullptr;
    if (lane == 0) {
        P.accepted_len[b] = (w.st == ROW_OK) ? w.depth : -1;
        if (P.row_status) P.row_status[b] = w.st;
        if (w.st == ROW_OK) {  // path written back to front, then the final token
            int n = w.depth;
            out[n] = final_tok;
            for (int i = w.node; i >= 0; i = par ? par[i] : i - 1) {
                --n;
                out[n] = tok[i];
                if (onodes) onodes[n] = i;
            }
        }
    }
    const int A = (w.st == ROW_OK) ? w.depth : -1;
    for (int i = lane; i < mo; i += 32) {
        if (w.st != ROW_OK || i > A) out[i] = -1;
        if (onodes && i < mo - 1 && (w.st != ROW_OK || i >= A)) onodes[i] = -1;
    }
}

}  // namespace sv
