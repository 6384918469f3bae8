/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding verify library.
 *
 * Three verify calls, each one pass of the target-side verify step over a batch of B independent
 * requests, entirely on the GPU:
 *
 *   spec_verify        exact speculative sampling with temperature
 *   spec_verify_topk   the same with a top-k processor applied identically to target and draft
 *   spec_verify_masked the same with a grammar mask (a valid-token set per position)
 *   spec_verify_topp   the same with a top-p (nucleus) processor applied identically to target and draft
 *   tree_verify_greedy Medusa-style greedy verification of a candidate tree
 *   spec_verify_greedy linear greedy verification of a draft (the greedy tree on a chain)
 *   tree_verify_sample stochastic verification of a candidate tree (residual update over children)
 *   tree_verify_typical Medusa-style tree verification by typical acceptance (entropy threshold)
 *   smc_verify         the verify side of one SMC-SD round: block weights, extension, resampling
 *
 * Sources (page title + section):
 *   "M7.1 - Speculative Decoding: Draft, Verify, Accept, Reject": 0x03 (accept probability and
 *     correction distribution), 0x03C-0x03D (positive residual, support and numerical cases),
 *     0x03G (stop at the first rejection), 0x03H (bonus token), 0x04 (round loop), 0x04J (online
 *     (m, l) merge over vocabulary blocks).
 *   Module 16 speculative-decoding lesson: "The Math: Speculative Sampling" (accept iff
 *     u < min(1, p(x)/q(x))), "Verify the Tree -- and Why It's Exact" (greedy tree walk).
 *   "M7.7 - Draft Sources, Dependent Heads, Hardware-Aware Trees": 0x07E (candidate row vs
 *     predictor row: a depth-1 node is scored by the frontier row, any other node by its
 *     parent's row), 0x08B-0x09A (several candidates at one node: test them in turn against the
 *     running residual, never against the original target row).
 *   Module 16 lesson, "SMC Speculative Decoding: Resample, Don't Reject": "The Math: Reweight, Don't
 *     Reject" (block weight, effective sample size, Algorithm 1), "Two Exact Anchors".
 *   "Exact speculative and assisted decoding for TinyRustLM": "Normative stochastic pseudocode"
 *     (separate accept / correction / extra-token random streams, abort without emitting on
 *     non-finite rows or a non-positive residual), "Minimum target API" (row i predicts proposal
 *     i, the last row predicts the extra token).
 *
 * Conventions shared by every call:
 *   - All tensors are dense, row-major, vocabulary (V) fastest.  Logits are bf16 (raw 16-bit
 *     patterns) or fp32 (spec_dtype).  Any alignment works; rows whose start is 16-byte aligned
 *     are read with 16-byte vector loads.
 *   - Every pointer passed to a verify call is a DEVICE pointer owned by the caller.  The library
 *     allocates nothing and never modifies inputs.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream); all work is enqueued asynchronously on it and the host never waits.
 *   - `workspace` is caller-owned device scratch of at least spec_workspace_bytes(...) bytes,
 *     16-byte aligned.  Its contents need no initialisation: each call first clears the few
 *     completion counters it uses (one cudaMemsetAsync on `stream`), then launches its kernels.
 *     Calls that share a workspace must not overlap on the GPU (issue them on one stream).
 *   - Call-level status (the return value) covers what the host can check: sizes, temperature,
 *     top_k, null or misaligned pointers, workspace size, and CUDA launch errors.  Per-request
 *     conditions found on the device are reported in row_status[b] (SPEC_ROW_*); such a request
 *     emits nothing: accepted_len[b] = -1 and every out_tokens entry of the request is -1.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* a size, temperature, top_k or pointer failed host validation */
    SPEC_ERR_CUDA = 2,        /* a CUDA launch, memset or attribute call failed */
    SPEC_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or smaller than required */
    SPEC_ERR_TOO_LARGE = 4    /* spec_verify_noalloc: the sizes need more scratch than its fixed
                                 device array holds (SPEC_NOALLOC_SCRATCH_BYTES) */
} spec_status;

/* Per-request status codes written to row_status[b]. */
enum {
    SPEC_ROW_OK = 0,
    SPEC_ROW_NONFINITE = 1,            /* a logit row of the request holds NaN or +inf, or has no
                                          finite entry left after the processors */
    SPEC_ROW_DEGENERATE_RESIDUAL = 2,  /* the correction residual mass is not positive */
    SPEC_ROW_BAD_TOKEN = 3,            /* a draft / node token is outside [0, V), or a drafted
                                          token has q(x) = 0 (it cannot have been sampled) */
    SPEC_ROW_TIMEOUT = 4,              /* a bounded wait inside a streaming kernel ran out (a
                                          bulk copy or a peer warp of the same CTA did not arrive
                                          within its limit of polls, see spec_set_wait_limit): the
                                          request is abandoned and emits nothing */
    SPEC_ROW_BAD_PARENT = 5,           /* tree: parents[b,i] is not in [-1, i) */
    SPEC_ROW_OUTPUT_OVERFLOW = 6,      /* tree: accepted path + bonus does not fit in max_out */
    SPEC_ROW_BAD_UNIFORM = 7,          /* a uniform of the request is not in [0, 1) */
    SPEC_ROW_BAD_PROPOSAL_ROW = 8      /* tree_verify_sample: qrow[b,i] is not in [0, Nq) */
};

/*
 * Bytes of workspace needed by one call.
 *   spec_verify:        spec_workspace_bytes(B, gamma, V, 0, 0)
 *   spec_verify_topk:   spec_workspace_bytes(B, gamma, V, top_k, 0)
 *   spec_verify_masked: spec_workspace_bytes(B, gamma, V, 0, 0)   (as spec_verify)
 *   spec_verify_topp:   spec_workspace_bytes(B, gamma, V, 0, 0)   (as spec_verify)
 *   tree_verify_greedy: spec_workspace_bytes(B, 0, V, 0, N)   (tree_nodes = N > 0)
 *   tree_verify_typical: spec_workspace_bytes(B, 0, V, 0, N)  (as tree_verify_greedy)
 * The value is an upper bound valid for both dtypes, any alignment and any GPU.
 * Returns 0 for invalid sizes.
 */
size_t spec_workspace_bytes(int B, int gamma, int V, int top_k, int tree_nodes);

/*
 * Exact speculative sampling verify (M7.1 0x03-0x04; Module 16 accept rule).
 *
 *   target_logits [B, gamma+1, V]  row i < gamma scores draft token i; row gamma scores the
 *                                  bonus position after the whole draft
 *   draft_logits  [B, gamma, V]    row i is the draft row that sampled draft token i
 *                                  (may be NULL when gamma == 0)
 *   draft_tokens  [B, gamma]       int32
 *   uniforms      [B, gamma+2]     fp32 in [0, 1): slots 0..gamma-1 are the accept draws,
 *                                  slot gamma the correction draw, slot gamma+1 the bonus draw
 *   temperature   > 0, finite;     p = softmax(target/T), q = softmax(draft/T)
 *
 * With A = the first i such that u[b,i] >= min(1, p_i(x_i)/q_i(x_i)) (A = gamma if none):
 *   accepted_len[b] = A
 *   out_tokens[b, 0..A-1] = draft_tokens[b, 0..A-1]
 *   out_tokens[b, A]      = correction: inverse-CDF draw with u[b,gamma] from max(p_A - q_A, 0)
 *                           when A < gamma; bonus: inverse-CDF draw with u[b,gamma+1] from p_gamma
 *                           when A == gamma.  The draw is the smallest token v, in ascending
 *                           index order, whose running mass exceeds u * (total mass).
 *   out_tokens[b, A+1..gamma] = -1
 * Optional outputs (NULL to skip): row_status [B]; aux_lse_p [B, gamma+1] and aux_lse_q
 * [B, gamma] (natural-log normaliser of logits/T over the kept tokens); aux_accept [B, gamma]
 * (min(1, p_i(x_i)/q_i(x_i)) at every position, reached or not).
 */
spec_status spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                        const int32_t* draft_tokens, const float* uniforms,
                        int B, int gamma, int V, float temperature,
                        int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                        float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify with a top-k processor on both p and q (M7.1 0x03D: truncation keeps exactness when
 * q is the truncated distribution that sampled the draft).  Each row keeps every token whose
 * stored logit is >= the row's k-th largest stored logit (counted with multiplicity, signed zeros
 * equal), so ties at the threshold are all kept; the rest get probability 0.  top_k in [1, V];
 * top_k == V is identical to spec_verify.  Other arguments as spec_verify.
 */
spec_status spec_verify_topk(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* draft_tokens, const float* uniforms,
                             int B, int gamma, int V, float temperature, int top_k,
                             int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                             float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify with a top-p (nucleus) processor on every target and draft row ("Exact speculative
 * and assisted decoding for TinyRustLM": top-p is one of the declared processors both distributions
 * pass through before the ratio is formed; M7.1 0x03D: truncation keeps the round exact when q is
 * the truncated distribution that sampled the draft).  With p = softmax(logits / temperature), a row
 * keeps the tokens of largest probability, whole groups of equal stored logit at a time in
 * descending order, until the kept mass first reaches top_p; every token tied with the last group
 * kept stays in.  The kept set is {v : logit_v >= g} and p is renormalised over it; the same rule
 * applies to each draft row.  top_p > 0; top_p >= 1 is exactly spec_verify.  The kept mass is
 * summed in fixed point (2^-40 of the row maximum's mass per unit), so a row whose cumulative mass
 * lies within about 1e-7 of top_p may keep one group more or less than an exact computation would.
 * A drafted token outside its draft row's kept set is SPEC_ROW_BAD_TOKEN.  Other arguments, outputs
 * and statuses as spec_verify.
 */
spec_status spec_verify_topp(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                             const int32_t* draft_tokens, const float* uniforms,
                             int B, int gamma, int V, float temperature, float top_p,
                             int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                             float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify under a grammar mask ("Exact speculative and assisted decoding for TinyRustLM",
 * "Grammar and deterministic opportunities"): with A_G the valid-token set of the grammar state at
 * a position, both distributions of that position become
 *   p_G(x) = p(x) 1[x in A_G] / sum_v p(v) 1[v in A_G]      (q_G likewise),
 * and the round is exact relative to p_G when the draft sampled from q_G.
 *
 *   allowed [B, gamma+1, ceil(V/32)] uint32, device, 4-byte aligned: bit (v mod 32) of word v/32 of
 *           position i is set when token v is in A_G at position i.  Position i < gamma masks
 *           target row i and draft row i (the draft sampled token i in the same grammar state);
 *           position gamma masks the bonus row.  Bits of tokens >= V are ignored.
 *
 * A disallowed token is removed before its logit is read, so a NaN or +inf there is not seen.  A
 * drafted token outside A_G has q_G(x) = 0: SPEC_ROW_BAD_TOKEN.  A position whose A_G is empty
 * leaves its rows without mass: SPEC_ROW_NONFINITE.  Temperature only (no top-k); every other
 * argument, output and status as spec_verify.  allowed == NULL is SPEC_ERR_INVALID_ARG (B > 0).
 */
spec_status spec_verify_masked(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, const float* uniforms,
                               const uint32_t* allowed, int B, int gamma, int V, float temperature,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                               float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Greedy tree verify (Module 16 "Verify the Tree"; M7.7 0x07E row convention).
 *
 *   logits  [B, N+1, V]  row 0 = prefix-frontier logits, row i+1 = logits produced at node i
 *   parents [B, N]       int32, parents[b,i] in [-1, i) (-1: depth-1 node)
 *   tokens  [B, N]       int32 candidate token of each node
 *   max_out >= 1         length of an out_tokens row; must hold depth(best)+1 entries
 *
 * amax(row) = argmax over V, ties to the lowest index.  Node i is valid when tokens[i] ==
 * amax(predictor row of i) and its parent is valid.  The accepted node is the deepest valid node
 * (lowest index on ties); with none valid, nothing is accepted.
 *   accepted_len[b]                = depth of the accepted node (0 if none)
 *   out_tokens[b, 0..A-1]          = tokens on the root->node path; out_tokens[b, A] = amax of the
 *                                    accepted node's own row (row 0 if none); rest -1
 *   out_nodes [B, max_out-1]       = node ids on the path, then -1 (nullable)
 *   row_status [B]                 nullable
 */
spec_status tree_verify_greedy(const void* logits, spec_dtype dtype,
                               const int32_t* parents, const int32_t* tokens,
                               int B, int N, int V, int max_out,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                               int32_t* row_status, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Linear greedy verify (temperature -> 0; M7.1 "greedy = the p/q rule with one-hot p"; Module 16
 * "Verify the Tree": a chain is the degenerate tree): tree_verify_greedy on the chain
 * node i -> parent i - 1, with the target rows as the tree's rows.
 *
 *   target_logits [B, gamma+1, V]  row i scores draft token i; row gamma the position after the draft
 *   draft_tokens  [B, gamma]       int32
 *
 *   accepted_len[b] = A, the length of the longest prefix with draft_tokens[b, i] = argmax(row i)
 *   out_tokens[b, 0..A-1] = that prefix; out_tokens[b, A] = argmax(row A) (the correction, or the
 *   bonus when A = gamma); rest -1.  Ties go to the lowest index.  row_status as tree_verify_greedy.
 * Workspace: spec_workspace_bytes(B, 0, V, 0, max(gamma, 1)).
 */
spec_status spec_verify_greedy(const void* target_logits, spec_dtype dtype,
                               const int32_t* draft_tokens, int B, int gamma, int V,
                               int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Tree verify with typical acceptance (Module 16 "Verify the Tree": Medusa's sampling mode swaps
 * the greedy check for typical acceptance, which accepts a token when the target's probability
 * clears min(eps, delta exp(-H))).  Same tree layout as tree_verify_greedy:
 *   logits   [B, N+1, V]  row 0 = prefix frontier, row i+1 = produced at candidate node i
 *   parents  [B, N]       int32, -1 for a depth-1 node, else in [0, i)
 *   tokens   [B, N]       int32
 *   uniforms [B]          fp32 in [0, 1): the draw of the token after the accepted path
 * Row j's distribution is p_j = softmax(logits[b,j] / temperature), its entropy
 * H_j = -sum p_j ln p_j.  Node i passes when p_r(tokens[b,i]) > min(epsilon, delta exp(-H_r)),
 * strictly, r its predictor row (0 at depth 1, parents[b,i] + 1 otherwise); it is valid when it
 * passes and its parent is valid.  The deepest valid node (lowest index on ties) is accepted:
 *   accepted_len[b] = its depth (0 when no node is valid)
 *   out_tokens[b, 0..A-1] = the tokens on its root path, out_tokens[b, A] = a draw from p of the
 *   accepted node's own row (the frontier row when A = 0) by inverse CDF with uniforms[b] (the
 *   smallest token whose running mass exceeds u * total, ascending index), then -1 up to max_out.
 * out_nodes [B, max_out-1] (nullable): the path's node ids, then -1.  Optional (nullable):
 * row_status [B]; aux_entropy [B, N+1] (H_j); aux_logp [B, N] (ln p_r(tokens[b,i]), NaN when the
 * request has a bad row, parent or token).  temperature > 0; epsilon, delta >= 0 and finite
 * (epsilon = 0 passes every token with p > 0); N <= 2048; V <= 16384 * 32 * w, w = 8 (bf16) or
 * 4 (fp32) elements per 16-byte vector, 1 when rows are not 16-byte aligned.
 * Statuses: SPEC_ROW_NONFINITE (a row with NaN, +inf or no finite entry), then BAD_PARENT,
 * BAD_TOKEN, BAD_UNIFORM, OUTPUT_OVERFLOW (path + 1 > max_out).
 */
spec_status tree_verify_typical(const void* logits, spec_dtype dtype, const int32_t* parents,
                                const int32_t* tokens, const float* uniforms, int B, int N, int V,
                                float temperature, float epsilon, float delta, int max_out,
                                int32_t* accepted_len, int32_t* out_tokens, int32_t* out_nodes,
                                int32_t* row_status, float* aux_entropy, float* aux_logp,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stochastic tree verify (M7.7 0x09A residual update over a node's children; 0x07E row
 * convention; Module 16 accept rule and inverse-CDF draw).  Exact: the emitted tokens, continued
 * by target draws, follow the target distribution.
 *
 *   target_logits [B, N+1, V]  row 0 = prefix frontier, row i+1 = target logits at node i
 *   draft_logits  [B, Nq, V]   proposal rows (may be NULL when N == 0)
 *   parents       [B, N]       int32 in [-1, i): -1 for a depth-1 node
 *   tokens        [B, N]       int32 token of node i
 *   qrow          [B, N]       int32 in [0, Nq): node i's token was drawn from draft row qrow[b,i]
 *                              (i.i.d. siblings share a row; e.g. qrow = parent + 1 with the draft
 *                              rows laid out like the target rows)
 *   uniforms      [B, N+1]     fp32 in [0, 1): slot i = the accept test of node i, slot N = the
 *                              final draw.  Every slot is validated, tested or not.
 *   temperature   > 0, finite; p = softmax(target/T), q = softmax(draft/T)
 *   max_out >= 1               length of an out_tokens row; must hold the path plus one token
 *
 * The walk starts at the frontier with r = p of the current node's row and tests the node's
 * children in ascending index: child s with token x is accepted when u[s] < min(1, r(x)/q_s(x)),
 * and the walk moves to s (r is reset to p of s's row).  On rejection r becomes the normalised
 * positive part of r - q_s.  When every child is rejected the final token is drawn from r; at a
 * node without children it is the bonus, drawn from p.  The draw uses u[N] and picks the smallest
 * token whose running mass (ascending index) exceeds u * (total mass).
 *   accepted_len[b]          = path length (0 if the first node's children were all rejected)
 *   out_tokens[b, 0..A-1]    = tokens on the path; out_tokens[b, A] = the final token; rest -1
 *   out_nodes [B, max_out-1] = node ids on the path, then -1 (nullable)
 *   row_status [B] (nullable); aux_accept [B, N] (nullable): the ratio of every tested node, NaN
 *   for nodes the walk never tested.
 * Only the rows the walk visits are read: a NaN or +inf there gives SPEC_ROW_NONFINITE, one in a
 * row the walk never reaches goes unseen.  q_s(x) = 0 (a -inf draft logit at x) gives
 * SPEC_ROW_BAD_TOKEN when node s is tested; a path plus final token longer than max_out gives
 * SPEC_ROW_OUTPUT_OVERFLOW.  Limits: N <= 4096; V <= 262144 for bf16 and 131072 for fp32 (larger
 * sizes return SPEC_ERR_INVALID_ARG).  No workspace: each request is one thread-block cluster
 * whose state lives in shared memory.
 */
spec_status tree_verify_sample(const void* target_logits, const void* draft_logits,
                               spec_dtype dtype, const int32_t* parents, const int32_t* tokens,
                               const int32_t* qrow, const float* uniforms, int B, int N, int Nq,
                               int V, float temperature, int max_out, int32_t* accepted_len,
                               int32_t* out_tokens, int32_t* out_nodes, int32_t* row_status,
                               float* aux_accept, void* stream);

/*
 * The verify side of one SMC-SD round (Module 16 lesson, "SMC Speculative Decoding: Resample, Don't
 * Reject", Algorithm 1 steps 2-5) for `groups` groups of `particles` particles; B = groups *
 * particles requests, particle n of group g at request g * particles + n.  Not exact: the method
 * trades exactness for a fixed K+1 tokens per particle and round.
 *
 *   target_logits [B, K+1, V], draft_logits [B, K, V] (NULL when K == 0), draft_tokens [B, K]:
 *                              as spec_verify with gamma = K
 *   log_weights_in [B]         fp32 natural-log weight of each particle before the round
 *   uniforms      [B, 2]       fp32 in [0, 1): slot 0 draws the extension token, slot 1 the
 *                              particle's ancestor
 *   temperature                as spec_verify (no top-k)
 *   ess_threshold              eta: a group resamples when its ESS < eta (N/2 is the usual choice)
 *
 * Per particle, with p and q processed as in spec_verify and every draft position kept:
 *   block_log_ratio[b] = sum_j log p_j(d_j) - log q_j(d_j)                     (nullable)
 *   out_tokens[b, 0..K-1] = d_1 .. d_K; out_tokens[b, K] = the extension token, an inverse-CDF
 *   draw from p_K with slot 0; accepted_len[b] = K; row_status[b] (nullable) as spec_verify.
 * Per group, with w = exp(log_weights_in + block_log_ratio):
 *   ess[g] = (sum w)^2 / sum w^2                                                (nullable)
 *   ESS < eta: resampled[g] = 1; ancestors[b] = the inverse-CDF draw over the group's normalised
 *              weights (particle order) with slot 1 of particle b; log_weights_out = log(1/particles)
 *   otherwise: resampled[g] = 0; ancestors[b] = n; log_weights_out[b] = log w
 *   A group holding a particle whose status is not OK: ess NaN, resampled -1, ancestors -1 and
 *   log_weights_out NaN for all its particles (its OK particles keep their tokens and block ratio).
 * The caller copies the resampled particles (tokens, caches) from their ancestors.  Workspace:
 * spec_workspace_bytes(B, K, V, 0, 0).  particles <= 4096.
 */
spec_status smc_verify(const void* target_logits, const void* draft_logits, spec_dtype dtype,
                       const int32_t* draft_tokens, const float* log_weights_in,
                       const float* uniforms, int groups, int particles, int K, int V,
                       float temperature, float ess_threshold, int32_t* accepted_len,
                       int32_t* out_tokens, float* log_weights_out, float* block_log_ratio,
                       float* ess, int32_t* resampled, int32_t* ancestors, int32_t* row_status,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify for callers that cannot allocate device memory.  The paper has no counterpart: this
 * call only changes where spec_verify's scratch lives.
 *
 * Some callers may not call cudaMalloc at all -- a host that hands the library only pre-placed
 * buffers, code running under an allocator that forbids new device allocations, or a caller
 * that must not grow its memory footprint after start-up -- and so cannot provide the
 * `workspace` that spec_verify needs.  This call takes the same inputs and outputs as
 * spec_verify (device pointers owned by the caller) and runs the same kernels, but keeps the
 * scratch in a fixed array of SPEC_NOALLOC_SCRATCH_BYTES bytes inside the library, one per GPU,
 * held from the moment the library's code is loaded on that GPU until the process exits.
 *
 *   - Work runs on the calling thread's current device.  The first call on a device looks up
 *     the array's device address there (cudaGetSymbolAddress, which may load the library's code
 *     onto that device); make that first call before any stream capture on the device.
 *   - Sizes whose spec_workspace_bytes(B, gamma, V, 0, 0) exceeds SPEC_NOALLOC_SCRATCH_BYTES
 *     are rejected with SPEC_ERR_TOO_LARGE before anything is enqueued; other invalid
 *     arguments give the same status as spec_verify.
 *   - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Every call on a device shares that device's array, and the array keeps the previous
 *     call's contents.  Each call clears the counters it relies on before its kernels run, so
 *     stale contents are harmless, but calls that overlap on the GPU (different streams without
 *     ordering between them, or several host threads) race on the array and give wrong results.
 *     Issue them on one stream, or order them.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

spec_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                spec_dtype dtype, const int32_t* draft_tokens,
                                const float* uniforms, int B, int gamma, int V, float temperature,
                                int32_t* accepted_len, int32_t* out_tokens, int32_t* row_status,
                                float* aux_lse_p, float* aux_lse_q, float* aux_accept,
                                void* stream);

/*
 * Measurement aid.  With both events non-NULL (cudaEvent_t created by the caller), every later
 * verify call records `start` on its stream just before launching the call's dominant kernel and
 * `stop` just after it, so that the caller can time that kernel alone with cudaEventElapsedTime:
 *   spec_verify        the row-statistics (one-pass normaliser) kernel
 *   spec_verify_topk   the streaming top-k kernel
 *   tree_verify_greedy the argmax kernel
 *   spec_verify_greedy the argmax kernel, as tree_verify_greedy
 *   tree_verify_sample its only kernel
 *   smc_verify         the row-statistics kernel, as spec_verify
 * spec_set_kernel_events(NULL, NULL) turns it off.  The setting is process-wide and not
 * synchronised: set it from the thread that issues the calls.
 */
void spec_set_kernel_events(void* start, void* stop);

/*
 * Test aid: the number of polls after which a bounded wait of the streaming kernels gives up.
 *
 * The streaming kernels (spec_verify and its processors, spec_verify_topk, tree_verify_greedy,
 * spec_verify_greedy, tree_verify_typical, smc_verify) wait only inside one CTA, on mbarriers:
 * for a bulk copy of a chunk to land, for the CTA's consumer warps to free a ring stage, and
 * (top-k) for a segment's first bound and its completion.  Each such wait is bounded.  When one
 * runs out, the CTA stops reading, marks every chunk it has not read, still waits for its copies
 * in flight (always with the full default limit, so no CTA leaves while a copy could land) and
 * every request with an unread chunk reports SPEC_ROW_TIMEOUT with accepted_len = -1 and
 * out_tokens = -1: the request is abandoned without emitting ("Exact speculative and assisted
 * decoding for TinyRustLM", "Normative edge-case behavior").
 *
 *   polls  < 0: back to the default (2^22 polls, far beyond any healthy wait);
 *          0: every such wait gives up at once, so every request of a streaming call reports
 *             SPEC_ROW_TIMEOUT (how the tests reach this path without a fault);
 *          otherwise min(polls, 2^22).
 * Returns the previous limit.  Process-wide, read when a call is issued; not synchronised: set it
 * from the thread that issues the calls.  The scalar paths (rows not 16-byte aligned) and
 * tree_verify_sample do not wait and ignore it.
 */
int spec_set_wait_limit(int polls);

/*
 * Measurement aid: the cluster size of tree_verify_sample.  A request's walk runs on one
 * thread-block cluster of CL CTAs that split the vocabulary into CL slices ("M7.7 - Draft Sources,
 * Dependent Heads, Hardware-Aware Trees", 0x09A: every step of the walk needs the whole row).  By
 * default (cl = 0) CL is the smallest power of two whose slices hold a row in registers (4 16-byte
 * vectors per thread of 512), widened up to 8 while the GPU has an SM for every CTA.  cl = 1, 2, 4,
 * 8 or 16 forces that size instead; a call whose row does not fit the forced slices returns
 * SPEC_ERR_INVALID_ARG.  Any other value restores the default.  Returns the previous setting.
 * Process-wide, read when a call is issued; not synchronised.
 */
int spec_set_tree_sample_cluster(int cl);

/* Static description of a call-level status code. */
const char* spec_status_string(spec_status s);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
