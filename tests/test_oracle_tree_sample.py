"""Pins of the stochastic tree-verify oracle (residual update over a node's children).

What fixes the answer, from outside the oracle:
  - "M7.7 - Draft Sources, Dependent Heads, Hardware-Aware Trees", 0x09A: for p = (0.5, 0.3, 0.2)
    and two i.i.d. proposals from q = (0.4, 0.4, 0.2), enumerating every proposal pair, every
    accept/reject branch and the final draw gives the output marginal p; testing each candidate
    against the original p instead does not (a planted copy of the oracle shows the check fails).
  - the same page, 0x08B: k copies of a token that the target gives probability 1/2 must come out
    with probability 1/2, while independent re-tests give 1 - 2^-k.
  - exactness of speculative sampling: the emitted tokens, continued by target draws, follow the
    target's sequence law.  Checked by brute force over every token assignment of small trees whose
    rows come from a tiny next-token "model", and by a chi-square test with random uniforms.
  - special cases: a chain is the plain speculative-sampling round (the chain oracle, pinned on its
    own); an empty tree is one inverse-CDF draw from the frontier row.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
BELOW_ONE = np.nextafter(np.float32(1.0), np.float32(0.0))  # largest float32 uniform < 1


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def logp(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64))


# ------------------------------------------------------------------------------ exact branch law

def branch_law(target, draft, parents, tokens, qrow, T=1.0, lib=None):
    """Exact law {emitted sequence: probability} of one request with fixed tokens.

    The uniforms are integrated out exactly: an accept test of node s branches with the ratio a_s
    the oracle reports (forced by u = 0 / u just below 1), and the final draw is swept over its CDF
    intervals [lo, hi) reported by the oracle.  Tested nodes come in ascending index along the walk,
    so the first tested node without a decision is the next branch point.
    """
    N = len(parents)
    law = {}

    def call(u):
        r = O.tree_verify_sample(target[None], draft[None], [parents], [tokens], [qrow], [u], T,
                                 lib=lib)
        assert r["row_status"][0] == O.ROW_OK, r["row_status"][0]
        return r

    def go(decided, weight):
        u = np.zeros(N + 1, np.float32)
        for s, acc in decided.items():
            u[s] = 0.0 if acc else BELOW_ONE
        r = call(u)
        a = r["accept"][0]
        pending = [s for s in range(N) if not np.isnan(a[s]) and s not in decided]
        if pending:
            s = pending[0]
            if a[s] > 0:
                go({**decided, s: True}, weight * a[s])
            if a[s] < 1:
                assert a[s] <= BELOW_ONE, "ratio too close to 1 to force a rejection"
                go({**decided, s: False}, weight * (1.0 - a[s]))
            return
        uN = np.float32(0.0)
        total = 0.0
        while True:
            u[N] = uN
            r = call(u)
            lo, hi = r["draw_lo"][0], r["draw_hi"][0]
            L = r["accepted_len"][0]
            seq = tuple(int(t) for t in r["out_tokens"][0][: L + 1])
            law[seq] = law.get(seq, 0.0) + weight * (hi - lo)
            total += hi - lo
            if hi >= 1.0:
                break
            nu = np.float32(hi)
            if nu < hi:
                nu = np.nextafter(nu, np.float32(2.0))
            assert nu > uN
            uN = nu
        assert abs(total - 1.0) < 1e-12

    go({}, 1.0)
    return law


def first_token_law(law, V):
    out = np.zeros(V)
    for seq, w in law.items():
        out[seq[0]] += w
    return out


def iid_children_first_law(p, q, k, lib=None):
    """First-token law when the frontier row is p and k children are i.i.d. draws from q."""
    V = len(p)
    target = np.tile(logp(p), (k + 1, 1))  # node rows only matter for a bonus after acceptance
    draft = logp(q)[None, :]
    law = np.zeros(V)
    for xs in itertools.product(range(V), repeat=k):
        w = np.prod([q[x] for x in xs])
        if w == 0:
            continue
        bl = branch_law(target, draft, [-1] * k, list(xs), [0] * k, lib=lib)
        law += w * first_token_law(bl, V)
    return law


NAIVE_RETEST = [("double ratio = r[x] / q[x];", "double ratio = p[x] / q[x];")]


def test_page_example_two_children_marginal_is_p():
    g = gold("specinfer_children.json")["residual_update"]
    law = iid_children_first_law(np.array(g["target"]), np.array(g["proposal"]), g["k"])
    np.testing.assert_allclose(law, g["output_marginal"], atol=1e-12)


@pytest.mark.parametrize("k", [1, 3, 4])
def test_page_example_more_children(k):
    g = gold("specinfer_children.json")["residual_update"]
    law = iid_children_first_law(np.array(g["target"]), np.array(g["proposal"]), k)
    np.testing.assert_allclose(law, g["output_marginal"], atol=1e-12)


def test_naive_retest_fails_the_page_example(tmp_path):
    g = gold("specinfer_children.json")["residual_update"]
    naive = O.build_planted(NAIVE_RETEST, str(tmp_path))
    law = iid_children_first_law(np.array(g["target"]), np.array(g["proposal"]), g["k"], lib=naive)
    assert not g["naive_retest_matches"]
    assert np.max(np.abs(law - np.array(g["output_marginal"]))) > 0.01
    # by hand: token 1 comes out with 0.4 * (0.75 + 0.25 * 0.4 * 0.75) = 0.33 under the re-test
    assert abs(law[1] - 0.33) < 1e-12


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_repeated_copies_keep_target_mass(k, tmp_path):
    g = gold("specinfer_children.json")["repeated_copies"]
    p, q, x = np.array(g["target"]), np.array(g["proposal"]), g["token"]
    target = np.tile(logp(p), (k + 1, 1))
    draft = logp(q)[None, :]
    law = first_token_law(branch_law(target, draft, [-1] * k, [x] * k, [0] * k), 2)
    assert abs(law[x] - g["exact_prob_token"]) < 1e-12
    naive = O.build_planted(NAIVE_RETEST, str(tmp_path))
    law_n = first_token_law(branch_law(target, draft, [-1] * k, [x] * k, [0] * k, lib=naive), 2)
    assert abs(law_n[x] - (1.0 - 2.0 ** -k)) < 1e-12


# ------------------------------------------------------------------------------ a tiny "model"

class TinyModel:
    """Next-token rows of a target and a draft model that depend only on the token path."""

    def __init__(self, V, seed, scale_p=1.5, scale_q=1.0):
        self.V, self.seed, self.sp, self.sq = V, seed, scale_p, scale_q

    def _row(self, path, salt, scale):
        rng = np.random.default_rng([self.seed, salt, len(path), *path])
        return rng.normal(0.0, scale, self.V)

    def p_logits(self, path):
        return self._row(path, 1, self.sp)

    def q_logits(self, path):
        # correlated with the target so that acceptance is common but not certain
        return 0.7 * self.p_logits(path) + self._row(path, 2, self.sq)

    @staticmethod
    def probs(z, T=1.0):
        e = np.exp((z - z.max()) / T)
        return e / e.sum()


def tree_paths(parents, tokens):
    paths = []
    for i, pr in enumerate(parents):
        paths.append((paths[pr] if pr >= 0 else ()) + (int(tokens[i]),))
    return paths


def tree_rows(model, parents, tokens):
    """target [N+1, V] by the predictor-row convention; draft rows likewise, qrow[i] = parent+1."""
    paths = tree_paths(parents, tokens)
    rows_at = [()] + paths  # row 0: frontier, row i+1: node i
    target = np.stack([model.p_logits(pa) for pa in rows_at])
    draft = np.stack([model.q_logits(pa) for pa in rows_at])
    qrow = [pr + 1 for pr in parents]
    return target, draft, qrow, paths


def depth_of(parents):
    d = []
    for pr in parents:
        d.append(1 if pr < 0 else d[pr] + 1)
    return max(d) if d else 0


def extended_law(model, parents, T=1.0):
    """Law of the emitted sequence, continued by target draws to depth+1 tokens, over all token
    assignments drawn from the draft model (children of one node i.i.d. given its path)."""
    V, N = model.V, len(parents)
    D = depth_of(parents) + 1
    law = {}
    for toks in itertools.product(range(V), repeat=N):
        target, draft, qrow, paths = tree_rows(model, parents, toks)
        w = 1.0
        for i, pr in enumerate(parents):
            w *= model.probs(draft[pr + 1], T)[toks[i]]
        bl = branch_law(target, draft, list(parents), list(toks), qrow, T)
        for seq, pw in bl.items():
            stack = [(seq, w * pw)]
            while stack:
                s, ws = stack.pop()
                if len(s) == D:
                    law[s] = law.get(s, 0.0) + ws
                    continue
                nxt = model.probs(model.p_logits(s), T)
                stack.extend((s + (y,), ws * nxt[y]) for y in range(V) if nxt[y] > 0)
    return law, D


def target_law(model, D, T=1.0):
    law = {}
    for s in itertools.product(range(model.V), repeat=D):
        w = 1.0
        for j in range(D):
            w *= model.probs(model.p_logits(s[:j]), T)[s[j]]
        law[s] = w
    return law


TREES = {
    "two_children": [-1, -1],
    "chain3": [-1, 0, 1],
    "fan_then_one": [-1, -1, 0],
    "mixed": [-1, -1, 0, 1],
    "three_then_two": [-1, -1, -1, 0, 0],
}


@pytest.mark.parametrize("name", list(TREES))
@pytest.mark.parametrize("T", [1.0, 0.6])
def test_tree_emits_target_sequence_law(name, T):
    parents = TREES[name]
    V = 3 if len(parents) <= 4 else 2
    model = TinyModel(V, seed=sum(map(ord, name)))
    got, D = extended_law(model, parents, T)
    want = target_law(model, D, T)
    assert abs(sum(got.values()) - 1.0) < 1e-12
    for s, w in want.items():
        assert abs(got.get(s, 0.0) - w) < 1e-12, (s, got.get(s, 0.0), w)


def test_wrong_predictor_row_breaks_sequence_law(tmp_path):
    """Reading node s's own row instead of the current node's row (an off-by-one of the predictor
    row convention, M7.7 0x07E) is caught by the same law."""
    planted = O.build_planted(
        [("size_t off = ((size_t)b * (size_t)(N + 1) + (size_t)(cur + 1)) * (size_t)V;",
          "size_t off = ((size_t)b * (size_t)(N + 1) + (size_t)(cur + 2 <= N ? cur + 2 : cur + 1)) * (size_t)V;")],
        str(tmp_path))
    parents = [-1, -1, 0, 1]
    model = TinyModel(3, seed=7)
    target, draft, qrow, _ = tree_rows(model, parents, [0, 1, 2, 0])
    law_ok = branch_law(target, draft, parents, [0, 1, 2, 0], qrow)
    law_bad = branch_law(target, draft, parents, [0, 1, 2, 0], qrow, lib=planted)
    keys = set(law_ok) | set(law_bad)
    assert max(abs(law_ok.get(s, 0) - law_bad.get(s, 0)) for s in keys) > 1e-3


# ------------------------------------------------------------------------------ special cases

def test_chain_is_plain_speculative_sampling():
    rng = np.random.default_rng(11)
    B, gamma, V = 400, 4, 12
    t = rng.normal(0, 2, (B, gamma + 1, V))
    d = t[:, :gamma] + rng.normal(0, 1, (B, gamma, V))
    toks = np.empty((B, gamma), np.int32)
    for b in range(B):
        for i in range(gamma):
            q = np.exp(d[b, i] - d[b, i].max())
            toks[b, i] = rng.choice(V, p=q / q.sum())
    u_tree = rng.random((B, gamma + 1)).astype(np.float32)
    u_chain = np.concatenate([u_tree, u_tree[:, -1:]], axis=1)
    parents = np.tile(np.arange(-1, gamma - 1, dtype=np.int32), (B, 1))
    qrow = np.tile(np.arange(gamma, dtype=np.int32), (B, 1))
    tr = O.tree_verify_sample(t, d, parents, toks, qrow, u_tree, 0.9)
    ch = O.spec_verify(t, d, toks, u_chain, 0.9)
    np.testing.assert_array_equal(tr["row_status"], ch["row_status"])
    np.testing.assert_array_equal(tr["accepted_len"], ch["accepted_len"])
    np.testing.assert_array_equal(tr["out_tokens"], ch["out_tokens"])
    for b in range(B):
        A = ch["accepted_len"][b]
        tested = min(A + 1, gamma)
        np.testing.assert_allclose(tr["accept"][b, :tested], ch["accept"][b, :tested], rtol=1e-15)
        assert np.all(np.isnan(tr["accept"][b, tested:]))
    assert 0 < np.mean(ch["accepted_len"]) < gamma  # both branches were exercised


def test_empty_tree_is_one_draw_from_the_frontier():
    rng = np.random.default_rng(5)
    V = 9
    for _ in range(50):
        z = rng.normal(0, 2, V)
        u = np.float32(rng.random())
        r = O.tree_verify_sample(z[None, None], np.zeros((1, 0, V)), np.zeros((1, 0)),
                                 np.zeros((1, 0)), np.zeros((1, 0)), [[u]], 1.3)
        st, p, _, _ = O.row_probs(z, 1.3)
        y, lo, hi = O.inverse_cdf(p, float(u))
        assert r["accepted_len"][0] == 0 and r["out_tokens"][0, 0] == y
        assert r["draw_lo"][0] == lo and r["draw_hi"][0] == hi


def test_monte_carlo_uses_independent_uniform_slots():
    """Random uniforms (not forced branches): the extended two-token law passes a chi-square test.
    A walk that reused one uniform for two decisions would bias it."""
    scipy_stats = pytest.importorskip("scipy.stats")
    parents = [-1, -1, 0, 0]
    V, B = 3, 40000
    model = TinyModel(V, seed=3)
    rng = np.random.default_rng(2024)
    # draw the tree tokens from the draft model, level by level
    T = 1.0
    tgt = np.empty((B, len(parents) + 1, V))
    dr = np.empty_like(tgt)
    toks = np.empty((B, len(parents)), np.int32)
    cache = {}
    for b in range(B):
        tk = []
        for i, pr in enumerate(parents):
            path = tree_paths(parents[:i], tk)[pr] if pr >= 0 else ()
            q = model.probs(model.q_logits(path), T)
            tk.append(int(rng.choice(V, p=q)))
        key = tuple(tk)
        if key not in cache:
            cache[key] = tree_rows(model, parents, tk)
        tgt[b], dr[b], qrow, _ = cache[key]
        toks[b] = tk
    qrows = np.tile(np.array(qrow, np.int32), (B, 1))
    u = rng.random((B, len(parents) + 1)).astype(np.float32)
    r = O.tree_verify_sample(tgt, dr, np.tile(parents, (B, 1)), toks, qrows, u, T)
    assert np.all(r["row_status"] == 0)
    D = 3
    counts = {}
    for b in range(B):
        L = r["accepted_len"][b]
        s = tuple(int(x) for x in r["out_tokens"][b, : L + 1])
        while len(s) < D:
            s = s + (int(rng.choice(V, p=model.probs(model.p_logits(s), T))),)
        counts[s] = counts.get(s, 0) + 1
    want = target_law(model, D, T)
    keys = sorted(want)
    obs = np.array([counts.get(k, 0) for k in keys], float)
    exp = np.array([want[k] for k in keys]) * B
    chi2 = float(np.sum((obs - exp) ** 2 / exp))
    assert scipy_stats.chi2.sf(chi2, len(keys) - 1) > 1e-4, chi2


# ------------------------------------------------------------------------------ statuses

def _one(parents, tokens, qrow, u, target=None, draft=None, V=5, max_out=None):
    N = len(parents)
    if target is None:
        target = np.zeros((N + 1, V))
    if draft is None:
        draft = np.zeros((max(N, 1), V))
    return O.tree_verify_sample(target[None], draft[None], [parents], [tokens], [qrow], [u], 1.0,
                                max_out=max_out)


def test_statuses():
    ok = _one([-1, 0], [1, 2], [0, 1], [0.1, 0.1, 0.5])
    assert ok["row_status"][0] == O.ROW_OK and ok["accepted_len"][0] == 2  # uniform rows: a = 1
    assert _one([-1, 1], [1, 2], [0, 1], [0.1] * 3)["row_status"][0] == O.ROW_BAD_PARENT
    assert _one([-1, 0], [1, 2], [0, 2], [0.1] * 3)["row_status"][0] == O.ROW_BAD_QROW
    assert _one([-1, 0], [1, 5], [0, 1], [0.1] * 3)["row_status"][0] == O.ROW_BAD_TOKEN
    assert _one([-1, 0], [1, 2], [0, 1], [0.1, 1.0, 0.1])["row_status"][0] == O.ROW_BAD_UNIFORM
    # the uniform of a node the walk never tests is still validated (it is part of the input)
    assert _one([-1, -1], [1, 2], [0, 0], [0.1, -0.5, 0.1])["row_status"][0] == O.ROW_BAD_UNIFORM
    # q(x) = 0 for a tested node
    d = np.zeros((2, 5))
    d[0, 1] = -np.inf
    assert _one([-1, 0], [1, 2], [0, 1], [0.1] * 3, draft=d)["row_status"][0] == O.ROW_BAD_TOKEN
    # non-finite in a visited row; the same in a row the walk never reaches is not seen
    t = np.zeros((3, 5))
    t[1, 3] = np.nan
    assert _one([-1, 0], [1, 2], [0, 1], [0.1] * 3, target=t)["row_status"][0] == O.ROW_NONFINITE
    t = np.zeros((3, 5))
    t[2, 3] = np.nan
    r = _one([-1, 0], [1, 2], [0, 1], [0.1, 0.99, 0.5], target=t,
             draft=np.array([[0, 5.0, 0, 0, 0], [0, 0, 5.0, 0, 0]]))
    assert r["row_status"][0] == O.ROW_OK and r["accepted_len"][0] == 1
    # overflow: a path of 2 plus the final token does not fit in 2 outputs
    assert _one([-1, 0], [1, 2], [0, 1], [0.1] * 3, max_out=2)["row_status"][0] == O.ROW_OVERFLOW
    assert _one([-1, 0], [1, 2], [0, 1], [0.1] * 3, max_out=3)["row_status"][0] == O.ROW_OK
