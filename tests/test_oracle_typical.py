"""The oracle's typical-acceptance tree verify against what the pages and the mathematics fix.

Module 16, "Verify the Tree": Medusa's sampling mode replaces the greedy check by typical
acceptance, which accepts a candidate token when the target's probability clears
min(eps, delta * exp(-H)), H the entropy of the target's distribution at that position.  Pins:
  - the entropy and the log-probabilities against scipy (a library routine);
  - the threshold rule on hand-computed rows (uniform, peaked);
  - with eps = 0 every candidate is typical: the walk picks the deepest node, lowest index first;
  - with a threshold of exactly 1/2 on rows whose largest probability exceeds 1/2, typical
    acceptance is the greedy check, so the accepted path equals the greedy tree oracle's (itself
    pinned to the lesson's worked example);
  - the token after the path follows p of the accepted node's row, exactly, by enumeration;
  - the statuses, and a planted mistake (max in place of min) that the threshold pin catches.
"""
import ctypes

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S


def run(lg, par, tok, u, T=1.0, eps=0.09, delta=0.3, max_out=None):
    return O.tree_verify_typical(np.asarray(lg, np.float64), par, tok, u, T, eps, delta, max_out)


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
def test_entropy_and_logp_match_scipy(T):
    rng = np.random.default_rng(1)
    B, N, V = 3, 6, 57
    lg = (rng.standard_normal((B, N + 1, V)) * 2.5).astype(np.float32)
    par = np.array([[-1, -1, 0, 0, 2, 4]] * B, np.int32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    o = O.tree_verify_typical(lg, par, tok, rng.random(B).astype(np.float32), T, 0.09, 0.3)
    p = scipy.special.softmax(lg.astype(np.float64) / T, axis=-1)
    np.testing.assert_allclose(o["entropy"], scipy.stats.entropy(p, axis=-1), rtol=0, atol=1e-12)
    lsm = scipy.special.log_softmax(lg.astype(np.float64) / T, axis=-1)
    rows = np.where(par < 0, 0, par + 1)
    want = np.stack([lsm[b, rows[b], tok[b]] for b in range(B)])
    np.testing.assert_allclose(o["logp"], want, rtol=0, atol=1e-12)


def test_threshold_rule_by_hand():
    """Uniform row over 4 tokens: H = ln 4, p = 1/4, threshold min(eps, delta / 4)."""
    V = 4
    uni = np.zeros((1, 2, V))
    par, tok, u = [[-1]], [[2]], [0.5]
    # eps 0.09, delta 0.3: threshold 0.075 < 0.25: accepted
    o = run(uni, par, tok, u, eps=0.09, delta=0.3)
    assert o["accepted_len"][0] == 1 and o["entropy"][0, 0] == pytest.approx(np.log(4), abs=1e-15)
    # eps 0.3, delta 2: threshold min(0.3, 0.5) = 0.3 > 0.25: rejected
    o = run(uni, par, tok, u, eps=0.3, delta=2.0)
    assert o["accepted_len"][0] == 0
    # eps 0.3, delta 0.9: threshold min(0.3, 0.225) = 0.225 < 0.25: accepted
    o = run(uni, par, tok, u, eps=0.3, delta=0.9)
    assert o["accepted_len"][0] == 1
    # a peaked row [10, 0, 0, 0]: p(1) = 1 / (e^10 + 3) is far below min(eps, delta e^-H)
    pk = np.array([[[10.0, 0, 0, 0], [0, 0, 0, 0]]])
    assert run(pk, par, [[1]], u)["accepted_len"][0] == 0
    assert run(pk, par, [[0]], u)["accepted_len"][0] == 1
    # strict inequality: p exactly at the threshold is not typical (uniform over 4, eps = 0.25)
    assert run(uni, par, tok, u, eps=0.25, delta=10.0)["accepted_len"][0] == 0


def test_planted_max_for_min_fails_the_threshold_pin(tmp_path):
    lib = O.build_planted([("const double thr = fmin(eps, delta * exp(-H[row]));",
                            "const double thr = fmax(eps, delta * exp(-H[row]));")], str(tmp_path))
    lib.oracle_tree_verify_typical.argtypes = [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int] * 3 + [ctypes.c_double] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 7
    lg = np.zeros((1, 2, 4))
    par, tok, u = np.array([[-1]], np.int32), np.array([[2]], np.int32), np.array([0.5], np.float32)
    acc = np.empty(1, np.int32)
    out = np.empty((1, 2), np.int32)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    # uniform row over 4 tokens, eps 0.3, delta 0.9: min gives 0.225 < 1/4 (typical), max 0.3
    lib.oracle_tree_verify_typical(P(lg), O.F64, P(par), P(tok), P(u), 1, 1, 4, 1.0, 0.3, 0.9, 2,
                                   P(acc), P(out), None, None, None, None, None)
    assert run(lg, par, tok, u, eps=0.3, delta=0.9)["accepted_len"][0] == 1
    assert acc[0] == 0


def depth_first_deepest(par):
    """The deepest node of a tree (lowest index on ties), from the parents alone."""
    d, best, bd = [], -1, 0
    for i, p in enumerate(par):
        d.append(1 if p < 0 else d[p] + 1)
        if d[i] > bd:
            bd, best = d[i], i
    return best, bd


@pytest.mark.parametrize("seed", range(3))
def test_eps_zero_accepts_every_candidate(seed):
    tb = S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c5"], B=4, V=300, seed=800 + seed))
    u = np.full(4, 0.5, np.float32)
    o = O.tree_verify_typical(tb.logits, tb.parents, tb.tokens, u, 1.0, 0.0, 0.3)
    for b in range(4):
        best, bd = depth_first_deepest(tb.parents[b].tolist())
        assert o["accepted_len"][b] == bd
        assert o["out_nodes"][b, bd - 1] == best


@pytest.mark.parametrize("seed", range(4))
def test_threshold_one_half_is_the_greedy_check(seed):
    """Rows with a probability mass above 1/2 on their argmax; eps = 1/2 and delta = V make the
    threshold exactly 1/2, which only the argmax clears: the accepted path is greedy's."""
    rng = np.random.default_rng(900 + seed)
    tb = S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c5"], B=6, V=200, seed=900 + seed))
    lg = S.stored_to_f64(tb.logits)
    top = lg.argmax(-1)
    np.put_along_axis(lg, top[..., None], lg.max(-1, keepdims=True) + 40.0, axis=-1)
    # node tokens: the predictor row's argmax with probability 0.7, else another token
    rows = np.where(tb.parents < 0, 0, tb.parents + 1)
    am = np.take_along_axis(top, rows, 1)
    tok = np.where(rng.random(am.shape) < 0.7, am, (am + 1 + rng.integers(0, 150, am.shape)) % 200)
    tok = tok.astype(np.int32)
    u = rng.random(6).astype(np.float32)
    ty = O.tree_verify_typical(lg, tb.parents, tok, u, 1.0, 0.5, 200.0)
    gr = O.tree_verify_greedy(lg, tb.parents, tok)
    assert np.array_equal(ty["accepted_len"], gr["accepted_len"])
    for b in range(6):
        A = gr["accepted_len"][b]
        assert np.array_equal(ty["out_tokens"][b, :A], gr["out_tokens"][b, :A])
        assert np.array_equal(ty["out_nodes"][b, :A], gr["out_nodes"][b, :A])
    assert (gr["accepted_len"] > 0).any()


def test_final_token_law_by_enumeration():
    """The token after the accepted path follows p of the accepted node's own row, exactly: p is
    dyadic and a midpoint grid of the uniform integrates the draw without error."""
    pr = [np.array([0.5, 0.25, 0.125, 0.125]), np.array([0.125, 0.125, 0.25, 0.5]),
          np.array([0.25, 0.25, 0.25, 0.25])]
    lg = np.log(np.stack(pr))[None]
    M = 1024
    u = ((np.arange(M) + 0.5) / M).astype(np.float32)
    for tok, row in (([[0, 3]], 2), ([[0, 1]], 1), ([[2, 3]], 0)):
        # eps 0.3 delta 1: row 0 threshold 0.3 -> token 0 (0.5) typical, 2 (0.125) not; row 1
        # (node 0's row) threshold 0.3 -> token 3 (0.5) typical, 1 not
        o = run(np.repeat(lg, M, 0), [[-1, 0]] * M, tok * M, u, eps=0.3, delta=1.0)
        assert np.all(o["row_status"] == 0)
        last = o["out_tokens"][np.arange(M), o["accepted_len"]]
        law = np.bincount(last, minlength=4) / M
        np.testing.assert_allclose(law, pr[row], atol=0)


def test_statuses():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((6, 4, 10))
    par = np.array([[-1, 0, 1]] * 6, np.int32)
    tok = np.array([[1, 2, 3]] * 6, np.int32)
    u = np.full(6, 0.5, np.float32)
    lg[0, 2, 4] = np.nan                  # a non-finite row
    par[1, 2] = 2                         # a parent that does not precede its node
    tok[2, 1] = 10                        # a token outside [0, V)
    u[3] = 1.0                            # a uniform outside [0, 1)
    lg[5, 1:] = -np.inf                   # rows with no finite entry
    o = run(lg, par, tok, u, eps=0.0)
    assert o["row_status"].tolist() == [O.ROW_NONFINITE, O.ROW_BAD_PARENT, O.ROW_BAD_TOKEN,
                                        O.ROW_BAD_UNIFORM, O.ROW_OK, O.ROW_NONFINITE]
    assert np.all(o["accepted_len"][[0, 1, 2, 3, 5]] == -1)
    assert o["accepted_len"][4] == 3
    # the path and the final token must fit in max_out
    o2 = run(lg[4:5], par[4:5], tok[4:5], u[4:5], eps=0.0, max_out=3)
    assert o2["row_status"][0] == O.ROW_OVERFLOW
    o3 = run(lg[4:5], par[4:5], tok[4:5], u[4:5], eps=0.0, max_out=4)
    assert o3["row_status"][0] == O.ROW_OK
