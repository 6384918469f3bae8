"""The oracle's top-p (nucleus) processor against what the pages and the mathematics fix.

"Exact speculative and assisted decoding for TinyRustLM" lists top-p among the declared processors
that both the target and the draft distribution pass through before the ratio is formed; M7.1
section 0x03D: truncation keeps the round exact when q is the truncated distribution that sampled
the draft.  Pins:
  - top_p >= 1 is the plain round, bit for bit; a top_p below the largest probability keeps only
    the argmax group;
  - when top_p lies strictly between the masses of the k - 1 and the k most probable tokens, the
    kept set is the top-k set, so the round equals the top-k round (pinned by its own tests);
  - by exhaustive enumeration the emitted tokens follow the processed (nucleus) target law;
  - ties at the threshold are kept whole; the boundary is inclusive (a planted strict comparison
    fails); the statuses.
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S


def batch(seed, B=5, gamma=3, V=60):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((B, gamma + 1, V)) * 2).astype(np.float32)
    d = (t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.7).astype(np.float32)
    tok = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = S.uniforms_from(rng, (B, gamma + 2))
    return t, d, tok, u


def test_top_p_one_is_the_plain_round():
    t, d, tok, u = batch(1)
    a = O.spec_verify(t, d, tok, u, 0.9)
    b = O.spec_verify(t, d, tok, u, 0.9, top_p=1.0)
    for k in ("accepted_len", "out_tokens", "row_status", "lse_p", "lse_q", "accept"):
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_tiny_top_p_keeps_the_argmax_group():
    x = np.array([0.5, 2.0, -1.0, 2.0, 1.0], np.float32)
    st, p, lse, thr, mg = O.row_probs_topp(x, 1.0, 1e-9)
    assert st == 0 and thr == 2.0
    np.testing.assert_array_equal(p, [0, 0.5, 0, 0.5, 0])
    assert lse == pytest.approx(2.0 + np.log(2.0), abs=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_nucleus_between_k_and_k_minus_1_is_top_k(seed):
    """Distinct logits: with top_p between the cumulative masses of the k - 1 and k most probable
    tokens (same for every row), the kept set is the top-k set in every row."""
    rng = np.random.default_rng(seed)
    B, g, V, T = 4, 2, 12, 0.8
    # every row a permutation of the same distinct values, so all rows share the sorted masses
    vals = np.linspace(-3, 3, V).astype(np.float32)
    t = np.stack([[rng.permutation(vals) for _ in range(g + 1)] for _ in range(B)])
    d = np.stack([[rng.permutation(vals) for _ in range(g)] for _ in range(B)])
    srt = np.sort(np.exp(vals.astype(np.float64) / T))[::-1]
    cum = np.cumsum(srt / srt.sum())
    u = S.uniforms_from(rng, (B, g + 2))
    for k in range(1, V):
        # draft tokens inside every draft row's top-k set
        keep = d >= np.sort(d, -1)[..., V - k][..., None]
        tok = np.array([[rng.choice(np.flatnonzero(keep[b, i])) for i in range(g)]
                        for b in range(B)], np.int32)
        top_p = 0.5 * (cum[k - 2] + cum[k - 1]) if k > 1 else 0.5 * cum[0]
        a = O.spec_verify(t, d, tok, u, T, top_k=k)
        b = O.spec_verify(t, d, tok, u, T, top_p=top_p)
        for key in ("accepted_len", "out_tokens", "row_status"):
            assert np.array_equal(a[key], b[key]), (k, key)
        np.testing.assert_allclose(b["lse_p"], a["lse_p"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(b["accept"], a["accept"], rtol=0, atol=1e-12)


def test_ties_at_the_threshold_are_kept_and_the_boundary_is_inclusive(tmp_path):
    # p = [0.5, 0.25, 0.25]: top_p = 0.5 is reached exactly by the first group
    x = np.log(np.array([0.5, 0.25, 0.25]))
    st, p, _, thr, mg = O.row_probs_topp(x, 1.0, 0.5)
    np.testing.assert_allclose(p, [1, 0, 0], atol=0)
    assert mg == pytest.approx(0.0, abs=1e-15)
    # top_p = 0.6 needs the tied pair, which comes in whole
    st, p, _, thr, _ = O.row_probs_topp(x, 1.0, 0.6)
    np.testing.assert_allclose(p, [0.5, 0.25, 0.25], rtol=1e-15)
    planted = O.build_planted([("        if (cum >= top_p) {\n            t = g;",
                                "        if (cum > top_p) {\n            t = g;")], str(tmp_path))
    import ctypes
    xx = np.ascontiguousarray(x)
    pp = np.zeros(3)
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    planted.oracle_row_probs_topp(xx.ctypes.data_as(ctypes.c_void_p), O.F64, 0, 3, 1.0, 0.5,
                                  pp.ctypes.data_as(ctypes.c_void_p), ctypes.byref(a),
                                  ctypes.byref(b), ctypes.byref(c))
    assert pp[1] > 0  # the strict comparison keeps the tied pair as well


def test_emitted_law_by_enumeration():
    """gamma = 1, V = 5: full rows whose nuclei are dyadic after renormalisation; enumerate every
    draft token (weighted by the processed q) and a midpoint grid of every uniform."""
    top_p = 0.75
    p_full = [np.array([0.4, 0.2, 0.2, 0.1, 0.1]), np.array([0.1, 0.1, 0.2, 0.4, 0.2])]
    q_full = np.array([0.2, 0.4, 0.1, 0.2, 0.1])
    # nuclei at 0.75: p0 keeps {0, 1, 2} -> [.5 .25 .25 0 0]; p1 keeps {3, 2, 4} -> [0 0 .25 .5 .25];
    # q keeps {1, 0, 3} -> [.25 .5 0 .25 0]
    pG = [np.array([0.5, 0.25, 0.25, 0, 0]), np.array([0, 0, 0.25, 0.5, 0.25])]
    qG = np.array([0.25, 0.5, 0, 0.25, 0])
    lg_t = np.log(np.stack(p_full))
    lg_d = np.log(q_full)[None]
    M = 16
    grid = (np.arange(M) + 0.5) / M
    G = np.stack(np.meshgrid(*([grid] * 3), indexing="ij"), -1).reshape(-1, 3)
    toks = [x for x in range(5) if qG[x] > 0]
    n = len(toks) * len(G)
    tok = np.repeat(np.array(toks, np.int32), len(G))[:, None]
    u = np.tile(G, (len(toks), 1)).astype(np.float32)
    w = np.repeat(qG[toks], len(G)) / len(G)
    out = O.spec_verify(np.broadcast_to(lg_t, (n, 2, 5)).copy(),
                        np.broadcast_to(lg_d, (n, 1, 5)).copy(), tok, u, 1.0, top_p=top_p)
    assert np.all(out["row_status"] == O.ROW_OK)
    first = np.zeros(5)
    np.add.at(first, out["out_tokens"][:, 0], w)
    np.testing.assert_allclose(first, pG[0], atol=1e-12)
    reached = out["accepted_len"] >= 1
    second = np.zeros(5)
    np.add.at(second, out["out_tokens"][reached, 1], w[reached])
    np.testing.assert_allclose(second / w[reached].sum(), pG[1], atol=1e-12)
    assert w[reached].sum() == pytest.approx(np.minimum(pG[0], qG).sum(), abs=1e-12)


def test_statuses():
    t, d, tok, u = batch(3, B=3)
    t[0, 1, 5] = np.nan
    # request 1: a drafted token outside its draft row's nucleus (the least probable token)
    tok[1, 0] = int(np.argmin(d[1, 0]))
    r = O.spec_verify(t, d, tok, u, 1.0, top_p=0.8)
    assert r["row_status"][0] == O.ROW_NONFINITE
    assert r["row_status"][1] == O.ROW_BAD_TOKEN
    assert np.all(r["out_tokens"][:2] == -1)


def test_margin_reports_the_closest_decision():
    x = np.log(np.array([0.5, 0.3, 0.2]))
    _, _, _, _, mg = O.row_probs_topp(x, 1.0, 0.79)
    assert mg == pytest.approx(0.01, abs=1e-12)  # 0.8 reached, 0.01 above top_p
