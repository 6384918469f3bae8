"""Pins of the fp64 oracle against values the pages print and against closed forms.

None of these tests needs a GPU.  Each check compares the oracle with something other than itself:
a printed value (tests/golden, cited there), a textbook identity, or an independent library routine
(scipy / numpy).
"""
import json
import os

import numpy as np
import pytest
import scipy.special

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def logs(rows):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(rows, dtype=np.float64))


def verify_rows(p_rows, q_rows, tokens, uniforms, T=1.0, top_k=0):
    """One request whose processed rows are given as probabilities (logits = log p, T = 1)."""
    t = logs(p_rows)[None]
    d = logs(q_rows)[None]
    return O.spec_verify(t, d, np.asarray(tokens)[None], np.asarray(uniforms, np.float32)[None],
                         T, top_k)


# ------------------------------------------------------------------ printed worked examples

def test_three_symbol_acceptance_and_residual():
    g = gold("three_symbol.json")
    p, q = np.array(g["target"]), np.array(g["draft"])
    # one position per drafted symbol, so a_i is the conditional acceptance of symbol i
    out = verify_rows([p, p, p, p], [q, q, q], [0, 1, 2], [0.0, 0.0, 0.0, 0.5, 0.5])
    np.testing.assert_allclose(out["accept"][0], g["conditional_acceptance"], atol=1e-12)
    np.testing.assert_allclose(q * out["accept"][0], g["accepted_mass"], atol=1e-12)
    assert O.alpha(p, q) == pytest.approx(g["acceptance_rate"], abs=1e-12)
    r, Z = O.residual(p, q)
    assert Z == pytest.approx(g["rejection_probability"], abs=1e-12)
    np.testing.assert_allclose(r, g["correction_distribution"], atol=1e-12)
    np.testing.assert_allclose(np.minimum(p, q) + Z * r, g["output_distribution"], atol=1e-12)


def _grid(M):
    return (np.arange(M) + 0.5) / M


def test_three_symbol_output_law_by_enumeration():
    """First emitted token over all draft proposals and a midpoint grid of the accept draw.

    Every decision boundary here is a multiple of 0.1, so a 1000-point midpoint grid integrates
    the step functions exactly; the law must equal the printed output distribution.
    """
    g = gold("three_symbol.json")
    p, q = np.array(g["target"]), np.array(g["draft"])
    M = 1000
    xs, us, w = [], [], []
    for x in range(3):
        for u in _grid(M):
            xs.append(x)
            us.append([u, 0.5, 0.5])
            w.append(q[x] / M)
    n = len(xs)
    t = np.broadcast_to(logs([p, p]), (n, 2, 3)).copy()
    d = np.broadcast_to(logs([q]), (n, 1, 3)).copy()
    out = O.spec_verify(t, d, np.array(xs)[:, None], np.array(us, np.float32), 1.0)
    law = np.zeros(3)
    np.add.at(law, out["out_tokens"][:, 0], np.array(w))
    np.testing.assert_allclose(law, g["output_distribution"], atol=1e-12)


def test_three_symbol_iid_output_counts():
    g = gold("three_symbol.json")
    p, q = np.array(g["target"]), np.array(g["draft"])
    M = 10  # accept boundaries are multiples of 0.2
    rows_t, rows_d, toks, us, w = [], [], [], [], []
    for x0 in range(3):
        for x1 in range(3):
            for u0 in _grid(M):
                for u1 in _grid(M):
                    toks.append([x0, x1])
                    us.append([u0, u1, 0.5, 0.5])
                    w.append(q[x0] * q[x1] / M**2)
    n = len(toks)
    t = np.broadcast_to(logs([p, p, p]), (n, 3, 3)).copy()
    d = np.broadcast_to(logs([q, q]), (n, 2, 3)).copy()
    out = O.spec_verify(t, d, np.array(toks), np.array(us, np.float32), 1.0)
    counts = out["accepted_len"] + 1
    probs = [np.sum(np.array(w)[counts == c]) for c in g["iid_output_counts"]]
    np.testing.assert_allclose(probs, g["iid_output_count_probabilities"], atol=1e-12)
    assert np.sum(np.array(w) * counts) == pytest.approx(g["iid_expected_output_count"], abs=1e-12)


def test_m71_one_token_example():
    g = gold("m71_one_token.json")
    p, q = np.array(g["target"]), np.array(g["draft"])
    out = verify_rows([p, p], [q], [g["drafted"]], [0.0, 0.5, 0.5])
    assert out["accept"][0, 0] == pytest.approx(g["accept"], abs=1e-12)
    r, Z = O.residual(p, q)
    assert Z == pytest.approx(g["Z"], abs=1e-12)
    np.testing.assert_allclose(r * Z, g["residual_unnormalised"], atol=1e-12)
    np.testing.assert_allclose(np.round(r, 3), g["residual_normalised_3dp"], atol=0)
    assert O.alpha(p, q) == pytest.approx(g["diagonal"], abs=1e-12)


def test_m16_four_token_and_exercises():
    g = gold("m16_examples.json")
    ft = g["four_token"]
    p, q = np.array(ft["target"]), np.array(ft["draft"])
    assert round(O.alpha(p, q), 3) == ft["alpha_3dp"]
    r, _ = O.residual(p, q)
    np.testing.assert_allclose(r, ft["residual"], atol=1e-12)
    e1 = g["exercise1"]
    p = np.array(e1["target"])
    for key, want in (("draft_close", e1["alpha_close_3dp"]), ("draft_far", e1["alpha_far_3dp"])):
        q = np.array(e1[key])
        a = O.alpha(p, q)
        assert round(a, 3) == want
        assert a == pytest.approx(1.0 - 0.5 * np.abs(p - q).sum(), abs=1e-12)  # alpha = 1 - TV
    e3 = g["exercise3"]
    p, q = np.array(e3["target"]), np.array(e3["draft"])
    r, Z = O.residual(p, q)
    a = O.alpha(p, q)
    np.testing.assert_allclose(np.minimum(p, q) + r * (1.0 - a), p, atol=1e-12)
    ud = g["uniform_draft"]
    a = O.alpha(np.array(ud["target"]), np.array(ud["draft"]))
    assert a == pytest.approx(ud["alpha"], abs=1e-12)
    assert round((1 - a ** (ud["gamma"] + 1)) / (1 - a), 1) == ud["tokens_per_pass_approx"]


def test_tokens_per_pass_by_enumeration():
    """Exercise 2's tokens/pass column: with the same (p, q) at every position the mean emitted
    count is 1 + alpha + ... + alpha^gamma.  p=[0.85,0.15], q=[1,0] makes every draft token 0 and
    alpha = 0.85 exactly; a 20-point grid per accept slot integrates u < 0.85 exactly."""
    g = gold("m16_examples.json")["exercise2"]
    p, q = [0.85, 0.15], [1.0, 0.0]
    M = 20
    for gamma, want in zip(g["gamma"][:4], g["tokens_per_pass_2dp"][:4]):
        grids = np.stack(np.meshgrid(*([_grid(M)] * gamma), indexing="ij"), -1).reshape(-1, gamma)
        n = grids.shape[0]
        u = np.concatenate([grids, np.full((n, 2), 0.5)], 1).astype(np.float32)
        t = np.broadcast_to(logs([p] * (gamma + 1)), (n, gamma + 1, 2)).copy()
        d = np.broadcast_to(logs([q] * gamma), (n, gamma, 2)).copy()
        out = O.spec_verify(t, d, np.zeros((n, gamma), np.int32), u, 1.0)
        mean = np.mean(out["accepted_len"] + 1)
        closed = (1 - 0.85 ** (gamma + 1)) / (1 - 0.85)
        assert mean == pytest.approx(closed, abs=1e-12)
        assert round(mean, 2) == want
    # the closed form against the whole printed column (a check of the formula the harness uses)
    for gamma, want in zip(g["gamma"], g["tokens_per_pass_2dp"]):
        assert round((1 - g["alpha"] ** (gamma + 1)) / (1 - g["alpha"]), 2) == want


# ------------------------------------------------------------------ identities on random rows

def test_coupling_identity_random_rows():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(2, 50))
        p = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 2))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 2))
        a = O.alpha(p, q)
        r, Z = O.residual(p, q)
        assert a == pytest.approx(1.0 - 0.5 * np.abs(p - q).sum(), abs=1e-14)
        assert Z == pytest.approx(1.0 - a, abs=1e-14)
        np.testing.assert_allclose(np.minimum(p, q) + Z * r, p, atol=1e-15)
        assert O.alpha(p, p) == pytest.approx(1.0, abs=1e-14)


def test_softmax_backends_agree():
    """Max-shift and online (m, l) block merge agree, and both equal scipy's logsumexp."""
    rng = np.random.default_rng(1)
    for n in (1, 7, 1000, 5000):
        z = rng.normal(0, 5, n)
        if n > 10:
            z[rng.choice(n, 5, replace=False)] = -np.inf
        ref = scipy.special.logsumexp(z)
        assert O.lse_maxshift(z) == pytest.approx(ref, abs=1e-12)
        for block in (1, 3, 64, 4096):
            assert O.lse_online(z, block) == pytest.approx(O.lse_maxshift(z), abs=1e-12)


def _bf16(x):
    from speculative_decoding_verification_spec_gb300.synth import f32_to_bf16_bits
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def _bf16_vals(h):
    from speculative_decoding_verification_spec_gb300.synth import bf16_bits_to_f32
    return bf16_bits_to_f32(h).astype(np.float64)


@pytest.mark.parametrize("T", [0.7, 1.0, 1.3])
def test_row_probs_match_scipy(T):
    rng = np.random.default_rng(2)
    x64 = rng.normal(0, 3, 4000)
    for stored, vals in ((x64, x64), (x64.astype(np.float32), x64.astype(np.float32).astype(float)),
                         (_bf16(x64), _bf16_vals(_bf16(x64)))):
        st, p, lse, thr = O.row_probs(stored, T)
        assert st == O.ROW_OK and thr == -np.inf
        np.testing.assert_allclose(p, scipy.special.softmax(vals / T), atol=1e-15, rtol=1e-12)
        assert lse == pytest.approx(scipy.special.logsumexp(vals / T), abs=1e-12)


def test_row_probs_topk_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(50):
        V = int(rng.integers(2, 300))
        x = np.round(rng.normal(0, 2, V) * 4) / 4  # coarse values: many ties
        k = int(rng.integers(1, V + 1))
        T = float(rng.uniform(0.5, 2))
        st, p, lse, thr = O.row_probs(x, T, k)
        srt = np.sort(x)[::-1]
        want_thr = srt[k - 1] if k < V else -np.inf
        assert thr == want_thr
        keep = x >= want_thr
        assert keep.sum() >= k
        ref = np.where(keep, scipy.special.softmax(np.where(keep, x / T, -np.inf)), 0.0)
        np.testing.assert_allclose(p, ref, atol=1e-15, rtol=1e-12)
        assert lse == pytest.approx(scipy.special.logsumexp(x[keep] / T), abs=1e-12)
        assert O.kth_largest(x, k) == srt[k - 1]


def test_topk_signed_zero_ties():
    x = np.array([0.0, -0.0, 1.0, -1.0, 0.0, -3.0])
    st, p, lse, thr = O.row_probs(x, 1.0, 2)
    assert thr == 0.0
    assert np.count_nonzero(p) == 4  # 1.0 and all three zeros (signed zeros are equal values)


def test_inverse_cdf_cases():
    r = np.array([0.0, 0.5, 0.0, 0.5])
    assert O.inverse_cdf(r, 0.0)[0] == 1
    assert O.inverse_cdf(r, 0.4999)[0] == 1
    assert O.inverse_cdf(r, 0.5)[0] == 3
    assert O.inverse_cdf(r, 1 - 2**-24)[0] == 3
    assert O.inverse_cdf(np.zeros(4), 0.3)[0] == -1
    rng = np.random.default_rng(4)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        r = rng.random(V) * (rng.random(V) < 0.6)
        if r.sum() == 0:
            continue
        u = float(rng.random())
        v = O.inverse_cdf(r, u)[0]
        want = int(np.searchsorted(np.cumsum(r), u * r.sum(), side="right"))
        assert v == min(want, V - 1) or (want >= V and r[v] > 0)
        assert r[v] > 0


# ------------------------------------------------------------------ statuses and special cases

def test_self_draft_accepts_everything():
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(6))
    for _ in range(20):
        toks = rng.integers(0, 6, 3)
        u = rng.random(5).astype(np.float32)
        out = verify_rows([p] * 4, [p] * 3, toks, u)
        assert out["accepted_len"][0] == 3
        np.testing.assert_array_equal(out["out_tokens"][0, :3], toks)
        np.testing.assert_allclose(out["accept"][0], 1.0, atol=1e-12)


def test_status_codes():
    rng = np.random.default_rng(6)
    t = rng.normal(size=(6, 3, 8))
    d = rng.normal(size=(6, 2, 8))
    tok = np.zeros((6, 2), np.int32)
    u = np.full((6, 4), 0.5, np.float32)
    t[0, 1, 3] = np.nan
    d[1, 0, 2] = np.inf
    t[2, 2, :] = -np.inf
    tok[3, 1] = 8
    d[4, 1, 0] = -np.inf      # q(x) = 0 for the token drafted at position 1
    u[5, 3] = 1.0
    out = O.spec_verify(t, d, tok, u, 1.0)
    np.testing.assert_array_equal(out["row_status"], [1, 1, 1, 3, 3, 7])
    np.testing.assert_array_equal(out["accepted_len"], -1)
    np.testing.assert_array_equal(out["out_tokens"], -1)


def test_topk_equals_masked_and_k_equal_V():
    rng = np.random.default_rng(7)
    B, g, V, k = 40, 3, 16, 4
    t = _bf16(np.round(rng.normal(0, 2, (B, g + 1, V)) * 2) / 2)
    d = _bf16(np.round(rng.normal(0, 2, (B, g, V)) * 2) / 2)
    tv, dv = _bf16_vals(t), _bf16_vals(d)
    kt = -np.sort(-tv, axis=-1)[..., k - 1:k]
    kd = -np.sort(-dv, axis=-1)[..., k - 1:k]
    tm = np.where(tv >= kt, tv, -np.inf)
    dm = np.where(dv >= kd, dv, -np.inf)
    tok = np.array([[rng.choice(np.flatnonzero(dv[b, i] >= kd[b, i, 0])) for i in range(g)]
                    for b in range(B)], np.int32)
    u = rng.random((B, g + 2)).astype(np.float32)
    a = O.spec_verify(t, d, tok, u, 0.9, k)
    m = O.spec_verify(tm, dm, tok, u, 0.9, 0)
    for key in ("accepted_len", "out_tokens", "row_status"):
        np.testing.assert_array_equal(a[key], m[key])
    np.testing.assert_allclose(a["accept"], m["accept"], atol=1e-14)
    full = O.spec_verify(t, d, tok, u, 0.9, V)
    none = O.spec_verify(t, d, tok, u, 0.9, 0)
    for key in ("accepted_len", "out_tokens", "row_status", "accept", "lse_p", "lse_q"):
        np.testing.assert_array_equal(full[key], none[key])
    # a drafted token outside the draft's top-k set cannot have been sampled from it
    tok2 = tok.copy()
    tok2[0, 0] = int(np.argmin(dv[0, 0]))
    bad = O.spec_verify(t, d, tok2, u, 0.9, k)
    assert bad["row_status"][0] == O.ROW_BAD_TOKEN
