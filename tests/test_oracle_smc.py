"""Pins of the SMC-SD verify round in the oracle (Module 16 lesson, "SMC Speculative Decoding:
Resample, Don't Reject").

What fixes the answer, from outside the oracle:
  - the page's printed effective sample sizes and its printed Algorithm-1 round (block ratios, ESS,
    resampling, reset weights), kept in tests/golden/smc_round.json;
  - its two exact anchors: q = p gives block ratio 1, ESS = N and no resampling; K = 0 leaves the
    weights alone and draws the extension from the first target row;
  - the block ratio is the product of per-position likelihood ratios (brute force on small rows);
  - resampling is faithful: a particle's ancestor falls on particle i with probability w_i / sum w,
    checked exactly by sweeping the ancestor uniform over the CDF boundaries.
"""
import json
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold():
    with open(os.path.join(GOLD, "smc_round.json")) as f:
        return json.load(f)


def logp(x):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(x, np.float64))


def page_round(u=0.5):
    g = gold()["round"]
    N, K = g["particles"], g["K"]
    t = np.tile(logp(g["target"]), (N, K + 1, 1))
    d = np.tile(logp(g["draft"]), (N, K, 1))
    uu = np.full((N, 2), u, np.float32)
    return g, O.smc_verify(t, d, g["draft_blocks"], np.log(g["weights_in"]), uu, 1, 1.0, g["eta"])


def test_ess_examples():
    ex = gold()["ess_examples"]
    assert O.ess(ex[0]["weights"]) == ex[0]["ess"]
    assert round(O.ess(ex[1]["weights"]), 3) == ex[1]["ess_3dp"]
    assert abs(O.ess(ex[1]["weights"]) - 13.0 ** 2 / 103.0) < 1e-12  # (sum w)^2 / sum w^2


def test_page_round():
    g, o = page_round()
    ratios = np.exp(o["log_ratio"])
    np.testing.assert_array_equal(np.round(ratios, 2), g["block_ratios_2dp"])
    p, q = np.array(g["target"]), np.array(g["draft"])
    exact = [np.prod([p[x] / q[x] for x in blk]) for blk in g["draft_blocks"]]
    np.testing.assert_allclose(ratios, exact, rtol=1e-12)
    assert round(float(o["ess"][0]), 2) == g["ess_2dp"]
    assert bool(o["resampled"][0]) == g["resampled"]
    np.testing.assert_allclose(np.exp(o["logw_out"]), g["weights_after"], rtol=1e-12)
    assert np.all(o["row_status"] == O.ROW_OK)
    # every particle grows by K drafts plus one extension token, nothing rolled back
    assert np.all(o["out_tokens"] >= 0) and o["out_tokens"].shape[1] == g["lengths_added"]
    np.testing.assert_array_equal(o["out_tokens"][:, :2], g["draft_blocks"])


def test_anchor_perfect_draft():
    rng = np.random.default_rng(4)
    N, K, V = 8, 3, 11
    t = rng.normal(0, 2, (N, K + 1, V))
    d = t[:, :K].copy()
    tok = rng.integers(0, V, (N, K))
    u = rng.random((N, 2)).astype(np.float32)
    o = O.smc_verify(t, d, tok, np.zeros(N), u, 1, 0.9, N / 2)
    assert np.all(o["log_ratio"] == 0.0)
    assert abs(o["ess"][0] - N) < 1e-12 and o["resampled"][0] == 0
    np.testing.assert_array_equal(o["ancestors"], np.arange(N))
    np.testing.assert_array_equal(o["logw_out"], np.zeros(N))


def test_anchor_no_draft():
    rng = np.random.default_rng(6)
    N, V = 8, 13
    t = rng.normal(0, 2, (N, 1, V))
    lw = rng.normal(0, 0.3, N)
    u = rng.random((N, 2)).astype(np.float32)
    o = O.smc_verify(t, np.zeros((N, 0, V)), np.zeros((N, 0)), lw, u, 1, 1.0, 1.0)
    assert np.all(o["log_ratio"] == 0.0)
    np.testing.assert_array_equal(o["logw_out"], lw)  # ESS >= 1 = eta: no resampling
    for n in range(N):
        _, p, _, _ = O.row_probs(t[n, 0], 1.0)
        y, _, _ = O.inverse_cdf(p, float(u[n, 0]))
        assert o["out_tokens"][n, 0] == y


def test_block_ratio_is_product_of_position_ratios():
    rng = np.random.default_rng(8)
    N, K, V, T = 6, 4, 9, 0.7
    t = rng.normal(0, 2, (N, K + 1, V))
    d = rng.normal(0, 2, (N, K, V))
    tok = rng.integers(0, V, (N, K))
    o = O.smc_verify(t, d, tok, np.zeros(N), np.full((N, 2), 0.3, np.float32), 2, T, 0.0)
    for n in range(N):
        want = 0.0
        for j in range(K):
            _, p, _, _ = O.row_probs(t[n, j], T)
            _, q, _, _ = O.row_probs(d[n, j], T)
            want += np.log(p[tok[n, j]] / q[tok[n, j]])
        assert abs(o["log_ratio"][n] - want) < 1e-12


def test_resampling_is_faithful():
    """Sweeping one particle's ancestor uniform over the CDF boundaries: the ancestor is particle i
    on an interval of length w_i / sum w."""
    g = gold()["round"]
    N, K = g["particles"], g["K"]
    t = np.tile(logp(g["target"]), (N, K + 1, 1))
    d = np.tile(logp(g["draft"]), (N, K, 1))
    ratios = None
    mass = np.zeros(N)
    edges = np.linspace(0, 1, 200001, dtype=np.float64)[:-1]
    # the ancestor of particle 0 as a function of its uniform, at fine resolution
    u = np.full((N, 2), 0.5, np.float32)
    prev, start = None, 0.0
    for x in np.unique(np.float32(edges)):
        u[0, 1] = x
        o = O.smc_verify(t, d, g["draft_blocks"], np.zeros(N), u, 1, 1.0, g["eta"])
        a = o["ancestors"][0]
        if ratios is None:
            ratios = np.exp(o["log_ratio"])
        if prev is not None and a != prev:
            mass[prev] += x - start
            start = x
        prev = a
    mass[prev] += 1.0 - start
    np.testing.assert_allclose(mass, ratios / ratios.sum(), atol=2e-5)


def test_failed_particle_fails_its_group_only():
    rng = np.random.default_rng(10)
    G, N, K, V = 3, 4, 2, 7
    B = G * N
    t = rng.normal(0, 1, (B, K + 1, V))
    d = rng.normal(0, 1, (B, K, V))
    tok = rng.integers(0, V, (B, K))
    u = rng.random((B, 2)).astype(np.float32)
    t[5, 1, 2] = np.nan      # group 1
    u[9, 1] = 1.0            # group 2: a bad ancestor uniform
    o = O.smc_verify(t, d, tok, np.zeros(B), u, G, 1.0, N / 2)
    assert o["row_status"][5] == O.ROW_NONFINITE and o["row_status"][9] == O.ROW_BAD_UNIFORM
    for g in (1, 2):
        assert np.isnan(o["ess"][g]) and o["resampled"][g] == -1
        assert np.all(o["ancestors"][g * N:(g + 1) * N] == -1)
        assert np.all(np.isnan(o["logw_out"][g * N:(g + 1) * N]))
    assert np.isfinite(o["ess"][0]) and o["resampled"][0] in (0, 1)
    assert np.all(o["out_tokens"][5] == -1) and np.all(o["out_tokens"][4] >= 0)


def test_q_zero_is_a_bad_token():
    V = 5
    t = np.zeros((1, 2, V))
    d = np.zeros((1, 1, V))
    d[0, 0, 3] = -np.inf
    o = O.smc_verify(t, d, [[3]], np.zeros(1), np.full((1, 2), 0.5, np.float32), 1, 1.0, 0.5)
    assert o["row_status"][0] == O.ROW_BAD_TOKEN


def test_status_precedence_matches_the_plain_round():
    """A non-finite row anywhere outranks a bad token, which outranks a bad uniform (as in the
    plain round's statuses)."""
    V = 6
    t = np.zeros((3, 3, V))
    d = np.zeros((3, 2, V))
    tok = np.array([[9, 1], [9, 1], [1, 1]])   # position 0 out of range in requests 0 and 1
    t[0, 2, 4] = np.nan                          # request 0: also a NaN in the extension row
    u = np.full((3, 2), 0.5, np.float32)
    u[1, 1] = 1.5                                # request 1: also a bad uniform
    u[2, 0] = -0.1                               # request 2: a bad uniform alone
    o = O.smc_verify(t, d, tok, np.zeros(3), u, 3, 1.0, 0.5)
    assert list(o["row_status"]) == [O.ROW_NONFINITE, O.ROW_BAD_TOKEN, O.ROW_BAD_UNIFORM]
