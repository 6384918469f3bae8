"""The emitted law of the oracle against the target law.

Exactness is the theorem of the pages (M7.1 sections 0x03C and 0x03F, the Module 16 proof): the
first emitted token follows p_1, and the token emitted at position i, given that position i is
reached, follows p_i.  These tests check the oracle against that law by exhaustive enumeration on
tiny vocabularies (with probabilities chosen so that every decision boundary is a dyadic rational
and a midpoint grid integrates the uniform draws exactly), against the direct target chain over a
three-token horizon (M7.1 section 0x04H), and by chi-square on the tiny fp32 configuration.
"""
import itertools

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S


def logs(rows):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(rows, dtype=np.float64))


def grid(M):
    return (np.arange(M) + 0.5) / M


def enumerate_round(p_rows, q_rows, M):
    """Run the oracle over every draft path (weighted by q) and every grid point of every uniform
    slot; returns (outputs, weights, token paths)."""
    p_rows = np.asarray(p_rows, float)
    q_rows = np.asarray(q_rows, float)
    gamma, V = q_rows.shape
    paths = list(itertools.product(range(V), repeat=gamma))
    pw = [np.prod([q_rows[i, x[i]] for i in range(gamma)]) for x in paths]
    keep = [i for i, w in enumerate(pw) if w > 0]
    paths = [paths[i] for i in keep]
    pw = np.array([pw[i] for i in keep])
    G = np.stack(np.meshgrid(*([grid(M)] * (gamma + 2)), indexing="ij"), -1).reshape(-1, gamma + 2)
    toks = np.repeat(np.array(paths, np.int32).reshape(len(paths), gamma), len(G), 0)
    u = np.tile(G, (len(paths), 1)).astype(np.float32)
    w = np.repeat(pw, len(G)) / len(G)
    n = len(toks)
    t = np.broadcast_to(logs(p_rows), (n, gamma + 1, V)).copy()
    d = np.broadcast_to(logs(q_rows), (n, gamma, V)).copy()
    out = O.spec_verify(t, d, toks, u, 1.0)
    assert np.all(out["row_status"] == 0)
    return out, w, toks


def dyadic_pair(rng, V, denom, q):
    """Random p with entries in (1/denom)Z summing to 1 such that the residual mass Z = TV(p, q)
    is 0 or a power of two over denom (so residual CDF boundaries stay in (1/denom)Z)."""
    while True:
        cuts = np.sort(rng.choice(np.arange(1, denom), V - 1, replace=True))
        p = np.diff(np.concatenate([[0], cuts, [denom]])) / denom
        Zn = int(round(np.maximum(p - q, 0).sum() * denom))
        if Zn == 0 or (Zn & (Zn - 1)) == 0:
            return p


@pytest.mark.parametrize("seed", range(4))
def test_exact_law_gamma1_V4(seed):
    rng = np.random.default_rng(seed)
    q = np.array([0.5, 0.25, 0.125, 0.125])
    p0 = dyadic_pair(rng, 4, 16, q)
    p1 = dyadic_pair(rng, 4, 16, q)
    out, w, toks = enumerate_round([p0, p1], [q], M=16)
    first = np.zeros(4)
    np.add.at(first, out["out_tokens"][:, 0], w)
    np.testing.assert_allclose(first, p0, atol=1e-12)
    reached = out["accepted_len"] >= 1
    assert w[reached].sum() == pytest.approx(np.minimum(p0, q).sum(), abs=1e-12)
    second = np.zeros(4)
    np.add.at(second, out["out_tokens"][reached, 1], w[reached])
    np.testing.assert_allclose(second / w[reached].sum(), p1, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_exact_law_gamma2_V3(seed):
    rng = np.random.default_rng(100 + seed)
    q0 = np.array([0.5, 0.25, 0.25])
    q1 = np.array([0.25, 0.5, 0.25])
    p0 = dyadic_pair(rng, 3, 8, q0)
    p1 = dyadic_pair(rng, 3, 8, q1)
    p2 = dyadic_pair(rng, 3, 8, q0)
    out, w, toks = enumerate_round([p0, p1, p2], [q0, q1], M=8)
    A = out["accepted_len"]
    for pos, p in ((0, p0), (1, p1), (2, p2)):
        reached = A >= pos
        law = np.zeros(3)
        np.add.at(law, out["out_tokens"][reached, pos], w[reached])
        np.testing.assert_allclose(law / w[reached].sum(), p, atol=1e-12)
    # first-rejection distribution: P(A >= 1) = alpha_0, P(A >= 2 | A >= 1) = alpha_1
    assert w[A >= 1].sum() == pytest.approx(np.minimum(p0, q0).sum(), abs=1e-12)
    assert w[A >= 2].sum() / w[A >= 1].sum() == pytest.approx(np.minimum(p1, q1).sum(), abs=1e-12)


def test_target_joint_two_token_vocab_horizon3():
    """Two-token vocabulary, two drafts, horizon three (M7.1 section 0x04H): the speculative round
    completed by ordinary target transitions must reproduce the target chain's joint law over
    all eight sequences.  Rows depend on the drafted prefix, as in a real causal model."""
    rng = np.random.default_rng(11)
    prefixes = [(), (0,), (1,), (0, 0), (0, 1), (1, 0), (1, 1)]
    P, Q = {}, {}
    for s in prefixes:
        p0 = rng.integers(1, 16) / 16
        P[s] = np.array([p0, 1 - p0])
        Q[s] = np.array([0.5, 0.5])  # accept ratios 2p: multiples of 1/8
    M = 16
    G = np.stack(np.meshgrid(grid(M), grid(M), grid(M), indexing="ij"), -1).reshape(-1, 3)
    joint = np.zeros((2, 2, 2))
    for d0 in range(2):
        for d1 in range(2):
            n = len(G)
            t = np.broadcast_to(logs([P[()], P[(d0,)], P[(d0, d1)]]), (n, 3, 2)).copy()
            d = np.broadcast_to(logs([Q[()], Q[(d0,)]]), (n, 2, 2)).copy()
            u = np.stack([G[:, 0], G[:, 1], np.full(n, 0.5), G[:, 2]], 1).astype(np.float32)
            toks = np.tile(np.array([[d0, d1]], np.int32), (n, 1))
            out = O.spec_verify(t, d, toks, u, 1.0)
            wpath = Q[()][d0] * Q[(d0,)][d1] / n
            for i in range(n):
                A = out["accepted_len"][i]
                y = tuple(int(v) for v in out["out_tokens"][i, :A + 1])
                # complete to horizon 3 with ordinary target transitions
                for rest in itertools.product(range(2), repeat=3 - len(y)):
                    seq = y + rest
                    pr = wpath
                    for j in range(len(y), 3):
                        pr *= P[seq[:j]][seq[j]]
                    joint[seq] += pr
    target = np.zeros((2, 2, 2))
    for x in itertools.product(range(2), repeat=3):
        target[x] = P[()][x[0]] * P[x[:1]][x[1]] * P[x[:2]][x[2]]
    np.testing.assert_allclose(joint, target, atol=1e-12)


def test_c1_chi_square_and_acceptance():
    """10,000 seeded trials of the tiny fp32 configuration (fixed logits, fresh draws)."""
    cfg = S.CONFIGS["c1"]
    b = S.trial_batches(cfg, 10000)
    out = O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, cfg.temperature)
    assert np.all(out["row_status"] == 0)
    T = cfg.temperature
    tv = b.target[0].astype(np.float64)
    dv = b.draft[0].astype(np.float64)
    p = scipy.special.softmax(tv / T, axis=-1)
    q = scipy.special.softmax(dv / T, axis=-1)

    def chi2(tokens, probs):
        counts = np.bincount(tokens, minlength=len(probs)).astype(float)
        exp = probs * len(tokens)
        big = exp >= 5
        f_obs = np.concatenate([counts[big], [counts[~big].sum()]])
        f_exp = np.concatenate([exp[big], [exp[~big].sum()]])
        if f_exp[-1] == 0:
            f_obs, f_exp = f_obs[:-1], f_exp[:-1]
        return scipy.stats.chisquare(f_obs, f_exp).pvalue

    assert chi2(out["out_tokens"][:, 0], p[0]) > 1e-4
    reached = out["accepted_len"] >= 1
    assert chi2(out["out_tokens"][reached, 1], p[1]) > 1e-4
    a0 = np.minimum(p[0], q[0]).sum()
    n = len(reached)
    assert abs(reached.mean() - a0) < 4 * np.sqrt(a0 * (1 - a0) / n)


def test_expected_tokens_survival_form_redrawn_logits():
    """Mean emitted count against E[G] = 1 + sum_j prod_{i<=j} alpha_i (M7.1 section 0x05A),
    each request with its own logits."""
    cfg = S.CONFIGS["c1"]
    b = S.trial_batches(cfg, 4000, redraw_logits=True)
    out = O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, cfg.temperature)
    p = scipy.special.softmax(b.target.astype(np.float64) / cfg.temperature, axis=-1)
    q = scipy.special.softmax(b.draft.astype(np.float64) / cfg.temperature, axis=-1)
    alpha = np.minimum(p[:, :cfg.gamma], q).sum(-1)
    eg = 1 + np.cumprod(alpha, axis=1).sum(1)
    G = out["accepted_len"] + 1
    se = G.std() / np.sqrt(len(G))
    assert abs(G.mean() - eg.mean()) < 4 * se
