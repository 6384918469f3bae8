"""The oracle's grammar mask against what the pages fix.

"Exact speculative and assisted decoding for TinyRustLM", "Grammar and deterministic
opportunities": a grammar mask replaces q by q_G(x) = q(x) 1[x in A_G] / sum_v q(v) 1[v in A_G],
and speculation stays exact relative to q_G when baseline and speculative execution mask alike.
So:
  - a masked row is the unmasked row restricted to A_G and renormalised (checked against the
    unmasked oracle row, itself pinned to scipy, and against scipy's logsumexp over A_G);
  - with one valid set for a whole request, the masked round is the plain round on the vocabulary
    compacted to A_G (the plain round is pinned by the worked examples and the exact-law tests);
  - by exhaustive enumeration, the emitted tokens follow the masked target p_G exactly, whatever
    the logits of the removed tokens hold;
  - the edge cases: a drafted token outside A_G, an empty A_G, a full mask.
"""
import ctypes
import itertools

import numpy as np
import pytest
import scipy.special

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S


def words(valid):
    return S.pack_valid_sets(np.asarray(valid, dtype=bool))


# ------------------------------------------------------------------------------ one row

@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("T", [0.7, 1.0, 1.6])
def test_masked_row_is_restricted_and_renormalised(seed, T):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 300))
    x = (rng.standard_normal(V) * 3).astype(np.float32)
    valid = rng.random(V) < rng.uniform(0.05, 0.95)
    valid[rng.integers(0, V)] = True
    st, p, _, _ = O.row_probs(x, T)
    stg, pg, lseg, _ = O.row_probs(x, T, allowed=words(valid))
    assert st == O.ROW_OK and stg == O.ROW_OK
    want = np.where(valid, p, 0.0)
    want /= want.sum()
    np.testing.assert_allclose(pg, want, rtol=1e-12, atol=1e-15)
    assert np.all(pg[~valid] == 0.0)
    assert lseg == pytest.approx(scipy.special.logsumexp(x[valid].astype(np.float64) / T), abs=1e-12)


def test_masked_row_ignores_removed_nan_and_inf():
    x = np.array([1.0, np.nan, 2.0, np.inf, -1.0], dtype=np.float32)
    valid = np.array([1, 0, 1, 0, 1], bool)
    st, p, _, _ = O.row_probs(x, 1.0, allowed=words(valid))
    assert st == O.ROW_OK
    e = np.exp(np.array([1.0, 2.0, -1.0]))
    np.testing.assert_allclose(p[[0, 2, 4]], e / e.sum(), rtol=1e-14)
    # an allowed NaN or +inf is still non-finite
    st2, _, _, _ = O.row_probs(x, 1.0, allowed=words(np.array([1, 1, 1, 0, 1], bool)))
    assert st2 == O.ROW_NONFINITE
    # an empty valid set leaves no mass
    st3, _, _, _ = O.row_probs(x, 1.0, allowed=words(np.zeros(5, bool)))
    assert st3 == O.ROW_NONFINITE


# ------------------------------------------------------------------------------ the round

def masked_batch(seed, B=6, gamma=3, V=97, density=0.4, shared=False):
    """Random logits, per-position valid sets (one per request when ``shared``), tokens from q_G."""
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((B, gamma + 1, V)) * 2).astype(np.float32)
    d = (t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.7).astype(np.float32)
    if shared:
        one = rng.random((B, 1, V)) < density
        valid = np.repeat(one, gamma + 1, axis=1)
    else:
        valid = rng.random((B, gamma + 1, V)) < density
    valid[:, :, 0] |= ~valid.any(-1)
    tok = S.gumbel_max_tokens(rng, d.astype(np.float64), valid[:, :gamma])
    u = S.uniforms_from(rng, (B, gamma + 2))
    return t, d, tok, u, valid


@pytest.mark.parametrize("seed", range(4))
def test_shared_mask_is_the_plain_round_on_the_compacted_vocabulary(seed):
    T = 0.9
    t, d, tok, u, valid = masked_batch(seed, shared=True)
    B, g1, V = t.shape
    got = O.spec_verify(t, d, tok, u, T, allowed=words(valid))
    for b in range(B):
        keep = np.flatnonzero(valid[b, 0])
        rank = -np.ones(V, np.int64)
        rank[keep] = np.arange(keep.size)
        ref = O.spec_verify(t[b:b + 1][:, :, keep], d[b:b + 1][:, :, keep],
                            rank[tok[b:b + 1]].astype(np.int32), u[b:b + 1], T)
        assert got["row_status"][b] == ref["row_status"][0] == O.ROW_OK
        assert got["accepted_len"][b] == ref["accepted_len"][0]
        A = ref["accepted_len"][0]
        assert np.array_equal(rank[got["out_tokens"][b, :A + 1]], ref["out_tokens"][0, :A + 1])
        assert np.all(got["out_tokens"][b, A + 1:] == -1)
        np.testing.assert_allclose(got["lse_p"][b], ref["lse_p"][0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["accept"][b], ref["accept"][0], rtol=1e-13, atol=0)


@pytest.mark.parametrize("seed", range(3))
def test_per_position_mask_equals_removed_logits(seed):
    """Each position with its own set: the round on -inf logits outside A_G (the pages' q_G).  The
    draft row of position i takes position i's set, the bonus row position gamma's."""
    t, d, tok, u, valid = masked_batch(100 + seed)
    g = d.shape[1]
    got = O.spec_verify(t, d, tok, u, 1.3, allowed=words(valid))
    tm = np.where(valid, t.astype(np.float64), -np.inf)
    dm = np.where(valid[:, :g], d.astype(np.float64), -np.inf)
    ref = O.spec_verify(tm, dm, tok, u, 1.3)
    for k in ("accepted_len", "out_tokens", "row_status"):
        assert np.array_equal(got[k], ref[k]), k
    np.testing.assert_allclose(got["lse_q"], ref["lse_q"], rtol=0, atol=1e-12)


def test_a_misplaced_draft_mask_fails_the_pin(tmp_path):
    """Plant a mistake (draft row i masked with position i + 1's set) and the pin above catches it."""
    lib = O.build_planted(
        [("/* the draft row of position i sampled under the same grammar state as target row i */\n"
          "            const uint32_t* m = allowed ? allowed + ((size_t)b * (size_t)(gamma + 1) + (size_t)i) * W : NULL;",
          "const uint32_t* m = allowed ? allowed + ((size_t)b * (size_t)(gamma + 1) + (size_t)i + 1) * W : NULL;")],
        str(tmp_path))
    t, d, tok, u, valid = masked_batch(7)
    B, g1, V = t.shape
    g = g1 - 1
    m = words(valid)
    acc = np.empty(B, np.int32)
    out = np.empty((B, g1), np.int32)
    st = np.empty(B, np.int32)
    lq = np.empty((B, g))
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    lib.oracle_spec_verify_masked.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] + \
        [ctypes.c_void_p] * 2 + [ctypes.c_int] * 3 + [ctypes.c_double] + [ctypes.c_void_p] * 8
    tok32 = np.ascontiguousarray(tok, np.int32)
    lib.oracle_spec_verify_masked(P(t), P(d), O.F32, P(tok32), P(u), B, g, V, 1.3, P(m), P(acc),
                                  P(out), P(st), None, P(lq), None, None)
    dm = np.where(valid[:, :g], d.astype(np.float64), -np.inf)
    ref = O.spec_verify(np.where(valid, t.astype(np.float64), -np.inf), dm, tok, u, 1.3)
    assert not (np.array_equal(st, ref["row_status"]) and np.array_equal(out, ref["out_tokens"])
                and np.allclose(lq, ref["lse_q"], atol=1e-9))


def test_full_mask_is_spec_verify_bit_for_bit():
    b = S.make_spec_batch(S.scaled(S.CONFIGS["c2"], B=4, V=1000))
    full = np.full((4, b.cfg.gamma + 1, (1000 + 31) // 32), 0xFFFFFFFF, np.uint32)
    a = O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, 1.0)
    m = O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, 1.0, allowed=full)
    for k in a:
        assert np.array_equal(a[k], m[k], equal_nan=True), k


def test_bits_beyond_V_are_ignored():
    t, d, tok, u, valid = masked_batch(3, V=45)
    w = words(valid)
    w2 = w.copy()
    w2[..., -1] |= np.uint32(0xFFFFFFFF) << np.uint32(45 % 32)
    a = O.spec_verify(t, d, tok, u, 1.0, allowed=w)
    m = O.spec_verify(t, d, tok, u, 1.0, allowed=w2)
    for k in a:
        assert np.array_equal(a[k], m[k], equal_nan=True), k


def test_edge_statuses():
    t, d, tok, u, valid = masked_batch(5, B=3)
    g = d.shape[1]
    v = valid.copy()
    v[0, 1, tok[0, 1]] = False          # a drafted token outside A_G: q_G(x) = 0
    v[1, g] = False                     # the bonus position has no valid token
    r = O.spec_verify(t, d, tok, u, 1.0, allowed=words(v))
    assert r["row_status"][0] == O.ROW_BAD_TOKEN
    assert r["row_status"][1] == O.ROW_NONFINITE
    assert r["row_status"][2] == O.ROW_OK
    assert np.all(r["out_tokens"][:2] == -1) and np.all(r["accepted_len"][:2] == -1)


# ------------------------------------------------------------------------------ exact law

def test_masked_emitted_law_by_enumeration():
    """gamma = 2, V = 5 with a different valid set at each of the three positions.  p_G and q_G are
    dyadic on their sets; the removed tokens carry junk logits (one of them NaN).  Enumerating every
    draft path (weighted by q_G) and a midpoint grid of every uniform gives the emitted law, which
    must be p_G at every reached position."""
    A_sets = [np.array([1, 1, 0, 1, 0], bool), np.array([0, 1, 1, 1, 1], bool),
              np.array([1, 0, 1, 0, 1], bool)]
    pG = [np.array([0.5, 0.25, 0, 0.25, 0]), np.array([0, 0.125, 0.375, 0.25, 0.25]),
          np.array([0.25, 0, 0.5, 0, 0.25])]
    qG = [np.array([0.25, 0.5, 0, 0.25, 0]), np.array([0, 0.25, 0.25, 0.25, 0.25])]
    junk = np.array([7.0, np.nan, -3.0, 40.0, 1.5])

    def row(probs, valid):
        with np.errstate(divide="ignore"):
            lg = np.log(probs)
        return np.where(valid, lg, junk)

    gamma, V, M = 2, 5, 8
    paths = [x for x in itertools.product(range(V), repeat=gamma)
             if all(qG[i][x[i]] > 0 for i in range(gamma))]
    pw = np.array([qG[0][x[0]] * qG[1][x[1]] for x in paths])
    grid = (np.arange(M) + 0.5) / M
    G = np.stack(np.meshgrid(*([grid] * (gamma + 2)), indexing="ij"), -1).reshape(-1, gamma + 2)
    n = len(paths) * len(G)
    toks = np.repeat(np.array(paths, np.int32), len(G), 0)
    u = np.tile(G, (len(paths), 1)).astype(np.float32)
    w = np.repeat(pw, len(G)) / len(G)
    t = np.broadcast_to(np.stack([row(pG[i], A_sets[i]) for i in range(3)]), (n, 3, V)).copy()
    d = np.broadcast_to(np.stack([row(qG[i], A_sets[i]) for i in range(2)]), (n, 2, V)).copy()
    m = np.broadcast_to(words(np.stack(A_sets)), (n, 3, 1)).copy()
    out = O.spec_verify(t, d, toks, u, 1.0, allowed=m)
    assert np.all(out["row_status"] == O.ROW_OK)
    A = out["accepted_len"]
    for pos in range(3):
        reached = A >= pos
        law = np.zeros(V)
        np.add.at(law, out["out_tokens"][reached, pos], w[reached])
        np.testing.assert_allclose(law / w[reached].sum(), pG[pos], atol=1e-12)
    assert w[A >= 1].sum() == pytest.approx(np.minimum(pG[0], qG[0]).sum(), abs=1e-12)
