"""GPU parity of the stochastic tree verify (tree_verify_sample) against the fp64 oracle.

Matching rule (the same as the chain verify's): status, path length, path tokens and the final
token bit-exact, except on requests where a uniform the walk used lies within 1e-6 of a decision
boundary (the oracle's margin); accept ratios of tested nodes within 1e-5 absolute, and the set of
tested nodes identical.  The full-size workload (B=32, 64 nodes, V=128256) is compared request by
request: the oracle reads only the rows the walk visits, so it finishes in well under a second.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import BOUNDARY, TOL, dev, guarded_call

pytestmark = pytest.mark.gpu

C6 = S.SAMPLE_TREE_CONFIGS["c6"]


def run_gpu(tb, T=None, max_out=None):
    return guarded_call(sv.tree_verify_sample, dev(tb.target), dev(tb.draft), dev(tb.parents),
                        dev(tb.tokens), dev(tb.qrow), dev(tb.uniforms),
                        tb.cfg.temperature if T is None else T, max_out=max_out, aux=True,
                        guard_ws=False)


def run_oracle(tb, T=None, max_out=None):
    return O.tree_verify_sample(tb.target, tb.draft, tb.parents, tb.tokens, tb.qrow, tb.uniforms,
                                tb.cfg.temperature if T is None else T, max_out=max_out)


def compare(g, o):
    """Returns (requests, near-boundary requests, mismatched requests); raises on a violation."""
    st = o["row_status"]
    flagged = o["margin"] < BOUNDARY
    same = ((g["row_status"] == st) & (g["accepted_len"] == o["accepted_len"])
            & np.all(g["out_tokens"] == o["out_tokens"], 1))
    if o["out_nodes"].size:
        same &= np.all(g["out_nodes"][:, : o["out_nodes"].shape[1]] == o["out_nodes"], 1)
    bad = ~same & ~flagged
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(
            f"{bad.sum()} unflagged mismatches; request {i}: gpu st={g['row_status'][i]} "
            f"A={g['accepted_len'][i]} tok={g['out_tokens'][i].tolist()} | oracle "
            f"st={st[i]} A={o['accepted_len'][i]} tok={o['out_tokens'][i].tolist()} "
            f"margin={o['margin'][i]:.3g}")
    # accept ratios: the same nodes tested, values within TOL
    N = o["accept"].shape[1]
    if N:
        ga = g["accept"][:, :N].astype(np.float64)
        ok = same & (st == 0)
        np.testing.assert_array_equal(np.isnan(ga[ok]), np.isnan(o["accept"][ok]))
        d = np.abs(np.nan_to_num(ga[ok]) - np.nan_to_num(o["accept"][ok]))
        assert d.size == 0 or d.max() <= TOL, f"accept ratio diff {d.max():.3g}"
    return len(st), int(flagged.sum()), int((~same).sum())


def test_c6_full_size():
    tb = S.make_sample_tree_batch(C6)
    g, o = run_gpu(tb), run_oracle(tb)
    n, flagged, mism = compare(g, o)
    assert np.all(o["row_status"] == 0)
    # the walk took both branches: some paths accepted, some corrections
    assert o["accepted_len"].max() >= 1 and (o["accepted_len"] == 0).any()


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (7, "bf16"), (1000, "bf16"), (1000, "f32"),
                                     (4099, "bf16"), (32000, "bf16"), (32001, "f32"),
                                     (70000, "f32"), (152064, "bf16"), (200000, "bf16")])
def test_shapes(V, dtype):
    """Several tiles and ragged tails; cluster sizes 1..16; aligned and unaligned rows."""
    cfg = S.scaled(C6, B=12, V=V, dtype=dtype, seed=2000 + V)
    tb = S.make_sample_tree_batch(cfg)
    compare(run_gpu(tb), run_oracle(tb))


@pytest.mark.parametrize("branching,max_nodes", [((1, 1, 1, 1, 1), 5), ((8,), 8), ((3, 3, 3), 39),
                                                 ((2, 2, 2, 2, 2, 2), 126)])
@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_tree_shapes_and_temperatures(branching, max_nodes, T):
    cfg = S.scaled(C6, B=48, V=5000, branching=branching, max_nodes=max_nodes, temperature=T,
                   seed=3000 + max_nodes)
    tb = S.make_sample_tree_batch(cfg)
    compare(run_gpu(tb), run_oracle(tb))


def test_many_requests_small_vocab():
    """Mismatches only on draws within 1e-6 of a decision boundary, and under 0.01% of requests:
    20,000 requests over a 64-token vocabulary, where residuals often hold tiny masses."""
    cfg = S.scaled(C6, B=20000, V=64, branching=(3, 2), max_nodes=9, temperature=1.0, seed=4242)
    tb = S.make_sample_tree_batch(cfg)
    n, flagged, mism = compare(run_gpu(tb), run_oracle(tb))
    print(f"requests={n} near-boundary={flagged} mismatched={mism}")
    assert mism < 1e-4 * n


def test_distinct_proposal_rows_per_child():
    """Siblings drawn from different proposal rows (several drafters): the walk loads each row."""
    cfg = S.scaled(C6, B=64, V=3000, branching=(4, 2), max_nodes=12, seed=77)
    tb = S.make_sample_tree_batch(cfg)
    rng = np.random.default_rng(5)
    B, N = tb.parents.shape
    qrow = rng.integers(0, N + 1, size=(B, N)).astype(np.int32)
    tok = np.empty_like(tb.tokens)
    for b in range(B):
        for i in range(N):
            z = S.stored_to_f64(tb.draft[b, qrow[b, i]]) / cfg.temperature
            tok[b, i] = S.gumbel_max_tokens(rng, z[None])[0]
    tb.qrow, tb.tokens = qrow, tok
    compare(run_gpu(tb), run_oracle(tb))


def test_chain_and_empty_tree():
    for par in ([-1, 0, 1, 2, 3], []):
        cfg = S.scaled(C6, B=40, V=2000, seed=9 + len(par))
        tb = S.make_sample_tree_batch(cfg, parents=par)
        compare(run_gpu(tb), run_oracle(tb))


def test_statuses_and_edge_cases():
    cfg = S.scaled(C6, B=12, V=600, branching=(2, 2), max_nodes=6, dtype="f32", seed=31)
    tb = S.make_sample_tree_batch(cfg)
    t, d = tb.target.copy(), tb.draft.copy()
    par, tok, qr, u = tb.parents.copy(), tb.tokens.copy(), tb.qrow.copy(), tb.uniforms.copy()
    par[0, 3] = 5                        # bad parent
    qr[1, 2] = 7                         # proposal row outside [0, Nq)
    tok[2, 4] = 600                      # token outside [0, V)
    u[3, 6] = 1.0                        # uniform outside [0, 1) (the final slot)
    t[4, 0, 17] = np.nan                 # NaN in the frontier row: always visited
    t[5, 5, 3] = np.inf                  # +inf in a leaf row: seen only if the walk reaches it
    d[6, 0, tok[6, 0]] = -np.inf         # q(x) = 0 for the first tested node
    d[7, 0, :] = -np.inf                 # a proposal row with no finite entry
    t[8, 0, :] = -np.inf                 # a target row with no finite entry
    t[9, 0, :] = 0.0                     # constant rows
    d[9, 0, :] = 0.0
    u[10, :] = 0.0                       # every test accepts (as far as a > 0)
    u[11, :] = np.nextafter(np.float32(1), np.float32(0))  # every test rejects unless a = 1
    tb.target, tb.draft, tb.parents, tb.tokens, tb.qrow, tb.uniforms = t, d, par, tok, qr, u
    g, o = run_gpu(tb), run_oracle(tb)
    compare(g, o)
    assert o["row_status"][0] == O.ROW_BAD_PARENT
    assert o["row_status"][1] == O.ROW_BAD_QROW
    assert o["row_status"][2] == O.ROW_BAD_TOKEN
    assert o["row_status"][3] == O.ROW_BAD_UNIFORM
    assert o["row_status"][4] == O.ROW_NONFINITE
    assert o["row_status"][6] == O.ROW_BAD_TOKEN
    assert o["row_status"][7] == O.ROW_NONFINITE
    assert o["row_status"][8] == O.ROW_NONFINITE
    for b in range(4):
        assert g["accepted_len"][b] == -1 and np.all(g["out_tokens"][b] == -1)
        assert np.all(np.isnan(g["accept"][b]))


def test_output_overflow():
    cfg = S.scaled(C6, B=30, V=500, branching=(1, 1, 1, 1), max_nodes=4, seed=12)
    tb = S.make_sample_tree_batch(cfg)
    tb.uniforms[:] = 0.0  # accept along the chain wherever a > 0
    for max_out in (1, 2, 3, 5):
        g, o = run_gpu(tb, max_out=max_out), run_oracle(tb, max_out=max_out)
        compare(g, o)
    assert (o["row_status"] == 0).any()


def test_repeat_calls_are_deterministic():
    tb = S.make_sample_tree_batch(S.scaled(C6, B=16, V=50000, seed=8))
    a, b = run_gpu(tb), run_gpu(tb)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_unaligned_rows_take_the_element_path():
    cfg = S.scaled(C6, B=8, V=5001, seed=21)
    tb = S.make_sample_tree_batch(cfg)
    g_ref = run_gpu(tb)
    # the same logits one element into a larger buffer: rows no longer start on 16 bytes
    for name in ("target", "draft"):
        a = getattr(tb, name)
        flat = np.empty(a.size + 1, a.dtype)
        flat[1:] = a.ravel()
        setattr(tb, name + "_shifted", flat)
    t = dev(tb.target_shifted)[1:].view(tb.target.shape)
    d = dev(tb.draft_shifted)[1:].view(tb.draft.shape)
    out = guarded_call(sv.tree_verify_sample, t, d, dev(tb.parents), dev(tb.tokens), dev(tb.qrow),
                       dev(tb.uniforms), cfg.temperature, aux=True, guard_ws=False)
    for k in out:
        np.testing.assert_array_equal(out[k], g_ref[k])
    compare(g_ref, run_oracle(tb))


@pytest.mark.parametrize("cl", [1, 2, 4, 8, 16])
def test_forced_cluster_sizes(cl):
    """The walk gives the oracle's results whatever the cluster size (the measurement aid that
    forces it); a size whose slices cannot hold the row is refused."""
    cfg = S.scaled(C6, B=6, V=16384, seed=2100 + cl)
    tb = S.make_sample_tree_batch(cfg)
    prev = sv.set_tree_sample_cluster(cl)
    try:
        compare(run_gpu(tb), run_oracle(tb))
        if cl < 8:  # V = 128256 needs 8 CTAs of 512 threads at 4 vectors per thread
            big = S.make_sample_tree_batch(S.scaled(C6, B=1, seed=2200))
            with pytest.raises(sv.SpecVerifyError):
                sv.tree_verify_sample(dev(big.target), dev(big.draft), dev(big.parents),
                                      dev(big.tokens), dev(big.qrow), dev(big.uniforms),
                                      big.cfg.temperature)
    finally:
        sv.set_tree_sample_cluster(prev)
