"""GPU parity of tree_verify_typical against the fp64 oracle on the same seeded inputs.

The typical-acceptance workload (c5's tree and logits, T = 0.7, eps = 0.09, delta = 0.3) runs at
full size in the launch configuration the benchmark uses.  Smaller shapes cover several stream
chunks, ragged tails, the scalar path (odd vocabularies, unaligned rows), trees from empty to
hundreds of nodes, and every status.

Matching rules: statuses, accepted lengths, path nodes and tokens bit-exact, except on requests
whose oracle margin (the smallest |ln p - ln threshold| of a deciding test, or |u - C| at the drawn
token's CDF boundaries) is below 1e-5; entropies and log-probabilities within 1e-5 absolute.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import dev, guarded_call

pytestmark = pytest.mark.gpu

FLAG = 1e-5
TOL = 1e-5


def run_gpu(tb, logits=None, eps=None, delta=None, max_out=None):
    c = tb.cfg
    return guarded_call(sv.tree_verify_typical, dev(tb.logits) if logits is None else logits,
                        dev(tb.parents), dev(tb.tokens), dev(tb.uniforms), c.temperature,
                        c.eps if eps is None else eps, c.delta if delta is None else delta,
                        max_out=max_out, aux=True)


def run_oracle(tb, eps=None, delta=None, max_out=None):
    c = tb.cfg
    return O.tree_verify_typical(tb.logits, tb.parents, tb.tokens, tb.uniforms, c.temperature,
                                 c.eps if eps is None else eps, c.delta if delta is None else delta,
                                 max_out)


def compare(g, o):
    np.testing.assert_array_equal(g["row_status"], o["row_status"], err_msg="status")
    flagged = o["margin"] < FLAG
    same = (g["accepted_len"] == o["accepted_len"]) & np.all(g["out_tokens"] == o["out_tokens"], 1)
    if o["out_nodes"].shape[1] > 0:
        same &= np.all(g["out_nodes"][:, :o["out_nodes"].shape[1]] == o["out_nodes"], 1)
    bad = ~same & ~flagged
    assert not bad.any(), (f"{bad.sum()} unflagged mismatches, first request "
                           f"{int(np.flatnonzero(bad)[0])}")
    ok = o["row_status"] == 0
    if ok.any():
        d = np.abs(g["entropy"][ok].astype(np.float64) - o["entropy"][ok])
        assert d.max() <= TOL, f"entropy: {d.max():.3g}"
        N = o["logp"].shape[1]
        if N:
            lo, lg = o["logp"][ok], g["logp"][ok][:, :N].astype(np.float64)
            fin = np.isfinite(lo)
            assert np.array_equal(fin, np.isfinite(lg))
            d = np.abs(lg[fin] - lo[fin])
            assert d.size == 0 or d.max() <= TOL, f"logp: {d.max():.3g}"
    return int(flagged.sum()), int((~same).sum())


def typical(**kw):
    return S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c10"], **kw))


def test_c10_typical_full_size():
    tb = typical()
    flagged, mism = compare(run_gpu(tb), run_oracle(tb))
    assert mism <= flagged


@pytest.mark.parametrize("V", [1, 7, 8, 33, 1000, 4099, 40003, 40000])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_typical_shapes(V, dtype):
    tb = typical(B=5, V=V, dtype=dtype, seed=10100 + V)
    if V == 1:
        tb.tokens[:] = 0
    compare(run_gpu(tb), run_oracle(tb))


@pytest.mark.parametrize("branching,max_nodes", [((4,), 0), ((1,), 1), ((4, 4, 2, 2), 64),
                                                 ((3, 3, 3, 3, 3), 200), ((1,) * 40, 40)])
def test_typical_tree_sizes(branching, max_nodes):
    tb = typical(B=6, V=5000, branching=branching, max_nodes=max_nodes, seed=10200 + max_nodes)
    compare(run_gpu(tb), run_oracle(tb))


def test_typical_unaligned_rows():
    tb = typical(B=4, V=3000, seed=10300)
    t = torch.empty(tb.logits.size + 1, dtype=torch.int16, device="cuda")
    t[1:] = dev(tb.logits).view(-1)
    compare(run_gpu(tb, logits=t[1:].view(tb.logits.shape)), run_oracle(tb))


@pytest.mark.parametrize("eps,delta", [(0.0, 0.3), (0.5, 1e6), (1.0, 1.0), (0.09, 0.0)])
def test_typical_thresholds(eps, delta):
    tb = typical(B=8, V=20000, seed=10400)
    compare(run_gpu(tb, eps=eps, delta=delta), run_oracle(tb, eps=eps, delta=delta))


def test_typical_statuses():
    tb = typical(B=6, V=2048, seed=10500)
    tb.logits[0, 3, 17] = 0x7FC0               # NaN in a row
    tb.parents[1, 5] = 5                       # a parent that does not precede its node
    tb.tokens[2, 7] = 2048                     # a token outside [0, V)
    tb.uniforms[3] = 1.0                       # a uniform outside [0, 1)
    tb.logits[4, 2, :] = 0xFF80                # a row with no finite entry
    g, o = run_gpu(tb), run_oracle(tb)
    compare(g, o)
    assert g["row_status"].tolist() == [O.ROW_NONFINITE, O.ROW_BAD_PARENT, O.ROW_BAD_TOKEN,
                                        O.ROW_BAD_UNIFORM, O.ROW_NONFINITE, O.ROW_OK]
    # the path and the final token must fit in max_out
    tb2 = typical(B=4, V=2048, seed=10501)
    compare(run_gpu(tb2, eps=0.0, max_out=3), run_oracle(tb2, eps=0.0, max_out=3))
    assert np.all(run_gpu(tb2, eps=0.0, max_out=3)["row_status"] == O.ROW_OVERFLOW)


def test_typical_repeat_calls_are_deterministic():
    tb = typical(B=8, seed=10600)
    a, b = run_gpu(tb), run_gpu(tb)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
