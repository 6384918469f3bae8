"""GPU parity of linear greedy verify (spec_verify_greedy) against the oracle: bit-exact, argmax
ties to the lowest index."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import dev, guarded_call

pytestmark = pytest.mark.gpu

C8 = S.TREE_CONFIGS["c8"]


def run(tb):
    return guarded_call(sv.spec_verify_greedy, dev(tb.logits), dev(tb.tokens))


def check(tb):
    g, o = run(tb), O.spec_verify_greedy(tb.logits, tb.tokens)
    for k in ("row_status", "accepted_len", "out_tokens"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    return o


def test_c8_full_size():
    o = check(S.make_tree_batch(C8))
    assert np.all(o["row_status"] == 0)
    assert o["accepted_len"].min() < 5 and o["accepted_len"].max() >= 1


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (9, "bf16"), (1000, "f32"), (32001, "bf16"),
                                     (152064, "bf16")])
@pytest.mark.parametrize("gamma", [0, 1, 5, 33])
def test_shapes(V, dtype, gamma):
    cfg = S.scaled(C8, B=6, V=V, dtype=dtype, branching=(1,) * max(gamma, 1), max_nodes=gamma,
                   seed=5000 + V + gamma)
    check(S.make_tree_batch(cfg))


def test_ties_and_statuses():
    cfg = S.scaled(C8, B=6, V=300, dtype="f32", seed=5100)
    tb = S.make_tree_batch(cfg)
    tb.logits[0, 2, :] = 1.0                  # a constant row: argmax is token 0
    tb.tokens[0, :2] = np.argmax(tb.logits[0, :2], axis=-1)
    tb.tokens[0, 2] = 0
    tb.logits[1, 3, 5] = np.nan               # a NaN row
    tb.tokens[2, 1] = 300                      # a token outside [0, V)
    tb.logits[3, :, :] = -np.inf              # no finite entry
    o = check(tb)
    assert o["accepted_len"][0] >= 3
    assert list(o["row_status"][1:4]) == [O.ROW_NONFINITE, O.ROW_BAD_TOKEN, O.ROW_NONFINITE]
