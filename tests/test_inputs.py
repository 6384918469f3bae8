"""The seeded input recipes of the processor and typical-acceptance workloads, and the benchmark's
host-side description of them (CPU only).

The draft tokens of a processed workload must be draws from the processed q: a token outside the
draft row's kept set would make the verify step report a bad token instead of verifying it.  These
tests check each recipe against the oracle's own reading of the processor.
"""
import os
import sys

import numpy as np

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_draft_nucleus_matches_the_oracle_kept_set():
    b = S.make_spec_batch(S.scaled(S.TOPP_CONFIGS["c11"], B=3, V=3000))
    keep = S.draft_nucleus_mask(S.stored_to_f64(b.draft), b.cfg.temperature, b.cfg.top_p)
    for r in range(3):
        for i in range(b.cfg.gamma):
            st, p, _, _, _ = O.row_probs_topp(b.draft[r, i], b.cfg.temperature, b.cfg.top_p)
            assert st == O.ROW_OK
            assert np.array_equal(p > 0, keep[r, i])
            assert keep[r, i, b.draft_tokens[r, i]]


def test_topp_workload_has_no_bad_tokens():
    b = S.make_spec_batch(S.scaled(S.TOPP_CONFIGS["c11"], B=4, V=5000))
    o = O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, b.cfg.temperature,
                      top_p=b.cfg.top_p)
    assert np.all(o["row_status"] == O.ROW_OK)


def test_grammar_sets_mix_and_drafts_stay_inside():
    b = S.make_spec_batch(S.scaled(S.MASK_CONFIGS["c9"], B=12, V=4000))
    valid = S.unpack_valid_sets(b.allowed, 4000)
    sizes = valid.sum(-1)
    assert (sizes == 64).any() and (sizes > 3800).any() and ((sizes > 1600) & (sizes < 2400)).any()
    for r in range(12):
        for i in range(b.cfg.gamma):
            assert valid[r, i, b.draft_tokens[r, i]]
    # the words round-trip and carry no bits past V
    assert np.array_equal(S.pack_valid_sets(valid), b.allowed)


def test_typical_workload_inputs():
    tb = S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c10"], B=3, V=2000))
    assert tb.uniforms is not None and tb.uniforms.shape == (3,)
    assert np.all((tb.uniforms >= 0) & (tb.uniforms < 1))
    o = O.tree_verify_typical(tb.logits, tb.parents, tb.tokens, tb.uniforms, tb.cfg.temperature,
                              tb.cfg.eps, tb.cfg.delta)
    assert np.all(o["row_status"] == O.ROW_OK)


def test_bench_describes_every_workload():
    import bench
    for n in ("c1", "c2", "c3", "c4", "c5", "c6", "c7", "c8", "c9", "c10", "c11"):
        text = bench.describe((n,))
        assert text.startswith(n + " ")
        assert n in bench.KERNEL_OF
    assert "spec_verify_topp" in bench.describe(("c11",))
    assert "spec_verify_masked" in bench.describe(("c9",))
    assert "tree_verify_typical" in bench.describe(("c10",))
