"""The bounded waits' give-up path, reached on the GPU without a fault.

Every wait of the streaming kernels (a chunk's bulk copy landing, a ring stage freed by the CTA's
consumer warps, a top-k segment's first bound and its completion) is bounded.  With the limit set
to 0 polls (spec_set_wait_limit, a test aid) every such wait gives up at once, so every request of
a streaming call must come back abandoned: row_status SPEC_ROW_TIMEOUT, accepted_len -1 and every
emitted token -1 ("Exact speculative and assisted decoding for TinyRustLM", "Normative edge-case
behavior": abort without emitting).  The copies already in flight are still waited for with the
full limit before a CTA leaves, so the next call, at the default limit, must match the oracle.
Outputs and workspaces sit inside guard bands here too.
"""
import numpy as np
import pytest

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import compare_spec, compare_tree, dev, guarded_call, run_oracle_spec

pytestmark = pytest.mark.gpu

TIMEOUT = 4


@pytest.fixture
def give_up_at_once():
    prev = sv.set_wait_limit(0)
    try:
        yield
    finally:
        sv.set_wait_limit(-1)
    assert prev == 1 << 22


def _abandoned(out, B):
    assert np.all(out["row_status"] == TIMEOUT), np.unique(out["row_status"]).tolist()
    assert np.all(out["accepted_len"] == -1)
    assert np.all(out["out_tokens"] == -1)
    assert out["row_status"].shape[0] == B


def _spec(b, **kw):
    return guarded_call(sv.spec_verify, dev(b.target), dev(b.draft), dev(b.draft_tokens),
                        dev(b.uniforms), b.cfg.temperature, aux=True, **kw)


@pytest.mark.parametrize("top_k", [0, 50])
def test_spec_verify_times_out_then_recovers(top_k):
    b = S.make_spec_batch(S.scaled(S.CONFIGS["c2"], top_k=top_k, seed=12000 + top_k))
    sv.set_wait_limit(0)
    try:
        _abandoned(_spec(b, top_k=top_k), b.cfg.B)
    finally:
        sv.set_wait_limit(-1)
    compare_spec(_spec(b, top_k=top_k), run_oracle_spec(b, top_k))


def test_processors_time_out(give_up_at_once):
    b = S.make_spec_batch(S.scaled(S.TOPP_CONFIGS["c11"], B=8, V=32000, seed=12100))
    _abandoned(_spec(b, top_p=b.cfg.top_p), 8)
    m = S.make_spec_batch(S.scaled(S.MASK_CONFIGS["c9"], B=8, V=32000, seed=12101))
    words = dev(np.ascontiguousarray(m.allowed, np.uint32).view(np.int32))
    _abandoned(_spec(m, allowed=words), 8)


def test_tree_verify_greedy_times_out_then_recovers():
    tb = S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c5"], B=8, V=32000, seed=12200))
    sv.set_wait_limit(0)
    try:
        g = guarded_call(sv.tree_verify_greedy, dev(tb.logits), dev(tb.parents), dev(tb.tokens))
        _abandoned(g, 8)
        assert np.all(g["out_nodes"] == -1)
        c = guarded_call(sv.spec_verify_greedy, dev(tb.logits[:, :5]), dev(tb.tokens[:, :4]))
        _abandoned(c, 8)
    finally:
        sv.set_wait_limit(-1)
    compare_tree(guarded_call(sv.tree_verify_greedy, dev(tb.logits), dev(tb.parents),
                              dev(tb.tokens)),
                 O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens))


def test_typical_and_smc_time_out(give_up_at_once):
    yb = S.make_tree_batch(S.scaled(S.TREE_CONFIGS["c10"], B=4, V=32000, seed=12300))
    c = yb.cfg
    g = guarded_call(sv.tree_verify_typical, dev(yb.logits), dev(yb.parents), dev(yb.tokens),
                     dev(yb.uniforms), c.temperature, c.eps, c.delta)
    _abandoned(g, 4)
    sb = S.make_smc_batch(S.scaled(S.SMC_CONFIGS["c7"], groups=2, V=32000, seed=12301))
    o = guarded_call(sv.smc_verify, dev(sb.target), dev(sb.draft), dev(sb.draft_tokens),
                     dev(sb.log_weights), dev(sb.uniforms), sb.cfg.groups, sb.cfg.temperature,
                     sb.cfg.eta)
    _abandoned(o, sb.cfg.B)
    assert np.all(o["resampled"] == -1) and np.all(np.isnan(o["ess"]))


def test_default_limit_is_restored():
    assert sv.set_wait_limit(-1) == 1 << 22
