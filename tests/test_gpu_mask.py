"""GPU parity of spec_verify_masked (grammar mask) against the fp64 oracle on the same seeded inputs.

The grammar-masked workload (c3's logits with a mixed valid-set recipe per position) runs at full
size in the launch configuration the benchmark uses; smaller shapes cover several stream chunks,
ragged tails, the scalar path (rows that are not 16-byte aligned) and gamma past one warp of rows.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import compare_spec, dev, guarded_call

pytestmark = pytest.mark.gpu


def words_dev(words):
    return torch.from_numpy(np.ascontiguousarray(words, np.uint32).view(np.int32)).cuda()


def run_gpu(b, allowed=None, target=None, draft=None):
    a = b.allowed if allowed is None else allowed
    return guarded_call(sv.spec_verify_masked, dev(b.target) if target is None else target,
                        dev(b.draft) if draft is None else draft,
                        dev(b.draft_tokens), dev(b.uniforms), words_dev(a),
                        b.cfg.temperature, aux=True)


def run_oracle(b, allowed=None, idx=None):
    a = b.allowed if allowed is None else allowed
    sl = slice(None) if idx is None else idx
    return O.spec_verify(b.target[sl], b.draft[sl], b.draft_tokens[sl], b.uniforms[sl],
                         b.cfg.temperature, allowed=a[sl])


def masked(name="c9", **kw):
    return S.make_spec_batch(S.scaled(S.MASK_CONFIGS[name], **kw))


def test_c9_grammar_masked_full_size():
    b = masked()
    n, flagged, mism = compare_spec(run_gpu(b), run_oracle(b))
    assert n == 64 and mism <= flagged


@pytest.mark.parametrize("V", [1, 7, 8, 33, 1000, 4099, 40003, 40000])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_masked_shapes(V, dtype):
    b = masked(B=6, V=V, dtype=dtype, seed=9100 + V)
    compare_spec(run_gpu(b), run_oracle(b))


@pytest.mark.parametrize("gamma", [0, 1, 31, 32, 40])
def test_masked_gamma_range(gamma):
    b = masked(B=3, gamma=gamma, V=5000, seed=9200 + gamma)
    compare_spec(run_gpu(b), run_oracle(b))


@pytest.mark.parametrize("gamma", [3, 40])
def test_masked_unaligned_rows(gamma):
    """Row starts that are not 16-byte aligned take the scalar path."""
    b = masked(B=4, gamma=gamma, V=3000, seed=9300 + gamma)
    t = torch.empty(b.target.size + 1, dtype=torch.int16, device="cuda")
    d = torch.empty(b.draft.size + 1, dtype=torch.int16, device="cuda")
    t[1:] = dev(b.target).view(-1)
    d[1:] = dev(b.draft).view(-1)
    g = run_gpu(b, target=t[1:].view(b.target.shape), draft=d[1:].view(b.draft.shape))
    compare_spec(g, run_oracle(b))


def test_full_mask_equals_spec_verify():
    b = masked(B=16, V=20000, seed=9400)
    full = np.full_like(b.allowed, 0xFFFFFFFF)
    g = run_gpu(b, allowed=full)
    out = guarded_call(sv.spec_verify, dev(b.target), dev(b.draft), dev(b.draft_tokens),
                       dev(b.uniforms), b.cfg.temperature, aux=True)
    for k, v in out.items():
        np.testing.assert_array_equal(g[k], v, err_msg=k)


def test_single_valid_token_is_forced():
    """A_G = {x} at every position: p_G = q_G = the point mass, so every draft is accepted and the
    bonus is the bonus position's one valid token."""
    b = masked(B=5, V=4099, seed=9500)
    B, g1, W = b.allowed.shape
    rng = np.random.default_rng(0)
    forced = rng.integers(0, 4099, size=(B, g1))
    valid = np.zeros((B, g1, 4099), bool)
    np.put_along_axis(valid, forced[..., None], True, axis=-1)
    a = S.pack_valid_sets(valid)
    b.draft_tokens[:] = forced[:, :-1]
    g = run_gpu(b, allowed=a)
    o = run_oracle(b, allowed=a)
    compare_spec(g, o)
    assert np.all(g["accepted_len"] == g1 - 1)
    np.testing.assert_array_equal(g["out_tokens"], forced)


def test_masked_statuses_and_removed_nan():
    b = masked(B=4, V=2048, seed=9600)
    g1 = b.cfg.gamma + 1
    valid = S.unpack_valid_sets(b.allowed, 2048)
    valid[0, 1, b.draft_tokens[0, 1]] = False      # drafted token outside A_G: BAD_TOKEN
    valid[1, g1 - 1] = False                       # empty valid set at the bonus position
    # a NaN and a +inf at removed tokens of request 2 are never read
    gone = np.flatnonzero(~valid[2, 0])[:2]
    b.target[2, 0, gone[0]] = 0x7FC0
    b.draft[2, 0, gone[1]] = 0x7F80
    a = S.pack_valid_sets(valid)
    g = run_gpu(b, allowed=a)
    o = run_oracle(b, allowed=a)
    compare_spec(g, o)
    assert g["row_status"].tolist()[:3] == [O.ROW_BAD_TOKEN, O.ROW_NONFINITE, O.ROW_OK]


def test_masked_repeat_calls_are_deterministic():
    b = masked(B=16, seed=9700)
    a1, a2 = run_gpu(b), run_gpu(b)
    for k in a1:
        np.testing.assert_array_equal(a1[k], a2[k])
