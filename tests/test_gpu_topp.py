"""GPU parity of spec_verify_topp (top-p processor on every row) against the fp64 oracle.

The top-p workload (c2's peaked target recipe at c3's sizes, T = 0.8, top_p = 0.9) runs at full size
in the launch configuration the benchmark uses; smaller shapes cover several stream chunks, ragged
tails, the scalar path, gamma past one warp of rows, ties at the threshold and the statuses.  The
matching rules are the plain round's; a request is exempt only when the oracle's margin (which also
covers how close each row's kept mass came to top_p) is below 1e-6.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import compare_spec, dev, guarded_call

pytestmark = pytest.mark.gpu


def run_gpu(b, top_p=None, target=None, draft=None):
    return guarded_call(sv.spec_verify_topp, dev(b.target) if target is None else target,
                        dev(b.draft) if draft is None else draft,
                        dev(b.draft_tokens), dev(b.uniforms), b.cfg.temperature,
                        b.cfg.top_p if top_p is None else top_p, aux=True)


def run_oracle(b, top_p=None):
    return O.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, b.cfg.temperature,
                         top_p=b.cfg.top_p if top_p is None else top_p)


def topp(**kw):
    return S.make_spec_batch(S.scaled(S.TOPP_CONFIGS["c11"], **kw))


def test_c11_topp_full_size():
    b = topp()
    n, flagged, mism = compare_spec(run_gpu(b), run_oracle(b))
    assert n == 64 and mism <= flagged


@pytest.mark.parametrize("V", [1, 7, 8, 33, 1000, 4099, 40003, 40000])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topp_shapes(V, dtype):
    b = topp(B=6, V=V, dtype=dtype, seed=11100 + V)
    compare_spec(run_gpu(b), run_oracle(b))


@pytest.mark.parametrize("top_p", [1e-6, 0.3, 0.75, 0.99, 0.9999])
def test_topp_levels(top_p):
    b = topp(B=8, V=20000, top_p=top_p, seed=11200)
    compare_spec(run_gpu(b), run_oracle(b))


@pytest.mark.parametrize("gamma", [0, 1, 31, 40])
def test_topp_gamma_range(gamma):
    b = topp(B=3, gamma=gamma, V=5000, seed=11300 + gamma)
    compare_spec(run_gpu(b), run_oracle(b))


def test_topp_unaligned_rows():
    b = topp(B=4, V=3000, seed=11400)
    t = torch.empty(b.target.size + 1, dtype=torch.int16, device="cuda")
    d = torch.empty(b.draft.size + 1, dtype=torch.int16, device="cuda")
    t[1:] = dev(b.target).view(-1)
    d[1:] = dev(b.draft).view(-1)
    g = run_gpu(b, target=t[1:].view(b.target.shape), draft=d[1:].view(b.draft.shape))
    compare_spec(g, run_oracle(b))


def test_topp_ties_at_the_threshold():
    """Logits on a coarse grid (many equal values): the group at the threshold is kept whole."""
    b = topp(B=8, V=4096, dtype="f32", seed=11500)
    b.target[:] = np.round(b.target)
    b.draft[:] = np.round(b.draft)
    keep = S.draft_nucleus_mask(b.draft.astype(np.float64), b.cfg.temperature, b.cfg.top_p)
    rng = np.random.default_rng(3)
    for r in range(b.draft.shape[0]):
        for i in range(b.draft.shape[1]):
            b.draft_tokens[r, i] = rng.choice(np.flatnonzero(keep[r, i]))
    compare_spec(run_gpu(b), run_oracle(b))


def test_topp_one_is_spec_verify():
    b = topp(B=8, V=20000, seed=11600)
    g = run_gpu(b, top_p=1.0)
    out = guarded_call(sv.spec_verify, dev(b.target), dev(b.draft), dev(b.draft_tokens),
                       dev(b.uniforms), b.cfg.temperature, aux=True)
    for k, v in out.items():
        np.testing.assert_array_equal(g[k], v, err_msg=k)


def test_topp_statuses():
    b = topp(B=4, V=2048, seed=11700)
    b.target[0, 2, 9] = 0x7FC0                               # NaN
    xd = S.stored_to_f64(b.draft[1, 0])
    b.draft_tokens[1, 0] = int(np.argmin(xd))                # outside the draft row's nucleus
    g, o = run_gpu(b), run_oracle(b)
    compare_spec(g, o)
    assert g["row_status"].tolist()[:2] == [O.ROW_NONFINITE, O.ROW_BAD_TOKEN]


def test_topp_repeat_calls_are_deterministic():
    b = topp(B=16, seed=11800)
    a1, a2 = run_gpu(b), run_gpu(b)
    for k in a1:
        np.testing.assert_array_equal(a1[k], a2[k])


def with_rows(b, xt, xd, seed=5):
    """b with its logits replaced by xt / xd (stored in b's dtype) and each draft token redrawn
    from its draft row's nucleus."""
    if b.target.dtype == np.uint16:
        b.target[:] = S.f32_to_bf16_bits(xt.astype(np.float32))
        b.draft[:] = S.f32_to_bf16_bits(xd.astype(np.float32))
    else:
        b.target[:] = xt.astype(np.float32)
        b.draft[:] = xd.astype(np.float32)
    keep = S.draft_nucleus_mask(S.stored_to_f64(b.draft), b.cfg.temperature, b.cfg.top_p)
    rng = np.random.default_rng(seed)
    for r in range(b.draft.shape[0]):
        for i in range(b.draft.shape[1]):
            b.draft_tokens[r, i] = rng.choice(np.flatnonzero(keep[r, i]))
    return b


def _rows(rng, b, f):
    xt = f(rng, b.target.shape)
    return xt, f(rng, b.draft.shape)


def _negative(rng, shape):
    return -3.0 + 0.3 * rng.standard_normal(shape)


def _zero_max(rng, shape):
    x = -np.abs(2.0 * rng.standard_normal(shape))
    flat = x.reshape(-1, shape[-1])
    for row in flat:
        at = rng.choice(shape[-1], 10, replace=False)
        row[at[:5]] = 0.0
        row[at[5:]] = -0.0
    return x


def _flat(rng, shape):
    return 0.05 * rng.standard_normal(shape)


def _deep(rng, shape):
    # one token at 20 and the rest about 15 bits of mass below it: the kept mass crosses top_p far
    # below the cut, where no candidate is
    x = 9.6 + 0.05 * rng.standard_normal(shape)
    x.reshape(-1, shape[-1])[:, 0] = 20.0
    return x


def _cluster(rng, shape):
    # a tight cluster of 1000 distinct values holds nearly all the mass: the bin where it crosses
    # top_p is crowded
    x = -5.0 + rng.standard_normal(shape)
    flat = x.reshape(-1, shape[-1])
    for row in flat:
        at = rng.choice(shape[-1], 1000, replace=False)
        row[at] = 2.0 + 1e-6 * np.arange(1000)
    return x


@pytest.mark.parametrize("case, dtype, V, T", [
    ("negative", "bf16", 20000, 0.5),   # per-value bins over negative keys
    ("zero_max", "bf16", 4096, 1.0),    # +0 and -0 at the maximum; the keys span zero: the list path
    ("flat", "bf16", 40000, 1.0),       # every element a candidate: the list overflows
    ("deep", "bf16", 40000, 1.0),       # per-value bins, but the crossing lies below the cut
    ("deep", "f32", 20000, 1.0),        # the list, and the crossing below the cut
    ("flat", "f32", 20000, 1.0),        # fp32 list overflow
    ("cluster", "f32", 4096, 1.0),      # a crowded crossing bin
    ("zero_max", "f32", 4096, 1.0),     # fp32 list path with +0 and -0
])
def test_topp_select_paths(case, dtype, V, T):
    """Rows built to take each branch of the threshold select: per-value bins, the candidate list
    with its crossing bin resolved, and the radix select when the list overflows, the crossing lies
    below the cut or the crossing bin is crowded."""
    b = topp(B=4, gamma=3, V=V, dtype=dtype, temperature=T, seed=11900)
    f = {"negative": _negative, "zero_max": _zero_max, "flat": _flat, "deep": _deep,
         "cluster": _cluster}[case]
    xt, xd = _rows(np.random.default_rng(11901), b, f)
    b = with_rows(b, xt, xd)
    g, o = run_gpu(b), run_oracle(b)
    compare_spec(g, o, label=f"top-p {case} {dtype}")
    assert np.all(g["row_status"] == O.ROW_OK)
