"""GPU parity: the C-ABI CUDA path against the fp64 oracle on the same seeded inputs.

Full-size configurations run exactly as the benchmark launches them; the oracle checks every
request of c1, c2, c3, c4 and c5 (large batches go through the oracle on all host cores).  Every
GPU call goes through the guarded allocator of parity.py (sentinel bands around each output and
the workspace, and a bit-identical repeat call).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import (compare_spec, compare_tree, dev, guarded_call, run_gpu_spec, run_gpu_tree,
                    run_oracle_spec, run_oracle_tree)

pytestmark = pytest.mark.gpu


def check_spec(batch, top_k=None, sample=None, seed=0, label=None):
    g = run_gpu_spec(batch, top_k)
    if sample is None:
        o = run_oracle_spec(batch, top_k)
        return compare_spec(g, o, label=label)
    idx = np.sort(np.random.default_rng(seed).choice(batch.cfg.B, sample, replace=False))
    o = run_oracle_spec(batch, top_k, idx)
    return compare_spec(g, o, idx, label=label)


# ------------------------------------------------------------------ the five configurations

def test_c1_tiny_10000_trials():
    b = S.trial_batches(S.CONFIGS["c1"], 10000)
    n, flagged, mism = check_spec(b, label="c1 (10,000 trials)")
    assert mism < n * 1e-4


def test_c1_redrawn_logits():
    b = S.trial_batches(S.CONFIGS["c1"], 4000, redraw_logits=True)
    check_spec(b, label="c1 redrawn logits")


def test_c2_batched():
    check_spec(S.make_spec_batch(S.CONFIGS["c2"]), label="c2")


def test_c3_large_vocab():
    check_spec(S.make_spec_batch(S.CONFIGS["c3"]), label="c3")


def test_c4_topk_all_requests():
    """All 256 requests of c4 at full size (V=152064, top_k=50), as the benchmark launches it."""
    n, flagged, mism = check_spec(S.make_spec_batch(S.CONFIGS["c4"]), label="c4")
    assert n == 256


def test_c5_tree():
    tb = S.make_tree_batch(S.TREE_CONFIGS["c5"])
    compare_tree(run_gpu_tree(tb), run_oracle_tree(tb), label="c5")


def test_boundary_exceptions_large_vocab():
    """The boundary rule at the large vocabulary, where the draw's segment sums run longest:
    2,048 requests of c3's recipe (V=128256, T=0.7) over eight seeds, plus 512 requests of c4's
    top-k recipe.  Mismatches only on flagged requests, and under 0.01% of requests."""
    tot = fl = mm = 0
    for s in range(8):
        b = S.make_spec_batch(S.scaled(S.CONFIGS["c3"], B=256, seed=7100 + s))
        n, f, m = check_spec(b, label="c3 recipe, 2,048 requests")
        tot, fl, mm = tot + n, fl + f, mm + m
    for s in range(2):
        b = S.make_spec_batch(S.scaled(S.CONFIGS["c4"], seed=7200 + s))
        n, f, m = check_spec(b, label="c4 recipe, 512 requests")
        tot, fl, mm = tot + n, fl + f, mm + m
    print(f"requests={tot} near-boundary={fl} mismatched={mm}")
    assert tot >= 2560 and mm < 1e-4 * tot


# ------------------------------------------------------------------ shapes: tiles and ragged tails

@pytest.mark.parametrize("V", [1, 7, 8, 33, 1000, 4099, 40000, 40003])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_spec_shapes(V, dtype):
    cfg = S.scaled(S.CONFIGS["c2"], B=6, V=V, dtype=dtype, seed=2000 + V)
    check_spec(S.make_spec_batch(cfg))


@pytest.mark.parametrize("V,k", [(1000, 1), (1000, 50), (4099, 7), (40003, 50), (152064, 50),
                                 (20480, 256), (20481, 300), (64, 64), (300, 299)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_shapes(V, k, dtype):
    cfg = S.scaled(S.CONFIGS["c4"], B=5, V=V, top_k=k, dtype=dtype, seed=3000 + V + k)
    check_spec(S.make_spec_batch(cfg))


@pytest.mark.parametrize("B,V,k,dtype", [(40, 152064, 50, "bf16"), (40, 40000, 50, "f32"),
                                         (80, 40003, 50, "bf16"), (40, 40000, 256, "bf16"),
                                         (40, 16384, 7, "bf16"), (40, 20481, 300, "f32")])
def test_topk_many_rows(B, V, k, dtype):
    """More rows than the top-k streaming grid has CTAs (gamma=4: 9 rows per request), so every
    CTA streams several rows: aligned and unaligned rows, one-chunk rows, k above the CTA's
    threads (dense rows)."""
    cfg = S.scaled(S.CONFIGS["c4"], B=B, gamma=4, V=V, top_k=k, dtype=dtype, seed=3500 + V + k)
    check_spec(S.make_spec_batch(cfg))


def test_topk_many_rows_ties():
    cfg = S.scaled(S.CONFIGS["c4"], B=40, gamma=4, V=30000, top_k=50, seed=3600)
    check_spec(_coarse(cfg, 1.0))


@pytest.mark.parametrize("gamma", [0, 1, 2, 31, 32, 40])
def test_gamma_range(gamma):
    cfg = S.scaled(S.CONFIGS["c3"], B=3, gamma=gamma, V=5000, seed=4000 + gamma)
    check_spec(S.make_spec_batch(cfg))
    cfg = S.scaled(cfg, top_k=20)
    check_spec(S.make_spec_batch(cfg))


def test_many_requests_small_vocab():
    cfg = S.scaled(S.CONFIGS["c2"], B=3000, V=64, seed=77)
    n, flagged, _ = check_spec(S.make_spec_batch(cfg))


# ------------------------------------------------------------------ degenerate cases

def _coarse(cfg, scale=4.0):
    b = S.make_spec_batch(cfg)
    # quantise to a coarse grid so that many logits tie (bf16 keeps these values exactly)
    t = np.round(S.stored_to_f64(b.target) * scale) / scale
    d = np.round(S.stored_to_f64(b.draft) * scale) / scale
    b.target = S.f32_to_bf16_bits(t.astype(np.float32))
    b.draft = S.f32_to_bf16_bits(d.astype(np.float32))
    xd = S.stored_to_f64(b.draft)
    rng = np.random.default_rng(cfg.seed)
    for i in range(cfg.B):
        keep = S.draft_keep_mask(xd[i], cfg.top_k)
        b.draft_tokens[i] = S.gumbel_max_tokens(rng, xd[i] / cfg.temperature, keep)
    return b


@pytest.mark.parametrize("k", [1, 5, 50, 200])
def test_topk_ties_at_threshold(k):
    cfg = S.scaled(S.CONFIGS["c4"], B=6, V=30000, top_k=k, seed=5000 + k)
    check_spec(_coarse(cfg, 1.0))


def test_constant_rows_and_signed_zero():
    cfg = S.scaled(S.CONFIGS["c4"], B=4, V=3000, top_k=50, seed=5100)
    b = S.make_spec_batch(cfg)
    b.target[0] = S.f32_to_bf16_bits(np.full((cfg.gamma + 1, cfg.V), 1.5, np.float32))
    b.draft[0] = S.f32_to_bf16_bits(np.full((cfg.gamma, cfg.V), 1.5, np.float32))
    b.draft_tokens[0] = np.arange(cfg.gamma)
    z = np.zeros((cfg.gamma + 1, cfg.V), np.float32)
    z[:, ::2] = -0.0
    b.target[1] = S.f32_to_bf16_bits(z)
    b.draft[1] = S.f32_to_bf16_bits(z[:cfg.gamma])
    check_spec(b)
    check_spec(b, top_k=0)
    check_spec(b, top_k=cfg.V)


def test_self_draft_accepts_everything():
    cfg = S.scaled(S.CONFIGS["c3"], B=8, V=5000, seed=5200)
    b = S.make_spec_batch(cfg)
    b.draft = b.target[:, :cfg.gamma].copy()
    rng = np.random.default_rng(1)
    x = S.stored_to_f64(b.draft)
    for i in range(cfg.B):
        b.draft_tokens[i] = S.gumbel_max_tokens(rng, x[i] / cfg.temperature)
    g = run_gpu_spec(b)
    assert np.all(g["accepted_len"] == cfg.gamma)
    compare_spec(g, run_oracle_spec(b))


def test_topk_k_equals_V_matches_plain():
    cfg = S.scaled(S.CONFIGS["c2"], B=8, V=3000, seed=5300)
    b = S.make_spec_batch(cfg)
    a = run_gpu_spec(b, top_k=cfg.V)
    p = run_gpu_spec(b, top_k=0)
    for key in a:
        np.testing.assert_array_equal(a[key], p[key])


def test_status_codes():
    cfg = S.scaled(S.CONFIGS["c2"], B=8, V=512, seed=5400)
    b = S.make_spec_batch(cfg)
    nan = S.f32_to_bf16_bits(np.array([np.nan], np.float32))[0]
    pinf = S.f32_to_bf16_bits(np.array([np.inf], np.float32))[0]
    ninf = S.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0]
    b.target[0, 2, 17] = nan
    b.draft[1, 1, 3] = pinf
    b.target[2, cfg.gamma, :] = ninf
    b.draft_tokens[3, 2] = cfg.V
    b.draft[4, 0, b.draft_tokens[4, 0]] = ninf
    b.uniforms[5, cfg.gamma + 1] = 1.0
    b.uniforms[6, 0] = -0.25
    for k in (0, 10):
        g = run_gpu_spec(b, top_k=k)
        o = run_oracle_spec(b, top_k=k)
        if k == 0:
            np.testing.assert_array_equal(o["row_status"][:7], [1, 1, 1, 3, 3, 7, 7])
        compare_spec(g, o)
        assert np.all(g["out_tokens"][:7] == -1) and np.all(g["accepted_len"][:7] == -1)


def test_topk_token_outside_draft_topk():
    cfg = S.scaled(S.CONFIGS["c4"], B=4, V=2000, seed=5500)
    b = S.make_spec_batch(cfg)
    xd = S.stored_to_f64(b.draft)
    b.draft_tokens[1, 0] = int(np.argmin(xd[1, 0]))
    g = run_gpu_spec(b)
    o = run_oracle_spec(b)
    assert o["row_status"][1] == O.ROW_BAD_TOKEN
    compare_spec(g, o)


def test_empty_batch():
    import speculative_decoding_verification_spec_gb300 as sv
    z = torch.empty(0, 5, 100, dtype=torch.bfloat16, device="cuda")
    for k in (0, 10):
        out = guarded_call(sv.spec_verify, z,
                           torch.empty(0, 4, 100, dtype=torch.bfloat16, device="cuda"),
                           torch.empty(0, 4, dtype=torch.int32, device="cuda"),
                           torch.empty(0, 6, dtype=torch.float32, device="cuda"), 1.0, top_k=k,
                           aux=True)
        assert out["accepted_len"].size == 0


def test_unaligned_rows():
    """Row starts that are not 16-byte aligned use the scalar path."""
    cfg = S.scaled(S.CONFIGS["c2"], B=4, V=3000, seed=5600)
    b = S.make_spec_batch(cfg)
    import speculative_decoding_verification_spec_gb300 as sv
    # offset the tensors by one element inside a larger buffer
    t = torch.empty(b.target.size + 1, dtype=torch.int16, device="cuda")
    d = torch.empty(b.draft.size + 1, dtype=torch.int16, device="cuda")
    t[1:] = dev(b.target).view(-1)
    d[1:] = dev(b.draft).view(-1)
    g = guarded_call(sv.spec_verify, t[1:].view(b.target.shape), d[1:].view(b.draft.shape),
                     dev(b.draft_tokens), dev(b.uniforms), cfg.temperature, aux=True)
    compare_spec(g, run_oracle_spec(b), label="unaligned rows")


def test_repeat_calls_are_deterministic():
    b = S.make_spec_batch(S.scaled(S.CONFIGS["c3"], B=16, seed=5700))
    a1 = run_gpu_spec(b)
    a2 = run_gpu_spec(b)
    for key in a1:
        np.testing.assert_array_equal(a1[key], a2[key])


def test_boundary_exceptions_large_sample():
    """Mismatches are allowed only on draws within 1e-6 of a decision boundary, and must stay
    under 0.01% of requests: 60,000 requests with a long-tailed 512-token vocabulary."""
    cfg = S.scaled(S.CONFIGS["c2"], B=20000, V=512, seed=5800)
    tot = fl = mm = 0
    for s in range(3):
        n, f, m = check_spec(S.make_spec_batch(S.scaled(cfg, seed=5800 + s)),
                             label="V=512, 60,000 requests")
        tot += n
        fl += f
        mm += m
    print(f"requests={tot} near-boundary={fl} mismatched={mm}")
    assert mm < 1e-4 * tot


# ------------------------------------------------------------------ tree edge cases

def _tree(B, N, V, seed, dtype="bf16"):
    cfg = S.scaled(S.TREE_CONFIGS["c5"], B=B, V=V, max_nodes=N, dtype=dtype, seed=seed)
    return S.make_tree_batch(cfg)


@pytest.mark.parametrize("V", [5, 64, 1001, 128256, 128259])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tree_shapes(V, dtype):
    tb = _tree(4, 64, V, 6000 + V, dtype)
    compare_tree(run_gpu_tree(tb), O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens))


def test_tree_ties_and_statuses():
    tb = _tree(8, 20, 300, 6100)
    x = S.stored_to_f64(tb.logits)
    # ties at the maximum in every row of request 0 -> lowest index
    x[0] = np.round(x[0])
    x[0, :, 5] = x[0].max(axis=1)
    x[0, :, 9] = x[0].max(axis=1)
    tb.logits = S.f32_to_bf16_bits(x.astype(np.float32))
    # request 0: nodes follow the argmax
    am = np.argmax(S.stored_to_f64(tb.logits[0]), axis=1)
    pred = np.where(tb.parents[0] < 0, 0, tb.parents[0] + 1)
    tb.tokens[0] = am[pred]
    tb.logits[1, 3, 7] = S.f32_to_bf16_bits(np.array([np.nan], np.float32))[0]
    tb.parents[2, 5] = 5
    tb.tokens[3, 2] = 300
    tb.logits[4, 0, :] = S.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0]
    o = O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens)
    compare_tree(run_gpu_tree(tb), o)
    assert o["row_status"][:5].tolist() == [0, 1, 5, 3, 1]
    ov = O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens, max_out=2)
    compare_tree(run_gpu_tree(tb, max_out=2), ov)


def test_tree_chain_and_empty():
    tb = _tree(3, 1, 1000, 6200)
    compare_tree(run_gpu_tree(tb), O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens))
    # N = 0: only the frontier row; output is its argmax
    lg = tb.logits[:, :1].copy()
    par = np.zeros((3, 0), np.int32)
    tok = np.zeros((3, 0), np.int32)
    import speculative_decoding_verification_spec_gb300 as sv
    out = guarded_call(sv.tree_verify_greedy, dev(lg), dev(np.zeros((3, 1), np.int32))[:, :0],
                       dev(np.zeros((3, 1), np.int32))[:, :0])
    o = O.tree_verify_greedy(lg, par, tok)
    np.testing.assert_array_equal(out["out_tokens"], o["out_tokens"])
    np.testing.assert_array_equal(out["accepted_len"], o["accepted_len"])
