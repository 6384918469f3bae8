"""GPU parity of the SMC-SD verify round (smc_verify) against the fp64 oracle.

Matching rule: statuses exact; tokens and ancestors exact except on particles whose extension or
ancestor uniform lies within 1e-6 of a boundary it was compared with (the oracle's margin); a
group's resampling decision exact except where its ESS lies within 1e-5 (relative) of eta; block
log-ratios and log weights within 1e-5 absolute; ESS within 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import BOUNDARY, TOL, dev, guarded_call

pytestmark = pytest.mark.gpu

C7 = S.SMC_CONFIGS["c7"]


def run_gpu(b, groups=None, eta=None, T=None):
    cfg = b.cfg
    return guarded_call(sv.smc_verify, dev(b.target), dev(b.draft), dev(b.draft_tokens),
                        dev(b.log_weights), dev(b.uniforms), groups or cfg.groups,
                        T or cfg.temperature, cfg.eta if eta is None else eta)


def run_oracle(b, groups=None, eta=None, T=None):
    cfg = b.cfg
    return O.smc_verify(b.target, b.draft, b.draft_tokens, b.log_weights.astype(np.float64),
                        b.uniforms, groups or cfg.groups, T or cfg.temperature,
                        cfg.eta if eta is None else eta)


def compare(g, o, Np):
    st = o["row_status"]
    np.testing.assert_array_equal(g["row_status"], st)
    flagged = o["margin"] < BOUNDARY
    gflag = o["ess_margin"] < TOL
    pflag = flagged | np.repeat(gflag, Np)
    ok = st == 0
    # tokens: drafts and extension
    same_tok = np.all(g["out_tokens"] == o["out_tokens"], 1)
    bad = ~same_tok & ~pflag
    assert not bad.any(), f"{bad.sum()} unflagged token mismatches, first {np.flatnonzero(bad)[0]}"
    np.testing.assert_array_equal(g["accepted_len"], np.where(ok, g["out_tokens"].shape[1] - 1, -1))
    # block log-ratios of OK particles
    d = np.abs(g["block_log_ratio"][ok].astype(np.float64) - o["log_ratio"][ok])
    assert d.size == 0 or d.max() <= TOL, f"block log-ratio diff {d.max():.3g}"
    assert np.all(np.isnan(g["block_log_ratio"][~ok]))
    # groups: ESS, decision, ancestors, weights
    gok = o["resampled"] >= 0
    np.testing.assert_array_equal(g["resampled"][~gok], -1)
    assert np.all(np.isnan(g["ess"][~gok]))
    e = np.abs(g["ess"][gok] / o["ess"][gok] - 1.0)
    assert e.size == 0 or e.max() <= TOL, f"ESS rel diff {e.max():.3g}"
    sure = gok & ~gflag
    np.testing.assert_array_equal(g["resampled"][sure], o["resampled"][sure])
    same_anc = g["ancestors"] == o["ancestors"]
    bad = ~same_anc & ~pflag
    assert not bad.any(), f"{bad.sum()} unflagged ancestor mismatches"
    lw_ok = np.repeat(sure, Np)
    d = np.abs(g["log_weights"][lw_ok].astype(np.float64) - o["logw_out"][lw_ok])
    assert d.size == 0 or d.max() <= TOL, f"log weight diff {d.max():.3g}"
    assert np.all(np.isnan(g["log_weights"][np.repeat(~gok, Np)]))
    return int(pflag.sum()), int((~same_tok | ~same_anc).sum())


def test_c7_full_size():
    b = S.make_smc_batch(C7)
    g, o = run_gpu(b), run_oracle(b)
    compare(g, o, C7.particles)
    assert np.all(o["row_status"] == 0)


@pytest.mark.parametrize("eta", [0.0, 1.5, 8.0])
def test_thresholds(eta):
    """Never, sometimes and always resampling."""
    b = S.make_smc_batch(S.scaled(C7, groups=16, particles=8, V=4000, temperature=1.5,
                                  draft_noise=0.3, seed=3100))
    g, o = run_gpu(b, eta=eta), run_oracle(b, eta=eta)
    compare(g, o, 8)
    if eta == 0.0:
        assert np.all(o["resampled"] == 0)
    if eta == 8.0:
        assert np.all(o["resampled"] == 1)


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (7, "bf16"), (1000, "bf16"), (32001, "f32"),
                                     (152064, "bf16")])
@pytest.mark.parametrize("K", [0, 1, 5, 20])
def test_shapes(V, dtype, K):
    b = S.make_smc_batch(S.scaled(C7, groups=3, particles=5, K=K, V=V, dtype=dtype,
                                  seed=3200 + V + K))
    compare(run_gpu(b), run_oracle(b), 5)


@pytest.mark.parametrize("particles", [1, 33, 300, 4096])
def test_particle_counts(particles):
    b = S.make_smc_batch(S.scaled(C7, groups=2, particles=particles, K=2, V=600, draft_noise=0.5,
                                  seed=3300 + particles))
    g, o = run_gpu(b, eta=particles / 2), run_oracle(b, eta=particles / 2)
    compare(g, o, particles)


def test_perfect_draft_anchor():
    b = S.make_smc_batch(S.scaled(C7, groups=4, particles=8, K=3, V=5000, seed=3400))
    b.draft = b.target[:, :3].copy()
    b.log_weights[:] = 0.0
    g = run_gpu(b)
    np.testing.assert_array_equal(g["block_log_ratio"], 0.0)
    np.testing.assert_allclose(g["ess"], 8.0, rtol=1e-6)
    np.testing.assert_array_equal(g["resampled"], 0)
    np.testing.assert_array_equal(g["ancestors"], np.tile(np.arange(8), 4))


def test_statuses_fail_their_group():
    b = S.make_smc_batch(S.scaled(C7, groups=4, particles=4, K=2, V=500, dtype="f32", seed=3500))
    b.target[1, 2, 7] = np.nan            # group 0
    b.draft_tokens[6, 1] = 500            # group 1: token out of range
    b.uniforms[9, 1] = 1.0                # group 2: a bad ancestor uniform
    b.draft[13, 0, b.draft_tokens[13, 0]] = -np.inf  # group 3: q(x) = 0
    g, o = run_gpu(b), run_oracle(b)
    compare(g, o, 4)
    assert list(o["row_status"][[1, 6, 9, 13]]) == [O.ROW_NONFINITE, O.ROW_BAD_TOKEN,
                                                     O.ROW_BAD_UNIFORM, O.ROW_BAD_TOKEN]
    np.testing.assert_array_equal(g["resampled"], -1)


def test_repeat_calls_are_deterministic():
    b = S.make_smc_batch(S.scaled(C7, groups=4, V=30000, seed=3600))
    a1, a2 = run_gpu(b), run_gpu(b)
    for k in a1:
        np.testing.assert_array_equal(a1[k], a2[k])


def test_many_groups_boundary_rate():
    """Mismatches only where flagged, and under 0.01% of particles."""
    b = S.make_smc_batch(S.scaled(C7, groups=2500, particles=8, K=2, V=48, temperature=1.0,
                                  draft_noise=0.5, seed=3700))
    g, o = run_gpu(b), run_oracle(b)
    flagged, mism = compare(g, o, 8)
    print(f"particles={b.cfg.B} flagged={flagged} mismatched={mism}")
    assert mism < 1e-4 * b.cfg.B
