"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the C-ABI path,
run the oracle on the same bits, and compare by the matching rules:

  * row status, accepted lengths and emitted tokens bit-exact, except on requests whose draw lies
    within 1e-6 of a decision boundary (the oracle's margin); such exceptions are counted and
    must stay under 0.01% of requests;
  * normalisers (lse) and accept ratios within 1e-5 absolute;
  * tree verify bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O

BOUNDARY = 1e-6
TOL = 1e-5


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def run_gpu_spec(batch, top_k=None, aux=True, workspace=None):
    cfg = batch.cfg
    k = cfg.top_k if top_k is None else top_k
    out = sv.spec_verify(dev(batch.target), dev(batch.draft), dev(batch.draft_tokens),
                         dev(batch.uniforms), cfg.temperature, top_k=k, aux=aux,
                         workspace=workspace)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def run_oracle_spec(batch, top_k=None, idx=None):
    cfg = batch.cfg
    k = cfg.top_k if top_k is None else top_k
    sl = slice(None) if idx is None else idx
    return O.spec_verify(batch.target[sl], batch.draft[sl], batch.draft_tokens[sl],
                         batch.uniforms[sl], cfg.temperature, k)


def compare_spec(g, o, idx=None, check_aux=True):
    """Returns (n_rows, n_flagged, n_mismatch).  Raises AssertionError on a violation."""
    if idx is not None:
        g = {k: v[idx] for k, v in g.items()}
    st_o = o["row_status"]
    np.testing.assert_array_equal(g["row_status"], st_o, err_msg="row status differs")
    flagged = o["margin"] < BOUNDARY
    same = (g["accepted_len"] == o["accepted_len"]) & np.all(g["out_tokens"] == o["out_tokens"], 1)
    bad = ~same & ~flagged
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(
            f"{bad.sum()} unflagged mismatches; first request {i}: gpu A={g['accepted_len'][i]} "
            f"tokens={g['out_tokens'][i].tolist()} oracle A={o['accepted_len'][i]} "
            f"tokens={o['out_tokens'][i].tolist()} margin={o['margin'][i]:.3g}")
    if check_aux and "lse_p" in g:
        # a flagged request may have decided a kept set (top-p) the other way: its normalisers are
        # then those of a different, equally valid set
        ok = (st_o == 0) & ~flagged
        for key in ("lse_p", "lse_q", "accept"):
            if g[key].size == 0 or not ok.any():
                continue
            d = np.abs(g[key][ok].astype(np.float64) - o[key][ok])
            assert np.all(d <= TOL), f"{key}: max abs diff {d.max():.3g}"
    return len(st_o), int(flagged.sum()), int((~same).sum())


def run_gpu_tree(tb, max_out=None, workspace=None):
    out = sv.tree_verify_greedy(dev(tb.logits), dev(tb.parents), dev(tb.tokens),
                                max_out=max_out, workspace=workspace)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def compare_tree(g, o):
    for key in ("row_status", "accepted_len", "out_tokens"):
        np.testing.assert_array_equal(g[key], o[key], err_msg=key)
    if o["out_nodes"].shape[1] > 0:
        np.testing.assert_array_equal(g["out_nodes"][:, :o["out_nodes"].shape[1]], o["out_nodes"])
