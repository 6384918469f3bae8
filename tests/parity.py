"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the C-ABI path,
run the oracle on the same bits, and compare by the matching rules:

  * row status, accepted lengths and emitted tokens bit-exact, except on requests whose draw lies
    within 1e-6 of a decision boundary (the oracle's margin); such exceptions are counted and
    must stay under 0.01% of requests;
  * normalisers (lse) and accept ratios within 1e-5 absolute on every request whose status is OK.
    They do not depend on the uniforms, so a request flagged by a draw still compares them; the
    one exemption is top-p, whose kept set (and so its normalisers) may legitimately differ when a
    row's kept mass lies within 1e-6 of top_p (the oracle's set_margin);
  * tree verify bit-exact.

Every GPU call made through ``guarded_call`` places each output and the workspace between two
guard bands of a sentinel byte, checks after the call that no band was written (the substitute
for a memory checker: an out-of-range write by any kernel shows up here), and checks that the
call's results are bit-identical to an ordinary call's on the same inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_verification_spec_gb300 as sv
from oracle import oracle as O
from oracle import pool as OP

BOUNDARY = 1e-6
TOL = 1e-5
SENTINEL = 0xA5   # guard-band byte
BAND = 4096       # guard bytes on each side of every guarded buffer

# (label) -> [requests, flagged, mismatched]; printed at the end of the run by conftest.py
COUNTS: dict[str, list[int]] = {}


def record(label: str, n: int, flagged: int, mismatched: int) -> None:
    c = COUNTS.setdefault(label, [0, 0, 0])
    c[0] += n
    c[1] += flagged
    c[2] += mismatched


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


# ------------------------------------------------------------------ guard bands

class Guarded:
    """Device buffers, each placed between two BAND-byte bands of SENTINEL bytes.  The buffer
    itself starts filled with SENTINEL too, so an output element a kernel never writes also shows
    up (as a value the oracle does not produce)."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype, name):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((BAND + n + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n, name))
        return raw[BAND:BAND + n].view(dtype).view(shape)

    def check(self):
        for raw, n, name in self.bufs:
            for side, band in (("before", raw[:BAND]), ("after", raw[BAND + n:])):
                bad = torch.nonzero(band != SENTINEL)
                if bad.numel():
                    i = int(bad[0, 0])
                    raise AssertionError(
                        f"{name}: guard band {side} the buffer was written ({bad.shape[0]} bytes, "
                        f"first at offset {i - BAND if side == 'before' else n + i} of {n})")


class GuardedWorkspace:
    """A workspace (the binding's ``Workspace`` interface) of exactly the size the call asks
    for, with guard bands on both sides; the band after it starts right after
    spec_workspace_bytes(...)."""

    def __init__(self, guard: Guarded):
        self.guard = guard
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        n = max(int(nbytes), 16)
        if self.buf is None or self.buf.numel() != n:
            self.buf = self.guard.empty((n,), torch.uint8, f"workspace[{nbytes} bytes]")
        return self.buf


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32) if t.element_size() == 4 else t


def guarded_call(fn, *args, guard_ws: bool = True, **kw):
    """Call binding function ``fn`` twice: once as a user would (the library's outputs and the
    default workspace), then with every output and the workspace inside guard bands.  Checks the
    bands and that both calls agree bit for bit; returns the guarded call's outputs on the host."""
    ref = fn(*args, **kw)
    g = Guarded()
    out = {k: g.empty(tuple(v.shape), v.dtype, k) for k, v in ref.items()}
    kw2 = dict(kw, out=out)
    if guard_ws and "workspace" not in kw:
        kw2["workspace"] = GuardedWorkspace(g)
    res = fn(*args, **kw2)
    torch.cuda.synchronize()
    g.check()
    for k in ref:
        if not torch.equal(_bits(ref[k]), _bits(res[k])):
            raise AssertionError(f"{k}: a repeat call on the same inputs differs")
    return {k: v.cpu().numpy() for k, v in res.items()}


# ------------------------------------------------------------------ spec_verify family

def run_gpu_spec(batch, top_k=None, aux=True, workspace=None):
    cfg = batch.cfg
    k = cfg.top_k if top_k is None else top_k
    kw = dict(top_k=k, aux=aux)
    if workspace is not None:
        kw["workspace"] = workspace
    return guarded_call(sv.spec_verify, dev(batch.target), dev(batch.draft),
                        dev(batch.draft_tokens), dev(batch.uniforms), cfg.temperature, **kw)


def run_oracle_spec(batch, top_k=None, idx=None, procs=None):
    """The oracle on all requests (or those in idx), over the host cores for large batches."""
    cfg = batch.cfg
    k = cfg.top_k if top_k is None else top_k
    sl = slice(None) if idx is None else idx
    t, d = batch.target[sl], batch.draft[sl]
    if procs is None and t.size * t.itemsize > (64 << 20):
        return OP.spec_verify(t, d, batch.draft_tokens[sl], batch.uniforms[sl], cfg.temperature, k)
    if procs and procs > 1:
        return OP.spec_verify(t, d, batch.draft_tokens[sl], batch.uniforms[sl], cfg.temperature, k,
                              procs=procs)
    return O.spec_verify(t, d, batch.draft_tokens[sl], batch.uniforms[sl], cfg.temperature, k)


def compare_spec(g, o, idx=None, check_aux=True, label=None):
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
        # only a top-p kept-set decision within 1e-6 of top_p exempts a request: the normalisers
        # and accept ratios are then those of a different, equally valid kept set
        set_flag = o.get("set_margin", np.full(len(st_o), np.inf)) < BOUNDARY
        ok = (st_o == 0) & ~set_flag
        for key in ("lse_p", "lse_q", "accept"):
            if g[key].size == 0 or not ok.any():
                continue
            d = np.abs(g[key][ok].astype(np.float64) - o[key][ok])
            assert np.all(d <= TOL), f"{key}: max abs diff {d.max():.3g}"
    n, f, m = len(st_o), int(flagged.sum()), int((~same).sum())
    if label:
        record(label, n, f, m)
    return n, f, m


# ------------------------------------------------------------------ greedy tree

def run_gpu_tree(tb, max_out=None, workspace=None):
    kw = dict(max_out=max_out)
    if workspace is not None:
        kw["workspace"] = workspace
    return guarded_call(sv.tree_verify_greedy, dev(tb.logits), dev(tb.parents), dev(tb.tokens), **kw)


def run_oracle_tree(tb, max_out=None):
    if tb.logits.size * tb.logits.itemsize > (64 << 20):
        return OP.tree_verify_greedy(tb.logits, tb.parents, tb.tokens, max_out=max_out)
    return O.tree_verify_greedy(tb.logits, tb.parents, tb.tokens, max_out=max_out)


def compare_tree(g, o, label=None):
    for key in ("row_status", "accepted_len", "out_tokens"):
        np.testing.assert_array_equal(g[key], o[key], err_msg=key)
    if o["out_nodes"].shape[1] > 0:
        np.testing.assert_array_equal(g["out_nodes"][:, :o["out_nodes"].shape[1]], o["out_nodes"])
    if label:
        record(label, len(o["row_status"]), 0, 0)
