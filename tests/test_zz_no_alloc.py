"""The entry point that allocates nothing (spec_verify_noalloc) against spec_verify.

spec_verify_noalloc serves callers that cannot call cudaMalloc (pre-placed buffers only, an
allocator that forbids new device allocations, a fixed memory footprint after start-up): its
scratch is a fixed per-GPU array inside the library instead of a caller-provided workspace.  It
runs the same kernels, so on the same inputs it must give what spec_verify gives -- on
consecutive calls too, since every call reuses the array the previous call left behind.

This file is collected last on purpose: a run that stops at the first failure has then run every
other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_spec_gb300 as sv
from speculative_decoding_verification_spec_gb300 import binding
from speculative_decoding_verification_spec_gb300 import synth as S

from parity import Guarded

pytestmark = pytest.mark.gpu

TOL = 1e-5  # absolute, on normalisers and accept ratios (the parity tests' bound)


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _inputs(batch):
    return (_dev(batch.target), _dev(batch.draft), _dev(batch.draft_tokens),
            _dev(batch.uniforms), batch.cfg.temperature)


def _host(out):
    return {k: v.cpu().numpy() for k, v in out.items()}


def _noalloc(x):
    """One spec_verify_noalloc call with every output inside sentinel guard bands (checked after
    the call: nothing outside the caller's buffers may be written)."""
    B, g1, _ = x[0].shape
    g = Guarded()
    out = dict(accepted_len=g.empty((B,), torch.int32, "accepted_len"),
               out_tokens=g.empty((B, g1), torch.int32, "out_tokens"),
               row_status=g.empty((B,), torch.int32, "row_status"),
               lse_p=g.empty((B, g1), torch.float32, "lse_p"),
               lse_q=g.empty((B, g1 - 1), torch.float32, "lse_q"),
               accept=g.empty((B, g1 - 1), torch.float32, "accept"))
    sv.spec_verify_noalloc(*x, out=out)
    torch.cuda.synchronize()
    g.check()
    return _host(out)


def _same(got, want):
    for key in ("row_status", "accepted_len", "out_tokens"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    for key in ("lse_p", "lse_q", "accept"):
        a, b = got[key].astype(np.float64), want[key].astype(np.float64)
        np.testing.assert_array_equal(np.isnan(a), np.isnan(b), err_msg=key)
        ok = ~np.isnan(b)
        assert np.all(np.abs(a[ok] - b[ok]) <= TOL), key


def test_noalloc_matches_spec_verify_on_two_calls_in_a_row():
    sv.load()
    # two different shapes, so the second call runs over what the first left in the array
    b1 = S.make_spec_batch(S.CONFIGS["c3"])                      # B=64, gamma=5, V=128256, bf16
    b2 = S.make_spec_batch(S.scaled(S.CONFIGS["c1"], B=48, V=1000))  # fp32, ragged V
    for b in (b1, b2):
        assert sv.workspace_bytes(b.cfg.B, b.cfg.gamma, b.cfg.V) <= sv.NOALLOC_SCRATCH_BYTES
    x1, x2 = _inputs(b1), _inputs(b2)
    g1 = _noalloc(x1)
    g2 = _noalloc(x2)
    w1 = _host(sv.spec_verify(*x1, aux=True))
    w2 = _host(sv.spec_verify(*x2, aux=True))
    _same(g1, w1)
    _same(g2, w2)
    # and once more on the first inputs, after the second shape used the array
    _same(_noalloc(x1), w1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = sv.load()
    B, gamma, V = 1024, 7, 152064
    assert sv.workspace_bytes(B, gamma, V) > sv.NOALLOC_SCRATCH_BYTES
    # small real buffers: the call must refuse before it reads or writes any of them
    dummy = torch.zeros(64, dtype=torch.int16, device="cuda")
    acc = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    d = P(dummy.data_ptr())
    rc = lib.spec_verify_noalloc(d, d, binding.SPEC_BF16, d, d, B, gamma, V, 1.0, P(acc.data_ptr()),
                                 P(acc.data_ptr()), None, None, None, None, None)
    assert rc == binding.SPEC_ERR_TOO_LARGE
    assert b"no-allocation" in lib.spec_status_string(rc)
    torch.cuda.synchronize()
    assert acc.cpu().tolist() == [7, 7, 7, 7]
