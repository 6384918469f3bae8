"""Python driver for the fp64 CPU oracle (``spec_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this module.  The CUDA product path never imports it, and it
imports nothing from the product package.

Every function here is argument marshalling around the C oracle; the arithmetic lives in
``spec_oracle.c`` and follows the pages cited there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
ROW_OK, ROW_NONFINITE, ROW_DEGENERATE, ROW_BAD_TOKEN = 0, 1, 2, 3
ROW_BAD_PARENT, ROW_OVERFLOW, ROW_BAD_UNIFORM, ROW_BAD_QROW = 5, 6, 7, 8

_lib = None


def build(force: bool = False) -> str:
    """Compile ``spec_oracle.c`` into ``liboracle.so`` next to it (plain gcc, -O2, fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def build_planted(replacements, workdir: str):
    """Compile a copy of ``spec_oracle.c`` with a mistake planted by text replacement.

    ``replacements`` is a list of (old, new) pairs; each ``old`` must occur exactly once.  The copy
    is built in ``workdir`` and returned bound like the real oracle, so that a test can show that a
    pin fails when the arithmetic is wrong.  The real oracle is untouched.
    """
    with open(_SRC) as f:
        src = f.read()
    for old, new in replacements:
        if src.count(old) != 1:
            raise ValueError(f"planted replacement target must occur once: {old!r}")
        src = src.replace(old, new)
    path_c = os.path.join(workdir, "planted_oracle.c")
    path_so = os.path.join(workdir, "libplanted_oracle.so")
    with open(path_c, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", path_so, path_c, "-lm"])
    return _bind(ctypes.CDLL(path_so))


def _bind(lib):
    P, I, D, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
    lib.oracle_spec_verify.argtypes = [P, P, I, P, P, I, I, I, D, I, P, P, P, P, P, P, P]
    lib.oracle_spec_verify.restype = I
    lib.oracle_tree_verify_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, P]
    lib.oracle_tree_verify_greedy.restype = I
    lib.oracle_tree_verify_sample.argtypes = [P, P, I, P, P, P, P, I, I, I, I, D, I,
                                              P, P, P, P, P, P, P, P]
    lib.oracle_tree_verify_sample.restype = I
    lib.oracle_smc_verify.argtypes = [P, P, I, P, P, P, I, I, I, I, D, I, D,
                                      P, P, P, P, P, P, P, P, P]
    lib.oracle_smc_verify.restype = I
    lib.oracle_tree_verify_typical.argtypes = [P, I, P, P, P, I, I, I, D, D, D, I,
                                               P, P, P, P, P, P, P]
    lib.oracle_tree_verify_typical.restype = I
    lib.oracle_ess.argtypes = [P, I]
    lib.oracle_ess.restype = D
    lib.oracle_spec_verify_masked.argtypes = [P, P, I, P, P, I, I, I, D, P, P, P, P, P, P, P, P]
    lib.oracle_spec_verify_masked.restype = I
    lib.oracle_spec_verify_topp.argtypes = [P, P, I, P, P, I, I, I, D, D, P, P, P, P, P, P, P, P]
    lib.oracle_spec_verify_topp.restype = I
    lib.oracle_row_probs_topp.argtypes = [P, I, Z, I, D, D, P, P, P, P]
    lib.oracle_row_probs_topp.restype = I
    lib.oracle_row_probs.argtypes = [P, I, Z, I, D, I, P, P, P]
    lib.oracle_row_probs.restype = I
    lib.oracle_row_probs_masked.argtypes = [P, I, Z, I, D, I, P, P, P, P]
    lib.oracle_row_probs_masked.restype = I
    lib.oracle_lse_online.argtypes = [P, I, I]
    lib.oracle_lse_online.restype = D
    lib.oracle_lse_maxshift.argtypes = [P, I]
    lib.oracle_lse_maxshift.restype = D
    lib.oracle_alpha.argtypes = [P, P, I]
    lib.oracle_alpha.restype = D
    lib.oracle_residual.argtypes = [P, P, I, P]
    lib.oracle_residual.restype = D
    lib.oracle_inverse_cdf.argtypes = [P, I, D, P, P]
    lib.oracle_inverse_cdf.restype = I
    lib.oracle_kth_largest.argtypes = [P, I, I]
    lib.oracle_kth_largest.restype = D
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a: np.ndarray):
    """Map a logits array to (contiguous array, oracle dtype code).  bf16 travels as uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype in (np.uint16, np.int16):
        return a.view(np.uint16), BF16
    raise TypeError(f"unsupported logits dtype {a.dtype}")


def mask_words(V: int) -> int:
    """32-bit words of one grammar-mask row over a vocabulary of V tokens."""
    return (V + 31) // 32


def spec_verify(target, draft, draft_tokens, uniforms, temperature: float, top_k: int = 0,
                allowed=None, top_p: float | None = None):
    """Exact speculative-sampling verify over B requests (fp64).

    target [B, gamma+1, V], draft [B, gamma, V] (float64, float32, or bf16 bits as uint16),
    draft_tokens [B, gamma] int32, uniforms [B, gamma+2] float32.  ``allowed`` (optional, no
    top-k with it) is the grammar mask [B, gamma+1, ceil(V/32)] uint32: bit v % 32 of word v // 32
    set when token v is valid at that position.  ``top_p`` (optional, alone) applies the top-p
    processor to every row.  Returns a dict with accepted_len, out_tokens, row_status, lse_p, lse_q,
    accept, margin and set_margin (top-p: the rows' kept-set margin alone; +inf otherwise).
    """
    lib = _load()
    t, dt = _logits(target)
    B, g1, V = t.shape
    gamma = g1 - 1
    if gamma > 0:
        d, dd = _logits(draft)
        assert dd == dt and d.shape == (B, gamma, V)
    else:
        d = np.zeros((B, 0, V), dtype=t.dtype)
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, gamma)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, gamma + 2)
    out = dict(
        accepted_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, gamma + 1), np.int32),
        row_status=np.empty(B, np.int32),
        lse_p=np.empty((B, gamma + 1)),
        lse_q=np.empty((B, gamma)),
        accept=np.empty((B, gamma)),
        margin=np.empty(B),
        set_margin=np.full(B, np.inf),
    )
    outs = (_ptr(out["accepted_len"]), _ptr(out["out_tokens"]), _ptr(out["row_status"]),
            _ptr(out["lse_p"]), _ptr(out["lse_q"]), _ptr(out["accept"]), _ptr(out["margin"]))
    if top_p is not None:
        if top_k or allowed is not None:
            raise ValueError("the top-p oracle takes no top-k or mask")
        rc = lib.oracle_spec_verify_topp(_ptr(t), _ptr(d), dt, _ptr(tok), _ptr(u), B, gamma, V,
                                         float(temperature), float(top_p), *outs,
                                         _ptr(out["set_margin"]))
    elif allowed is None:
        rc = lib.oracle_spec_verify(_ptr(t), _ptr(d), dt, _ptr(tok), _ptr(u), B, gamma, V,
                                    float(temperature), int(top_k), *outs)
    else:
        if top_k:
            raise ValueError("the masked oracle takes no top-k")
        m = np.ascontiguousarray(allowed, dtype=np.uint32).reshape(B, gamma + 1, mask_words(V))
        rc = lib.oracle_spec_verify_masked(_ptr(t), _ptr(d), dt, _ptr(tok), _ptr(u), B, gamma, V,
                                           float(temperature), _ptr(m), *outs)
    if rc != 0:
        raise ValueError("oracle_spec_verify rejected its arguments")
    return out


def tree_verify_greedy(logits, parents, tokens, max_out: int | None = None):
    """Greedy tree verify (fp64 / exact compares).  logits [B, N+1, V]; parents, tokens [B, N]."""
    lib = _load()
    lg, dt = _logits(logits)
    B, n1, V = lg.shape
    N = n1 - 1
    if max_out is None:
        max_out = N + 1
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    out = dict(
        accepted_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, max_out), np.int32),
        out_nodes=np.empty((B, max(max_out - 1, 0)), np.int32),
        row_status=np.empty(B, np.int32),
        amax=np.empty((B, N + 1), np.int32),
    )
    rc = lib.oracle_tree_verify_greedy(
        _ptr(lg), dt, _ptr(par), _ptr(tok), B, N, V, int(max_out),
        _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
        _ptr(out["out_nodes"]) if max_out > 1 else None, _ptr(out["row_status"]), _ptr(out["amax"]),
    )
    if rc != 0:
        raise ValueError("oracle_tree_verify_greedy rejected its arguments")
    return out


def spec_verify_greedy(target, draft_tokens):
    """Linear greedy verify: the greedy tree verify on the chain node i -> parent i - 1."""
    t = np.asarray(target)
    B, g1, _ = t.shape
    gamma = g1 - 1
    parents = np.tile(np.arange(-1, gamma - 1, dtype=np.int32), (B, 1))
    return tree_verify_greedy(t, parents, draft_tokens, max_out=gamma + 1)


def tree_verify_sample(target, draft, parents, tokens, qrow, uniforms, temperature: float,
                       max_out: int | None = None, lib=None):
    """Stochastic tree verify by the residual update over children (fp64).

    target [B, N+1, V], draft [B, Nq, V] (same dtype), parents / tokens / qrow [B, N] int32,
    uniforms [B, N+1] float32.  Returns a dict with accepted_len, out_tokens, out_nodes,
    row_status, accept (NaN where a node was not tested), margin, draw_lo, draw_hi.  ``lib`` selects
    a planted copy (``build_planted``) instead of the oracle.
    """
    lib = lib or _load()
    t, dt = _logits(target)
    B, n1, V = t.shape
    N = n1 - 1
    d, dd = _logits(draft)
    assert dd == dt and d.shape[0] == B and d.shape[2] == V
    Nq = d.shape[1]
    if max_out is None:
        max_out = N + 1
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    qr = np.ascontiguousarray(qrow, dtype=np.int32).reshape(B, N)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, N + 1)
    out = dict(
        accepted_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, max_out), np.int32),
        out_nodes=np.empty((B, max(max_out - 1, 0)), np.int32),
        row_status=np.empty(B, np.int32),
        accept=np.empty((B, N)),
        margin=np.empty(B),
        draw_lo=np.empty(B),
        draw_hi=np.empty(B),
    )
    rc = lib.oracle_tree_verify_sample(
        _ptr(t), _ptr(d), dt, _ptr(par), _ptr(tok), _ptr(qr), _ptr(u), B, N, Nq, V,
        float(temperature), int(max_out),
        _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
        _ptr(out["out_nodes"]) if max_out > 1 else None, _ptr(out["row_status"]),
        _ptr(out["accept"]), _ptr(out["margin"]), _ptr(out["draw_lo"]), _ptr(out["draw_hi"]),
    )
    if rc != 0:
        raise ValueError("oracle_tree_verify_sample rejected its arguments")
    return out


def smc_verify(target, draft, draft_tokens, logw_in, uniforms, groups: int, temperature: float,
               eta: float, top_k: int = 0):
    """One SMC-SD verify round over ``groups`` groups of particles (fp64).

    target [B, K+1, V], draft [B, K, V], draft_tokens [B, K], logw_in [B] (natural-log weights),
    uniforms [B, 2] (extension draw, ancestor draw); B = groups * particles.  Returns a dict with
    out_tokens, row_status, log_ratio, logw_out, ess, resampled, ancestors, margin, ess_margin.
    """
    lib = _load()
    t, dt = _logits(target)
    B, k1, V = t.shape
    K = k1 - 1
    if K > 0:
        d, dd = _logits(draft)
        assert dd == dt and d.shape == (B, K, V)
    else:
        d = np.zeros((B, 0, V), dtype=t.dtype)
    assert B % groups == 0
    Np = B // groups
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    lw = np.ascontiguousarray(logw_in, dtype=np.float64).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, 2)
    out = dict(
        out_tokens=np.empty((B, K + 1), np.int32),
        row_status=np.empty(B, np.int32),
        log_ratio=np.empty(B),
        logw_out=np.empty(B),
        ess=np.empty(groups),
        resampled=np.empty(groups, np.int32),
        ancestors=np.empty(B, np.int32),
        margin=np.empty(B),
        ess_margin=np.empty(groups),
    )
    rc = lib.oracle_smc_verify(
        _ptr(t), _ptr(d), dt, _ptr(tok), _ptr(lw), _ptr(u), groups, Np, K, V, float(temperature),
        int(top_k), float(eta), _ptr(out["out_tokens"]), _ptr(out["row_status"]),
        _ptr(out["log_ratio"]), _ptr(out["logw_out"]), _ptr(out["ess"]), _ptr(out["resampled"]),
        _ptr(out["ancestors"]), _ptr(out["margin"]), _ptr(out["ess_margin"]),
    )
    if rc != 0:
        raise ValueError("oracle_smc_verify rejected its arguments")
    return out


def ess(weights) -> float:
    """Effective sample size of positive weights (given as weights, not logs)."""
    lw = np.log(np.ascontiguousarray(weights, dtype=np.float64))
    return _load().oracle_ess(_ptr(lw), lw.shape[0])


def tree_verify_typical(logits, parents, tokens, uniforms, temperature: float, eps: float,
                        delta: float, max_out: int | None = None):
    """Tree verify with typical acceptance (fp64).  logits [B, N+1, V]; parents, tokens [B, N];
    uniforms [B].  Returns accepted_len, out_tokens, out_nodes, row_status, entropy [B, N+1],
    logp [B, N], margin [B]."""
    lib = _load()
    lg, dt = _logits(logits)
    B, n1, V = lg.shape
    N = n1 - 1
    if max_out is None:
        max_out = N + 1
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B)
    out = dict(
        accepted_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, max_out), np.int32),
        out_nodes=np.empty((B, max(max_out - 1, 0)), np.int32),
        row_status=np.empty(B, np.int32),
        entropy=np.empty((B, N + 1)),
        logp=np.empty((B, N)),
        margin=np.empty(B),
    )
    rc = lib.oracle_tree_verify_typical(
        _ptr(lg), dt, _ptr(par), _ptr(tok), _ptr(u), B, N, V, float(temperature), float(eps),
        float(delta), int(max_out), _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
        _ptr(out["out_nodes"]) if max_out > 1 else None, _ptr(out["row_status"]),
        _ptr(out["entropy"]), _ptr(out["logp"]), _ptr(out["margin"]))
    if rc != 0:
        raise ValueError("oracle_tree_verify_typical rejected its arguments")
    return out


def row_probs(logits_row, temperature: float, top_k: int = 0, allowed=None):
    """Processed probability row p = softmax(topk(mask(logits))/T).  ``allowed``: the row's
    grammar-mask words (ceil(V/32) uint32) or None.  Returns (status, p, lse, thr)."""
    lib = _load()
    x, dt = _logits(np.asarray(logits_row).reshape(-1))
    V = x.shape[0]
    p = np.zeros(V)
    lse = ctypes.c_double(0.0)
    thr = ctypes.c_double(0.0)
    if allowed is None:
        st = lib.oracle_row_probs(_ptr(x), dt, 0, V, float(temperature), int(top_k), _ptr(p),
                                  ctypes.byref(lse), ctypes.byref(thr))
    else:
        m = np.ascontiguousarray(allowed, dtype=np.uint32).reshape(mask_words(V))
        st = lib.oracle_row_probs_masked(_ptr(x), dt, 0, V, float(temperature), int(top_k), _ptr(m),
                                         _ptr(p), ctypes.byref(lse), ctypes.byref(thr))
    return st, p, lse.value, thr.value


def row_probs_topp(logits_row, temperature: float, top_p: float):
    """Processed probability row under temperature and top-p.  Returns (status, p, lse, thr,
    margin)."""
    lib = _load()
    x, dt = _logits(np.asarray(logits_row).reshape(-1))
    V = x.shape[0]
    p = np.zeros(V)
    lse, thr, mg = ctypes.c_double(0.0), ctypes.c_double(0.0), ctypes.c_double(0.0)
    st = lib.oracle_row_probs_topp(_ptr(x), dt, 0, V, float(temperature), float(top_p), _ptr(p),
                                   ctypes.byref(lse), ctypes.byref(thr), ctypes.byref(mg))
    return st, p, lse.value, thr.value, mg.value


def lse_online(z, block: int) -> float:
    z = np.ascontiguousarray(z, dtype=np.float64)
    return _load().oracle_lse_online(_ptr(z), z.shape[0], int(block))


def lse_maxshift(z) -> float:
    z = np.ascontiguousarray(z, dtype=np.float64)
    return _load().oracle_lse_maxshift(_ptr(z), z.shape[0])


def alpha(p, q) -> float:
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    return _load().oracle_alpha(_ptr(p), _ptr(q), p.shape[0])


def residual(p, q):
    """Returns (normalised residual, Z)."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.empty_like(p)
    Z = _load().oracle_residual(_ptr(p), _ptr(q), p.shape[0], _ptr(out))
    return out, Z


def inverse_cdf(r, u: float):
    """Returns (token, C(v-1)/Z, C(v)/Z); token -1 when the mass is not positive."""
    r = np.ascontiguousarray(r, dtype=np.float64)
    lo = ctypes.c_double(0.0)
    hi = ctypes.c_double(0.0)
    v = _load().oracle_inverse_cdf(_ptr(r), r.shape[0], float(u), ctypes.byref(lo), ctypes.byref(hi))
    return v, lo.value, hi.value


def kth_largest(x, k: int) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return _load().oracle_kth_largest(_ptr(x), x.shape[0], int(k))
