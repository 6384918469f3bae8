"""Thin ctypes binding over the C ABI in ``include/spec_verify.h``.

Argument marshalling only: every step of the verify path runs in the CUDA kernels of
``libspecverify.so``.  PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the library is missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build_ext

SPEC_F32, SPEC_BF16 = 0, 1
ROW_OK, ROW_NONFINITE, ROW_DEGENERATE, ROW_BAD_TOKEN, ROW_TIMEOUT = 0, 1, 2, 3, 4
ROW_BAD_PARENT, ROW_OVERFLOW, ROW_BAD_UNIFORM, ROW_BAD_QROW = 5, 6, 7, 8

# every symbol the header declares
EXPORTS = ("spec_workspace_bytes", "spec_verify", "spec_verify_topk", "spec_verify_topp",
           "spec_verify_masked",
           "tree_verify_greedy", "spec_verify_greedy",
           "tree_verify_sample", "tree_verify_typical", "smc_verify", "spec_verify_noalloc", "spec_set_kernel_events", "spec_set_wait_limit",
           "spec_set_tree_sample_cluster", "spec_status_string")

# fixed scratch of spec_verify_noalloc (SPEC_NOALLOC_SCRATCH_BYTES in the header)
NOALLOC_SCRATCH_BYTES = 8 << 20
SPEC_ERR_TOO_LARGE = 4

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def load(path: str | None = None):
    """Load the compiled library (building it first if the sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or build_ext.LIB
    if not os.path.exists(path):
        raise SpecVerifyError(
            f"CUDA extension {path} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.spec_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.spec_workspace_bytes.restype = Z
    lib.spec_verify.argtypes = [P, P, I, P, P, I, I, I, F, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify.restype = I
    lib.spec_verify_topk.argtypes = [P, P, I, P, P, I, I, I, F, I, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_topk.restype = I
    lib.spec_verify_topp.argtypes = [P, P, I, P, P, I, I, I, F, F, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_topp.restype = I
    lib.spec_verify_masked.argtypes = [P, P, I, P, P, P, I, I, I, F, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_masked.restype = I
    lib.tree_verify_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, P, Z, P]
    lib.tree_verify_greedy.restype = I
    lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, P, Z, P]
    lib.spec_verify_greedy.restype = I
    lib.tree_verify_sample.argtypes = [P, P, I, P, P, P, P, I, I, I, I, F, I, P, P, P, P, P, P]
    lib.tree_verify_sample.restype = I
    lib.tree_verify_typical.argtypes = [P, I, P, P, P, I, I, I, F, F, F, I, P, P, P, P, P, P, P, Z, P]
    lib.tree_verify_typical.restype = I
    lib.smc_verify.argtypes = [P, P, I, P, P, P, I, I, I, I, F, F, P, P, P, P, P, P, P, P, P, Z, P]
    lib.smc_verify.restype = I
    lib.spec_verify_noalloc.argtypes = [P, P, I, P, P, I, I, I, F, P, P, P, P, P, P, P]
    lib.spec_verify_noalloc.restype = I
    lib.spec_set_kernel_events.argtypes = [P, P]
    lib.spec_set_kernel_events.restype = None
    lib.spec_set_wait_limit.argtypes = [I]
    lib.spec_set_wait_limit.restype = I
    lib.spec_set_tree_sample_cluster.argtypes = [I]
    lib.spec_set_tree_sample_cluster.restype = I
    lib.spec_status_string.argtypes = [I]
    lib.spec_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        raise SpecVerifyError(load().spec_status_string(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype in (torch.bfloat16, torch.int16):  # int16 = raw bf16 bit patterns
        return SPEC_BF16
    raise TypeError(f"logits must be bfloat16 (or its int16 bits) or float32, got {t.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise SpecVerifyError("verify inputs must be CUDA tensors (there is no CPU path)")


class Workspace:
    """Device scratch for the verify calls, grown on demand (plain torch allocation)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace(ws, device):
    if ws is not None:
        return ws
    key = str(device)
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


def set_kernel_events(start=None, stop=None):
    """Time the dominant kernel of later calls: torch.cuda.Event pair (recorded around it on the
    call's stream), or None to stop."""
    if start is None or stop is None:
        load().spec_set_kernel_events(None, None)
        return
    for e in (start, stop):
        if not e.cuda_event:
            e.record()  # creates the underlying CUDA event
    load().spec_set_kernel_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))


def set_wait_limit(polls: int) -> int:
    """Test aid: polls after which a bounded wait of the streaming kernels gives up (0: at once,
    so every request of a streaming call reports ROW_TIMEOUT; negative: the default).  Returns
    the previous limit."""
    return int(load().spec_set_wait_limit(int(polls)))


def set_tree_sample_cluster(cl: int) -> int:
    """Measurement aid: force tree_verify_sample's cluster size (1, 2, 4, 8 or 16 CTAs per request;
    anything else: the automatic choice).  Returns the previous setting (0: automatic)."""
    return int(load().spec_set_tree_sample_cluster(int(cl)))


def workspace_bytes(B, gamma, V, top_k=0, tree_nodes=0) -> int:
    return int(load().spec_workspace_bytes(B, gamma, V, top_k, tree_nodes))


def spec_verify(target, draft, draft_tokens, uniforms, temperature: float, *, top_k: int = 0,
                allowed=None, top_p: float | None = None, aux: bool = False, out=None,
                workspace: Workspace | None = None, stream=None):
    """Exact speculative-sampling verify on the GPU.

    target [B, gamma+1, V], draft [B, gamma, V] (bf16 / int16 bf16 bits / fp32, CUDA),
    draft_tokens [B, gamma] int32, uniforms [B, gamma+2] fp32.  ``top_k`` > 0 applies the top-k
    processor (spec_verify_topk).  ``allowed`` (CUDA int32/uint32 [B, gamma+1, ceil(V/32)]) is a
    grammar mask (spec_verify_masked; not with top_k); ``top_p`` applies the top-p processor
    (spec_verify_topp; alone).  Returns a dict of CUDA tensors:
    accepted_len, out_tokens, row_status (and lse_p, lse_q, accept when ``aux``).
    """
    lib = load()
    _need_cuda(target, draft, draft_tokens, uniforms)
    B, g1, V = target.shape
    gamma = g1 - 1
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, gamma + 1, dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
        if aux:
            out["lse_p"] = torch.empty(B, gamma + 1, dtype=torch.float32, device=dev)
            out["lse_q"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
            out["accept"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
    nbytes = workspace_bytes(B, gamma, V, top_k)
    ws = _workspace(workspace, dev).get(nbytes)
    common = [_ptr(target), _ptr(draft), _dtype_code(target), _ptr(draft_tokens), _ptr(uniforms),
              B, gamma, V, float(temperature)]
    tail = [_ptr(out["accepted_len"]), _ptr(out["out_tokens"]), _ptr(out.get("row_status")),
            _ptr(out.get("lse_p")), _ptr(out.get("lse_q")), _ptr(out.get("accept")),
            _ptr(ws), ws.numel(), _stream(stream)]
    if top_p is not None:
        if top_k or allowed is not None:
            raise ValueError("spec_verify_topp takes no top_k or mask")
        rc = lib.spec_verify_topp(*common, float(top_p), *tail)
    elif allowed is not None:
        if top_k:
            raise ValueError("spec_verify_masked takes no top_k")
        _need_cuda(allowed)
        W = (V + 31) // 32
        if tuple(allowed.shape) != (B, gamma + 1, W) or allowed.element_size() != 4 \
                or not allowed.is_contiguous():
            raise ValueError(f"allowed must be a contiguous 32-bit [B, gamma+1, {W}] tensor")
        rc = lib.spec_verify_masked(*common[:5], _ptr(allowed), *common[5:], *tail)
    elif top_k:
        rc = lib.spec_verify_topk(*common, int(top_k), *tail)
    else:
        rc = lib.spec_verify(*common, *tail)
    _check(rc)
    return out


def spec_verify_topp(target, draft, draft_tokens, uniforms, temperature: float, top_p: float, **kw):
    """spec_verify with the top-p (nucleus) processor on every row."""
    return spec_verify(target, draft, draft_tokens, uniforms, temperature, top_p=top_p, **kw)


def spec_verify_masked(target, draft, draft_tokens, uniforms, allowed, temperature: float, **kw):
    """spec_verify under a grammar mask ``allowed`` [B, gamma+1, ceil(V/32)] (32-bit words)."""
    return spec_verify(target, draft, draft_tokens, uniforms, temperature, allowed=allowed, **kw)


def spec_verify_noalloc(target, draft, draft_tokens, uniforms, temperature: float, *,
                        aux: bool = False, out=None, stream=None):
    """spec_verify through the entry point that allocates no device scratch.

    For callers that cannot allocate device memory: the library keeps the scratch in a fixed
    per-GPU array of NOALLOC_SCRATCH_BYTES, shared by every call on that GPU, so calls must not
    overlap on the GPU.  Pass ``out`` (preallocated CUDA tensors, same keys as spec_verify's
    result) to keep this wrapper itself from allocating.  Sizes that need more scratch than the
    array holds raise SpecVerifyError.
    """
    lib = load()
    _need_cuda(target, draft, draft_tokens, uniforms)
    B, g1, V = target.shape
    gamma = g1 - 1
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, gamma + 1, dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
        if aux:
            out["lse_p"] = torch.empty(B, gamma + 1, dtype=torch.float32, device=dev)
            out["lse_q"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
            out["accept"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
    rc = lib.spec_verify_noalloc(
        _ptr(target), _ptr(draft), _dtype_code(target), _ptr(draft_tokens), _ptr(uniforms),
        B, gamma, V, float(temperature), _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
        _ptr(out.get("row_status")), _ptr(out.get("lse_p")), _ptr(out.get("lse_q")),
        _ptr(out.get("accept")), _stream(stream))
    _check(rc)
    return out


def spec_verify_topk(target, draft, draft_tokens, uniforms, temperature: float, top_k: int, **kw):
    if top_k < 1:
        raise ValueError("top_k must be >= 1")
    return spec_verify(target, draft, draft_tokens, uniforms, temperature, top_k=top_k, **kw)


def tree_verify_greedy(logits, parents, tokens, *, max_out: int | None = None, out=None,
                       workspace: Workspace | None = None, stream=None):
    """Greedy tree verify on the GPU.  logits [B, N+1, V]; parents, tokens [B, N] int32."""
    lib = load()
    _need_cuda(logits, parents, tokens)
    B, n1, V = logits.shape
    N = n1 - 1
    max_out = N + 1 if max_out is None else int(max_out)
    dev = logits.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, max_out, dtype=torch.int32, device=dev),
            out_nodes=torch.empty(B, max(max_out - 1, 0), dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
    nbytes = workspace_bytes(B, 0, V, 0, max(N, 1))
    ws = _workspace(workspace, dev).get(nbytes)
    rc = lib.tree_verify_greedy(_ptr(logits), _dtype_code(logits), _ptr(parents), _ptr(tokens),
                                B, N, V, max_out, _ptr(out["accepted_len"]),
                                _ptr(out["out_tokens"]), _ptr(out.get("out_nodes")),
                                _ptr(out.get("row_status")), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc)
    return out


def tree_verify_typical(logits, parents, tokens, uniforms, temperature: float, epsilon: float,
                        delta: float, *, max_out: int | None = None, aux: bool = False, out=None,
                        workspace: Workspace | None = None, stream=None):
    """Tree verify with typical acceptance on the GPU.  logits [B, N+1, V] (bf16 / int16 bf16
    bits / fp32, CUDA), parents and tokens [B, N] int32, uniforms [B] fp32.  Returns a dict of CUDA
    tensors: accepted_len, out_tokens [B, max_out], out_nodes, row_status (and entropy [B, N+1],
    logp [B, N] when ``aux``)."""
    lib = load()
    _need_cuda(logits, parents, tokens, uniforms)
    B, R, V = logits.shape
    N = R - 1
    mo = N + 1 if max_out is None else int(max_out)
    dev = logits.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, mo, dtype=torch.int32, device=dev),
            out_nodes=torch.empty(B, max(mo - 1, 0), dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
        if aux:
            out["entropy"] = torch.empty(B, R, dtype=torch.float32, device=dev)
            out["logp"] = torch.empty(B, N, dtype=torch.float32, device=dev)
    nbytes = workspace_bytes(B, 0, V, 0, max(N, 1))
    ws = _workspace(workspace, dev).get(nbytes)
    rc = lib.tree_verify_typical(
        _ptr(logits), _dtype_code(logits), _ptr(parents), _ptr(tokens), _ptr(uniforms), B, N, V,
        float(temperature), float(epsilon), float(delta), mo, _ptr(out["accepted_len"]),
        _ptr(out["out_tokens"]), _ptr(out.get("out_nodes")), _ptr(out.get("row_status")),
        _ptr(out.get("entropy")), _ptr(out.get("logp")), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc)
    return out


def tree_verify_sample(target, draft, parents, tokens, qrow, uniforms, temperature: float, *,
                       max_out: int | None = None, aux: bool = False, out=None, stream=None):
    """Stochastic tree verify on the GPU (residual update over each node's children).

    target [B, N+1, V], draft [B, Nq, V] (same dtype), parents / tokens / qrow [B, N] int32,
    uniforms [B, N+1] float32; all CUDA tensors.  Returns accepted_len, out_tokens, out_nodes,
    row_status and, with ``aux``, accept [B, N] (NaN where a node was not tested).
    """
    lib = load()
    _need_cuda(target, draft, parents, tokens, qrow, uniforms)
    B, n1, V = target.shape
    N = n1 - 1
    Nq = draft.shape[1] if draft is not None and draft.dim() == 3 else 0
    if draft is not None and N > 0 and (draft.shape[0] != B or draft.shape[2] != V or
                                        _dtype_code(draft) != _dtype_code(target)):
        raise ValueError("draft must be [B, Nq, V] with the target's dtype")
    max_out = N + 1 if max_out is None else int(max_out)
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, max_out, dtype=torch.int32, device=dev),
            out_nodes=torch.empty(B, max(max_out - 1, 0), dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
        if aux:
            out["accept"] = torch.empty(B, N, dtype=torch.float32, device=dev)
    rc = lib.tree_verify_sample(_ptr(target), _ptr(draft) if Nq > 0 else None, _dtype_code(target),
                                _ptr(parents), _ptr(tokens), _ptr(qrow), _ptr(uniforms), B, N, Nq,
                                V, float(temperature), max_out, _ptr(out["accepted_len"]),
                                _ptr(out["out_tokens"]), _ptr(out.get("out_nodes")),
                                _ptr(out.get("row_status")), _ptr(out.get("accept")),
                                _stream(stream))
    _check(rc)
    return out


def smc_verify(target, draft, draft_tokens, log_weights, uniforms, groups: int, temperature: float,
               ess_threshold: float, *, out=None, workspace: Workspace | None = None, stream=None):
    """The verify side of one SMC-SD round on the GPU.

    target [B, K+1, V], draft [B, K, V], draft_tokens [B, K] int32, log_weights [B] float32,
    uniforms [B, 2] float32, B = groups * particles.  Returns out_tokens, accepted_len, row_status,
    log_weights (after the round), block_log_ratio, ess, resampled and ancestors.
    """
    lib = load()
    _need_cuda(target, draft, draft_tokens, log_weights, uniforms)
    B, k1, V = target.shape
    K = k1 - 1
    if groups < 1 or B % groups:
        raise ValueError("the batch must split into equal groups of particles")
    Np = B // groups
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
            log_weights=torch.empty(B, dtype=torch.float32, device=dev),
            block_log_ratio=torch.empty(B, dtype=torch.float32, device=dev),
            ess=torch.empty(groups, dtype=torch.float32, device=dev),
            resampled=torch.empty(groups, dtype=torch.int32, device=dev),
            ancestors=torch.empty(B, dtype=torch.int32, device=dev),
        )
    nbytes = workspace_bytes(B, K, V)
    ws = _workspace(workspace, dev).get(nbytes)
    rc = lib.smc_verify(_ptr(target), _ptr(draft) if K > 0 else None, _dtype_code(target),
                        _ptr(draft_tokens), _ptr(log_weights), _ptr(uniforms), groups, Np, K, V,
                        float(temperature), float(ess_threshold), _ptr(out["accepted_len"]),
                        _ptr(out["out_tokens"]), _ptr(out["log_weights"]),
                        _ptr(out.get("block_log_ratio")), _ptr(out.get("ess")),
                        _ptr(out.get("resampled")), _ptr(out.get("ancestors")),
                        _ptr(out.get("row_status")), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc)
    return out


def spec_verify_greedy(target, draft_tokens, *, out=None, workspace: Workspace | None = None,
                       stream=None):
    """Linear greedy verify on the GPU.  target [B, gamma+1, V]; draft_tokens [B, gamma] int32."""
    lib = load()
    _need_cuda(target, draft_tokens)
    B, g1, V = target.shape
    gamma = g1 - 1
    dev = target.device
    if out is None:
        out = dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_tokens=torch.empty(B, gamma + 1, dtype=torch.int32, device=dev),
            row_status=torch.empty(B, dtype=torch.int32, device=dev),
        )
    nbytes = workspace_bytes(B, 0, V, 0, max(gamma, 1))
    ws = _workspace(workspace, dev).get(nbytes)
    rc = lib.spec_verify_greedy(_ptr(target), _dtype_code(target), _ptr(draft_tokens), B, gamma, V,
                                _ptr(out["accepted_len"]), _ptr(out["out_tokens"]),
                                _ptr(out.get("row_status")), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc)
    return out
