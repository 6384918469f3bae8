"""Run the fp64 oracle over many requests on all host cores.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this module.  Requests are independent, so a batch is split into
contiguous blocks of requests and each block goes through the unchanged oracle in a worker process.
The workers are started with the ``spawn`` method: a pool forked from a process that already holds
a CUDA context can hang, and spawn is safe before or after the first GPU call.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

from oracle import oracle as O


def cores() -> int:
    """Host threads this process may use."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu's "Model name", else /proc/cpuinfo's first model line)."""
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model", "processor\t: ")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _spec_block(args):
    target, draft, tokens, uniforms, T, top_k, allowed, top_p = args
    return O.spec_verify(target, draft, tokens, uniforms, T, top_k, allowed=allowed, top_p=top_p)


def _tree_block(args):
    logits, parents, tokens, max_out = args
    return O.tree_verify_greedy(logits, parents, tokens, max_out=max_out)


def _merge(parts):
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def _blocks(n: int, procs: int):
    """Contiguous request blocks, a few per worker so that uneven blocks even out."""
    nb = max(1, min(n, procs * 4))
    return [b for b in np.array_split(np.arange(n), nb) if len(b)]


def _map(fn, work, procs):
    """fn over the work items in worker processes, results in order.  A worker that cannot start
    or dies raises BrokenProcessPool here instead of being replaced again and again."""
    if procs <= 1 or len(work) <= 1:
        return [fn(w) for w in work]
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=min(procs, len(work)), mp_context=ctx) as ex:
        return list(ex.map(fn, work))


def spec_verify(target, draft, tokens, uniforms, temperature, top_k=0, allowed=None, top_p=None,
                procs=None):
    """``oracle.spec_verify`` over requests split across ``procs`` worker processes (all host
    threads by default).  Same arguments and result as the oracle."""
    procs = procs or cores()
    n = target.shape[0]
    work = [(target[b[0]:b[-1] + 1], draft[b[0]:b[-1] + 1], tokens[b[0]:b[-1] + 1],
             uniforms[b[0]:b[-1] + 1], temperature, top_k,
             None if allowed is None else allowed[b[0]:b[-1] + 1], top_p)
            for b in _blocks(n, procs)]
    return _merge(_map(_spec_block, work, procs))


def tree_verify_greedy(logits, parents, tokens, max_out=None, procs=None):
    """``oracle.tree_verify_greedy`` over requests split across worker processes."""
    procs = procs or cores()
    n = logits.shape[0]
    work = [(logits[b[0]:b[-1] + 1], parents[b[0]:b[-1] + 1], tokens[b[0]:b[-1] + 1], max_out)
            for b in _blocks(n, procs)]
    return _merge(_map(_tree_block, work, procs))
