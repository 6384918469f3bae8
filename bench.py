"""Benchmark of the GB300 speculative-decoding verify step.

One step = one pass of the whole hot path over one batch of synthetic inputs per workload:
  c3  spec_verify       B=64  gamma=5 V=128256 bf16 T=0.7         (temperature softmax, residual)
  c4  spec_verify_topk  B=256 gamma=7 V=152064 bf16 T=0.8 k=50    (top-k processor)
  c5  tree_verify_greedy B=32 N=64(+1) V=128256 bf16              (greedy tree walk)
issued back to back on one stream.  ``--workload`` selects a single configuration instead, among
them c6 (tree_verify_sample, B=32 N=64(+1) V=128256 bf16 T=0.7: the stochastic tree walk).  c6
reads only the rows its walk visits (about 31 MB per call, inside L2), so each of its timed calls
follows an L2 flush outside the call's events and its rates come from the per-call event times.
c7 is one SMC-SD round through smc_verify (8 groups x 8 particles, K=5, V=128256 bf16, T=0.7);
c8 linear greedy verify through spec_verify_greedy (B=64 gamma=5 V=128256 bf16); c9 grammar-masked
verify through spec_verify_masked (c3's logits with a valid-token set per position); c10 tree verify
by typical acceptance through tree_verify_typical (c5's tree and logits, T=0.7, eps=0.09, delta=0.3);
c11 top-p verify through spec_verify_topp (B=64 gamma=5 V=128256 bf16, T=0.8, top_p=0.9).

value     logit rows per second, inputs resident in HBM (whole job, all ranks)
e2e       the same metric through the C ABI with host buffers: pinned host -> device copies of
          each step's inputs and a device -> host read of its outputs inside the timed region
roofline  the dominant kernel (the top-k streaming kernel of c4) against measured HBM copy
          bandwidth; achieved = algorithmic bytes per launch / that kernel's event-timed duration
cpu_baseline  the fp64 oracle on the host cores over a bounded sample of the same workload

Multi-GPU (torchrun): every rank verifies its own batch (independent requests, no collective on
the data path); only the timing uses a barrier and a max over ranks.  ``--impl reference`` times
the oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify rows/sec and achieved HBM GB/s (fraction of GB300 peak) per config"
L2_BYTES = 129 * 10**6
SUITE = ("c3", "c4", "c5")
SMALL = ("c1", "c2")   # timed per call beside the suite
PER_CALL = 300         # back-to-back calls per configuration for the per-call times
# the dominant kernel of each workload's call (timed alone through spec_set_kernel_events) and
# the sources it is built from
KERNEL_OF = {
    "c1": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c2": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c3": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c4": ("topk_stream_kernel", ["sv_topk.cu", "sv_common.cuh", "sv_plan.cuh"]),
    "c5": ("tree_stream_kernel", ["sv_tree.cu", "sv_common.cuh"]),
    "c6": ("tree_sample_kernel", ["sv_tree_sample.cu", "sv_tree_sample.cuh", "sv_common.cuh"]),
    "c7": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c8": ("tree_stream_kernel", ["sv_tree.cu", "sv_common.cuh"]),
    "c9": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c11": ("spec_stream_kernel", ["sv_softmax.cu", "sv_draw.cuh", "sv_common.cuh", "sv_plan.cuh"]),
    "c10": ("typical_stream_kernel", ["sv_typical.cu", "sv_typical.cuh", "sv_tree_walk.cuh",
                                      "sv_common.cuh", "sv_plan.cuh"]),
}
DOMINANT_CFG = "c4"


# ------------------------------------------------------------------ workloads

def workload_batches(names, rank, requests=None):
    from speculative_decoding_verification_spec_gb300 import synth as S
    out = {}
    for n in names:
        cfg = (S.CONFIGS.get(n) or S.MASK_CONFIGS.get(n) or S.TOPP_CONFIGS.get(n)
               or S.TREE_CONFIGS.get(n) or S.SAMPLE_TREE_CONFIGS.get(n) or S.SMC_CONFIGS[n])
        kw = dict(seed=rank_seed(cfg, rank))
        if requests:
            kw["groups" if n in S.SMC_CONFIGS else "B"] = requests
        cfg = S.scaled(cfg, **kw)
        if n in S.CONFIGS or n in S.MASK_CONFIGS or n in S.TOPP_CONFIGS:
            out[n] = S.make_spec_batch(cfg)
        elif n in S.TREE_CONFIGS:
            out[n] = S.make_tree_batch(cfg)
        elif n in S.SAMPLE_TREE_CONFIGS:
            out[n] = S.make_sample_tree_batch(cfg)
        else:
            out[n] = S.make_smc_batch(cfg)
    return out


def is_sample_tree(b) -> bool:
    return hasattr(b, "qrow")


def is_greedy_tree(b) -> bool:
    return hasattr(b, "logits")


def is_smc(b) -> bool:
    return hasattr(b, "log_weights")


def sample_tree_rows_read(b, accepted_len, accept) -> int:
    """Rows one tree_verify_sample call reads: the target row of every node its walk arrives at,
    and one proposal row for each of those nodes whose children it tested (the children of a node
    share the proposal row at their parent)."""
    rows = 0
    for i in range(b.parents.shape[0]):
        rows += int(accepted_len[i]) + 1
        tested = np.flatnonzero(~np.isnan(accept[i]))
        rows += len(set(zip(b.parents[i, tested].tolist(), b.qrow[i, tested].tolist())))
    return rows


# ------------------------------------------------------------------ ranks

def rank_seed(cfg, rank: int) -> int:
    """Each rank verifies its own requests: the configuration's seed offset by the rank."""
    return cfg.seed + 7919 * rank


def dist_max(x: float, world: int, device) -> float:
    """The maximum of x over all ranks (x itself on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step_per_rank: float, world: int, steps: int, elapsed_max: float) -> float:
    """Units all ranks processed per second of the slowest rank (weak scaling)."""
    return units_per_step_per_rank * world * steps / elapsed_max


def describe(names):
    from speculative_decoding_verification_spec_gb300 import synth as S
    parts = []
    for n in names:
        if n in S.TOPP_CONFIGS:
            c = S.TOPP_CONFIGS[n]
            parts.append(f"{n} spec_verify_topp B={c.B} gamma={c.gamma} V={c.V} {c.dtype} "
                         f"T={c.temperature} top_p={c.top_p}")
        elif n in S.MASK_CONFIGS:
            c = S.MASK_CONFIGS[n]
            parts.append(f"{n} spec_verify_masked B={c.B} gamma={c.gamma} V={c.V} {c.dtype} "
                         f"T={c.temperature} grammar valid sets per position (narrow 64 tokens / "
                         f"half / wide 99%, equal odds)")
        elif n in S.CONFIGS:
            c = S.CONFIGS[n]
            op = "spec_verify_topk" if c.top_k else "spec_verify"
            parts.append(f"{n} {op} B={c.B} gamma={c.gamma} V={c.V} {c.dtype} T={c.temperature}"
                         + (f" top_k={c.top_k}" if c.top_k else ""))
        elif n in S.TREE_CONFIGS and S.TREE_CONFIGS[n].typical:
            c = S.TREE_CONFIGS[n]
            parts.append(f"{n} tree_verify_typical B={c.B} N={c.max_nodes}(+1 frontier row) V={c.V} "
                         f"{c.dtype} T={c.temperature} eps={c.eps} delta={c.delta} tree "
                         f"{'/'.join(map(str, c.branching))}")
        elif n in S.TREE_CONFIGS and S.TREE_CONFIGS[n].chain:
            c = S.TREE_CONFIGS[n]
            parts.append(f"{n} spec_verify_greedy B={c.B} gamma={c.max_nodes} V={c.V} {c.dtype}")
        elif n in S.TREE_CONFIGS:
            c = S.TREE_CONFIGS[n]
            parts.append(f"{n} tree_verify_greedy B={c.B} N={c.max_nodes}(+1 frontier row) V={c.V} "
                         f"{c.dtype} tree {'/'.join(map(str, c.branching))}")
        elif n in S.SMC_CONFIGS:
            c = S.SMC_CONFIGS[n]
            parts.append(f"{n} smc_verify {c.groups} groups x {c.particles} particles K={c.K} "
                         f"V={c.V} {c.dtype} T={c.temperature} eta={c.eta}")
        else:
            c = S.SAMPLE_TREE_CONFIGS[n]
            parts.append(f"{n} tree_verify_sample B={c.B} N={c.max_nodes}(+1 frontier row) V={c.V} "
                         f"{c.dtype} T={c.temperature} tree {'/'.join(map(str, c.branching))}, "
                         f"children i.i.d. from the draft row at their parent")
    return " + ".join(parts)


def kernels_per_call(batch):
    """Kernels one verify call launches on the 16-byte-vector (streaming) paths the suite uses."""
    if is_sample_tree(batch):
        return 1                              # the clustered walk
    if is_greedy_tree(batch):
        return 2                              # argmax stream + tree finish
    if is_smc(batch):
        return 4                              # stream + row plan + extension draw + group step
    if batch.cfg.top_k:
        return 2                              # stream + finish (dense rows inside the finish)
    return 3                                  # stream + row plan + residual


# ------------------------------------------------------------------ clocks

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"sv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ acceptance diagnostics

def acceptance_diagnostics(accepted_len, row_status, K: int) -> dict:
    """The per-round measurements M7.1 ("0x05A/0x05B": the accepted-prefix law and round progress)
    lists for diagnosis, from one call's outputs: over the requests whose status is OK,
    Pr(A = a) for a = 0..K, the tails s_j = Pr(A >= j) for j = 1..K, the reach-conditioned rates
    alpha_j^reach = Pr(A >= j | A >= j-1) (averaged only over requests that reach position j), and
    the expected round progress E[G] = 1 + sum_j s_j (the accepted drafts plus the correction or
    bonus token).  For a tree, A is the depth of the accepted node and K the deepest level."""
    a = np.asarray(accepted_len)[np.asarray(row_status) == 0].astype(np.int64)
    n = int(a.size)
    out = {"requests": n, "K": int(K)}
    if n == 0:
        return out
    pa = np.bincount(np.clip(a, 0, K), minlength=K + 1)[:K + 1] / n
    tail = [float((a >= j).mean()) for j in range(0, K + 1)]  # tail[0] = 1
    alpha = [tail[j] / tail[j - 1] if tail[j - 1] > 0 else None for j in range(1, K + 1)]
    out.update({
        "pr_A": [round(float(x), 6) for x in pa],
        "pr_A_ge": [round(x, 6) for x in tail[1:]],
        "alpha_reach": [None if x is None else round(x, 6) for x in alpha],
        "mean_A": round(float(a.mean()), 6),
        "E_G": round(1.0 + float(sum(tail[1:])), 6),
    })
    return out


def read_bytes_nominal(b) -> int:
    """Bytes of the inputs one call is handed: every logit, plus the grammar mask's words.  This is
    the algorithmic byte count of every call except the sampled tree, whose walk reads only the
    rows it visits (counted after its first call)."""
    if is_sample_tree(b):
        return b.target.nbytes + b.draft.nbytes
    return b.logit_bytes + (b.allowed.nbytes if getattr(b, "allowed", None) is not None else 0)


def needs_flush(b) -> bool:
    """Calls whose reads fit in L2 are timed after an L2 flush: the sampled tree always (its walk
    reads a few rows), the others when all their inputs fit."""
    return is_sample_tree(b) or read_bytes_nominal(b) < L2_BYTES


def run_config(names, batches, world: int, requests=None) -> dict:
    """The ``config`` object of the JSON line, the same in both arms: it depends only on the
    workload's inputs."""
    rows_step = sum(batches[n].rows for n in names)
    bytes_step = sum(read_bytes_nominal(batches[n]) for n in names)
    if any(needs_flush(batches[n]) for n in names):
        l2 = "L2 flushed (256 MB write) before every call, outside its events"
    else:
        l2 = f"inputs larger than L2 ({bytes_step / 1e6:.0f} MB per step > 129 MB); no flush"
    return {"workload": describe(names), "input_dtype": "bf16",
            "logit_rows_per_step": rows_step, "input_bytes_per_step": bytes_step,
            "l2": l2, "parallelism": f"replicas x{world} (independent requests per rank)",
            **({"requests_override": requests} if requests else {})}


# ------------------------------------------------------------------ helpers

def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_verification_spec_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def recorded_traffic(kernel, sha):
    """dram bytes per launch from the committed ncu summary, if taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[kernel]
        if rec.get("source_sha") == sha:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def _oracle_one(O, b, i):
    """The oracle on request i (for SMC: group i) of batch b; returns (rows verified, outputs)."""
    if is_sample_tree(b):
        o = O.tree_verify_sample(b.target[i:i + 1], b.draft[i:i + 1], b.parents[i:i + 1],
                                 b.tokens[i:i + 1], b.qrow[i:i + 1], b.uniforms[i:i + 1],
                                 b.cfg.temperature)
        return b.target.shape[1], o
    if is_greedy_tree(b) and b.cfg.typical:
        o = O.tree_verify_typical(b.logits[i:i + 1], b.parents[i:i + 1], b.tokens[i:i + 1],
                                  b.uniforms[i:i + 1], b.cfg.temperature, b.cfg.eps, b.cfg.delta)
        return b.logits.shape[1], o
    if is_greedy_tree(b):
        return b.logits.shape[1], O.tree_verify_greedy(b.logits[i:i + 1], b.parents[i:i + 1],
                                                       b.tokens[i:i + 1])
    if is_smc(b):
        Np = b.cfg.particles
        sl = slice(i * Np, (i + 1) * Np)
        o = O.smc_verify(b.target[sl], b.draft[sl], b.draft_tokens[sl],
                         b.log_weights[sl].astype(np.float64), b.uniforms[sl], 1,
                         b.cfg.temperature, b.cfg.eta)
        return Np * (2 * b.cfg.K + 1), o
    o = O.spec_verify(b.target[i:i + 1], b.draft[i:i + 1], b.draft_tokens[i:i + 1],
                      b.uniforms[i:i + 1], b.cfg.temperature, b.cfg.top_k,
                      allowed=None if b.allowed is None else b.allowed[i:i + 1],
                      top_p=b.cfg.top_p if b.cfg.top_p < 1.0 else None)
    return 2 * b.cfg.gamma + 1, o


def _units(b) -> int:
    return b.cfg.groups if is_smc(b) else b.cfg.B


def _parity_counts(b, gpu, idx, outs):
    """{requests, flagged, mismatched} of the matching rules over the requests in idx: the GPU's
    accepted lengths and tokens against the oracle's, a request flagged when its oracle margin
    (a used uniform's distance to a decision boundary) is below the rule's bound."""
    if gpu is None or not idx or is_smc(b):
        return None
    bound = 1e-5 if (is_greedy_tree(b) and b.cfg.typical) else 1e-6
    n = f = m = 0
    for i, o in zip(idx, outs):
        same = (int(gpu["accepted_len"][i]) == int(o["accepted_len"][0])
                and np.array_equal(gpu["out_tokens"][i][:o["out_tokens"].shape[1]], o["out_tokens"][0])
                and int(gpu["row_status"][i]) == int(o["row_status"][0]))
        flag = bool(o.get("margin", np.array([np.inf]))[0] < bound)
        n, f, m = n + 1, f + flag, m + (not same)
    return {"requests": n, "flagged": f, "mismatched": m,
            "rule": f"bit-exact tokens, lengths and statuses except draws within {bound:g} of a "
                    "boundary (flagged)" + ("; trees bit-exact" if is_greedy_tree(b) and not b.cfg.typical else "")}


def cpu_baseline(names, budget_s=15.0, gpu_outs=None, all_cores=True):
    """The oracle as it stands on a bounded sample of each workload: single-threaded (the line's
    value), and over every host core with a process pool over whole requests.  With ``gpu_outs``
    (the bench's first call of each configuration, same inputs) the sampled requests also give the
    matching rules' counts.  Returns (cpu_baseline, parity)."""
    from oracle import oracle as O
    from oracle import pool as OP
    batches = workload_batches(names, 0)
    per_row_s, sample, parity = {}, [], {}
    share = budget_s / len(names)
    for n, b in batches.items():
        rows_done, t_used, i = 0, 0.0, 0
        idx, outs = [], []
        while t_used < share and i < _units(b):
            t0 = time.perf_counter()
            r, o = _oracle_one(O, b, i)
            t_used += time.perf_counter() - t0
            rows_done += r
            idx.append(i)
            outs.append(o)
            i += 1
        per_row_s[n] = t_used / rows_done
        sample.append(f"{n}: {i} {'groups of particles' if is_smc(b) else 'requests'} "
                      f"({rows_done} rows)")
        parity[n] = _parity_counts(b, (gpu_outs or {}).get(n), idx, outs)
    rows = {n: batches[n].rows for n in names}
    step_s = sum(per_row_s[n] * rows[n] for n in names)
    base = {"value": sum(rows.values()) / step_s, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": "; ".join(sample) + "; single-threaded fp64 C oracle, scaled to one step",
            "host": {"nproc": os.cpu_count(), "cpu_model": OP.cpu_model()}}
    # every host core: whole configurations through a pool of worker processes (spawn), one block
    # of requests per task; only calls the pool covers (plain, processors, top-k, greedy tree)
    pooled = [n for n in names if not is_sample_tree(batches[n]) and not is_smc(batches[n])
              and not (is_greedy_tree(batches[n]) and batches[n].cfg.typical)]
    if all_cores and pooled:
        procs = OP.cores()
        t0 = time.perf_counter()
        for n in pooled:
            b = batches[n]
            if is_greedy_tree(b):
                OP.tree_verify_greedy(b.logits, b.parents, b.tokens, procs=procs)
            else:
                OP.spec_verify(b.target, b.draft, b.draft_tokens, b.uniforms, b.cfg.temperature,
                               b.cfg.top_k, allowed=b.allowed,
                               top_p=b.cfg.top_p if b.cfg.top_p < 1.0 else None, procs=procs)
        el = time.perf_counter() - t0
        done = sum(rows[n] for n in pooled)
        base["all_cores"] = {"value": done / el, "unit": "rows/s", "cores": procs,
                             "cpu_model": base["host"]["cpu_model"],
                             "sample": f"every request of {', '.join(pooled)} ({done} rows) in "
                                       f"{el:.2f} s, worker start-up included"}
    return base, parity


# ------------------------------------------------------------------ our arm

def percentiles(ms):
    """median and p10 / p90 of per-call times (ms)."""
    q = np.percentile(np.asarray(ms, dtype=np.float64), [10, 50, 90])
    return {"p10": round(float(q[0]), 5), "median": round(float(q[1]), 5), "p90": round(float(q[2]), 5),
            "mean": round(float(np.mean(ms)), 5), "calls": len(ms)}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_spec_gb300 as sv

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    names = SUITE if args.workload == "suite" else (args.workload,)
    # the suite's step is the large configurations; the small ones (c1, c2) are timed per call
    # beside it, since each is a few microseconds of launch-bound work
    extra = tuple(n for n in SMALL if n not in names) if args.workload == "suite" else ()
    batches = workload_batches(names + extra, rank, args.requests)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    host, devin, outs, wss = {}, {}, {}, {}
    for n, b in batches.items():
        if is_sample_tree(b):
            arrs = dict(target=b.target, draft=b.draft, parents=b.parents, tokens=b.tokens,
                        qrow=b.qrow, uniforms=b.uniforms)
        elif is_greedy_tree(b):
            arrs = dict(logits=b.logits, parents=b.parents, tokens=b.tokens)
            if b.uniforms is not None:
                arrs["uniforms"] = b.uniforms
        elif is_smc(b):
            arrs = dict(target=b.target, draft=b.draft, tokens=b.draft_tokens,
                        log_weights=b.log_weights, uniforms=b.uniforms)
        else:
            arrs = dict(target=b.target, draft=b.draft, tokens=b.draft_tokens, uniforms=b.uniforms)
            if b.allowed is not None:
                arrs["allowed"] = b.allowed.view(np.int32)
        host[n] = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16
                                       else np.ascontiguousarray(v)).pin_memory()
                   for k, v in arrs.items()}
        devin[n] = {k: v.to(dev) for k, v in host[n].items()}
        wss[n] = sv.Workspace(dev)

    def call(n, ins, out=None, st=stream):
        b = batches[n]
        if is_sample_tree(b):
            return sv.tree_verify_sample(ins["target"], ins["draft"], ins["parents"], ins["tokens"],
                                         ins["qrow"], ins["uniforms"], b.cfg.temperature, out=out,
                                         aux=True, stream=st)
        if is_smc(b):
            return sv.smc_verify(ins["target"], ins["draft"], ins["tokens"], ins["log_weights"],
                                 ins["uniforms"], b.cfg.groups, b.cfg.temperature, b.cfg.eta,
                                 out=out, workspace=wss[n], stream=st)
        if is_greedy_tree(b) and b.cfg.typical:
            return sv.tree_verify_typical(ins["logits"], ins["parents"], ins["tokens"],
                                          ins["uniforms"], b.cfg.temperature, b.cfg.eps,
                                          b.cfg.delta, out=out, workspace=wss[n], stream=st)
        if is_greedy_tree(b) and b.cfg.chain:
            return sv.spec_verify_greedy(ins["logits"], ins["tokens"], out=out, workspace=wss[n],
                                         stream=st)
        if is_greedy_tree(b):
            return sv.tree_verify_greedy(ins["logits"], ins["parents"], ins["tokens"], out=out,
                                         workspace=wss[n], stream=st)
        return sv.spec_verify(ins["target"], ins["draft"], ins["tokens"], ins["uniforms"],
                              b.cfg.temperature, top_k=b.cfg.top_k, allowed=ins.get("allowed"),
                              top_p=b.cfg.top_p if b.cfg.top_p < 1.0 else None,
                              out=out, workspace=wss[n], stream=st)

    for n in batches:  # allocate outputs once
        outs[n] = call(n, devin[n])
    torch.cuda.synchronize()
    first = {n: {k: v.cpu().numpy() for k, v in outs[n].items()} for n in batches}
    # algorithmic bytes of one call: the logits it reads (all of them, except on the sampled tree,
    # whose walk reads only the rows it visits)
    read_bytes = {}
    for n, b in batches.items():
        if is_sample_tree(b):
            rows = sample_tree_rows_read(b, first[n]["accepted_len"], first[n]["accept"])
            read_bytes[n] = rows * b.cfg.V * b.target.itemsize
        else:
            read_bytes[n] = read_bytes_nominal(b)
    # calls whose reads fit in L2 are timed after an L2 flush (a 256 MB write), outside their events
    flush_buf = None
    if any(needs_flush(b) for b in batches.values()):
        flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_step = any(needs_flush(batches[n]) for n in names)

    def flush(n):
        if needs_flush(batches[n]):
            flush_buf.zero_()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- device-resident timing
    for _ in range(args.warmup):
        for n in names:
            call(n, devin[n], outs[n])
    ev = {n: [] for n in names}
    barrier()
    torch.cuda.synchronize()
    dom_cfg = DOMINANT_CFG if DOMINANT_CFG in names else names[0]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:  # create the CUDA events before the timed region
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            for n in names:
                if flush_step:
                    flush(n)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if n == dom_cfg:
                    sv.set_kernel_events(*kev[i])
                call(n, devin[n], outs[n])
                if n == dom_cfg:
                    sv.set_kernel_events(None, None)
                e1.record(stream)
                ev[n].append((e0, e1))
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    if not flush_step:
        elapsed = dist_max(start.elapsed_time(end) / 1e3, world, dev)
    else:  # the flushes are not verify work: the step time is the sum of the calls' event times
        elapsed = dist_max(sum(a.elapsed_time(b) for n in names for a, b in ev[n]) / 1e3, world, dev)
    call_ms_timed = {n: statistics.mean(a.elapsed_time(b) for a, b in ev[n]) for n in names}
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)

    # ---- per-configuration call times: PER_CALL back-to-back calls of each configuration alone,
    # each bracketed by events on the call's stream (no event inside a call, so its dependent
    # launches overlap as in use); configurations that fit in L2 are flushed before every call
    per_ms = {n: [] for n in batches}
    for n in batches:
        for _ in range(3):
            call(n, devin[n], outs[n])
        pairs = []
        for i in range(PER_CALL):
            if flush_buf is not None:
                flush(n)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(n, devin[n], outs[n])
            e1.record(stream)
            pairs.append((e0, e1))
        torch.cuda.synchronize()
        per_ms[n] = [a.elapsed_time(b) for a, b in pairs]

    # the small configurations once more as CUDA-graph replays: one captured call, replayed, so
    # the host's launch cost is out of the time (how a serving loop would issue them)
    graph_ms = {}
    for n in extra:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(2):
                    call(n, devin[n], outs[n], st=side)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call(n, devin[n], outs[n], st=torch.cuda.current_stream())
            torch.cuda.synchronize()
            pairs = []
            for i in range(PER_CALL):
                flush(n)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                pairs.append((e0, e1))
            torch.cuda.synchronize()
            graph_ms[n] = [a.elapsed_time(b) for a, b in pairs]
            del g
        except Exception as exc:  # reported, not fatal: the direct calls are timed above
            graph_ms[n] = f"capture failed: {type(exc).__name__}: {exc}"[:200]

    # c1 is one request: its acceptance law is read from its 10,000 seeded trials in one call
    diag_outs = {}
    if "c1" in batches and not args.requests:
        from speculative_decoding_verification_spec_gb300 import synth as S
        tb = S.trial_batches(S.scaled(batches["c1"].cfg), 10000)
        t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
             for k, v in dict(target=tb.target, draft=tb.draft, tokens=tb.draft_tokens,
                              uniforms=tb.uniforms).items()}
        o = sv.spec_verify(t["target"], t["draft"], t["tokens"], t["uniforms"], tb.cfg.temperature,
                           stream=stream)
        torch.cuda.synchronize()
        diag_outs["c1"] = {k: v.cpu().numpy() for k, v in o.items()}

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        host_out = {n: {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                        for k, v in outs[n].items()} for n in names}
        h2d = sum(v.numel() * v.element_size() for n in names for v in host[n].values())
        d2h = sum(v.numel() * v.element_size() for n in names for v in host_out[n].values())
        e2e_steps = max(3, min(args.steps, args.e2e_steps))

        def e2e_step():
            for n in names:
                for k, v in host[n].items():
                    devin[n][k].copy_(v, non_blocking=True)
                call(n, devin[n], outs[n])
                for k, v in outs[n].items():
                    host_out[n][k].copy_(v, non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_el = dist_max(s0.elapsed_time(s1) / 1e3, world, dev)
        rows_step = sum(batches[n].rows for n in names)
        e2e = {"value": whole_job_rate(rows_step, world, e2e_steps, e_el), "unit": "rows/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": e2e_steps}

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return

    peak, peak_kind = measured_peak()
    rows_step = sum(batches[n].rows for n in names)
    bytes_step = sum(read_bytes[n] for n in names)
    per_cfg = {}
    for n, b in batches.items():
        pc = percentiles(per_ms[n])
        med = pc["median"]
        gbs = read_bytes[n] / (med / 1e3) / 1e9
        per_cfg[n] = {"call_ms": pc, "rows_per_s": b.rows / (med / 1e3),
                      "requests_per_s": _units(b) / (med / 1e3), "calls_per_s": 1e3 / med,
                      "logit_bytes": read_bytes[n], "hbm_gbs": round(gbs, 1),
                      "frac_of_measured_peak": round(gbs / peak, 4),
                      "frac_of_8tbs": round(gbs / 8000.0, 4),
                      "l2": "flushed before every call (its reads fit in L2)" if needs_flush(b)
                            else "inputs larger than L2, no flush"}
        if n in call_ms_timed:
            per_cfg[n]["call_ms_timed_region"] = round(call_ms_timed[n], 5)
        if n in graph_ms:
            gm = graph_ms[n]
            per_cfg[n]["graph_replay"] = (gm if isinstance(gm, str) else
                                          {"call_ms": percentiles(gm),
                                           "calls_per_s": 1e3 / percentiles(gm)["median"]})
        if not is_sample_tree(b) and not is_smc(b):
            K = b.cfg.max_nodes if is_greedy_tree(b) and b.cfg.chain else (
                int(S_tree_depth(b)) if is_greedy_tree(b) else b.cfg.gamma)
            acc = diag_outs.get(n, first[n])
            per_cfg[n]["acceptance"] = acceptance_diagnostics(acc["accepted_len"],
                                                              acc["row_status"], K)
            if n in diag_outs:
                per_cfg[n]["acceptance"]["sample"] = (f"{len(acc['accepted_len'])} seeded trials "
                                                      "of the configuration (one call)")
            eg = per_cfg[n]["acceptance"].get("E_G")
            if eg:
                per_cfg[n]["acceptance"]["bytes_per_committed_token"] = round(
                    read_bytes[n] / (eg * _units(b)), 1)
    dom_kernel, dom_files = KERNEL_OF[dom_cfg]
    sha = source_sha(dom_files)
    achieved = read_bytes[dom_cfg] / (kernel_ms / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": whole_job_rate(rows_step, world, args.steps, elapsed),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": run_config(names, batches, world, args.requests),
        "hbm_gbs": bytes_step * world * args.steps / elapsed / 1e9,
        "per_config": per_cfg,
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "workload": dom_cfg,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic(dom_kernel, sha), "source_sha": sha,
                     "kernel_ms": round(kernel_ms, 5),
                     "timing": "CUDA events recorded on the call's stream around this kernel's "
                               "launch (spec_set_kernel_events), mean over the timed steps; "
                               "algorithmic bytes = the logit bytes the call reads, once"
                               + (" (the sampled tree: the rows its walk visits)"
                                  if is_sample_tree(batches[dom_cfg]) else "")},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps * sum(kernels_per_call(batches[n]) for n in names),
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        cb, parity = cpu_baseline(names + extra, args.cpu_budget, first)
        line["cpu_baseline"] = cb
        line["parity"] = parity
    print(json.dumps(line), flush=True)


def S_tree_depth(b) -> int:
    """The deepest level of a greedy tree batch (depth of a node = 1 + its parent's)."""
    par = b.parents[0]
    depth = np.zeros(len(par), np.int64)
    for i, p in enumerate(par):
        depth[i] = 1 if p < 0 else depth[p] + 1
    return int(depth.max()) if len(depth) else 0


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return
    names = SUITE if args.workload == "suite" else (args.workload,)
    from oracle import oracle as O
    O.build()
    batches = workload_batches(names, 0, args.requests)
    # each step verifies a bounded sample: one request of one workload, the workloads in turn, so
    # that the default --steps run ends within a few minutes on one host core
    def step(i):
        b = batches[names[i % len(names)]]
        rows, _ = _oracle_one(O, b, (i // len(names)) % _units(b))
        return rows

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    rows = 0
    for i in range(args.steps):
        rows += step(args.warmup + i)
    el = time.perf_counter() - t0
    value = rows / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(names, batches, world, args.requests),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": "each step verifies one request (a group of particles for "
                                       "SMC) of one workload, the workloads in turn, single "
                                       "thread; value = rows verified / time"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["suite", "c1", "c2", "c3", "c4", "c5", "c6", "c7", "c8",
                                           "c9", "c10", "c11"],
                    default="suite")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--requests", type=int, default=None,
                    help="profiling aid: run the selected workload with this many requests instead "
                         "of its own B (the line's config records it; not a bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
