"""The multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

The verify path does not shard anything: on N GPUs every rank verifies its own independent requests
(weak scaling).  What the ranks share is host logic: each rank draws its own seeded inputs, the
timing takes the maximum over ranks, the whole-job rate counts every rank's rows, and only rank 0
prints.  These tests run that logic with world_size 2 over gloo; no GPU is involved.
"""
import hashlib
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def digest(batch):
    h = hashlib.sha256()
    for a in (batch.target, batch.draft, batch.draft_tokens, batch.uniforms):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        b = bench.workload_batches(["c1", "c2"], rank)
        again = bench.workload_batches(["c1", "c2"], rank)
        mine = {n: digest(b[n]) for n in b}
        same = all(digest(again[n]) == mine[n] for n in b)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        # elapsed times that differ per rank: the job's time is the slowest rank's
        el = 0.5 + 0.25 * rank
        mx = bench.dist_max(el, world, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"same": same, "gathered": gathered, "max": mx, "rows": b["c2"].rows}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_draw_their_own_inputs_and_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["same"], "a rank's inputs must be reproducible from its seed"
        assert r["max"] == pytest.approx(0.75)
    g = res[0]["gathered"]
    assert g == res[1]["gathered"]
    for n in ("c1", "c2"):
        assert g[0][n] != g[1][n], "ranks must verify different requests"


def test_whole_job_rate_and_rank_seeds():
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verification_spec_gb300 import synth as S
    # 2 ranks x 72 rows per step x 10 steps in 0.5 s of the slowest rank
    assert bench.whole_job_rate(72, 2, 10, 0.5) == pytest.approx(2880.0)
    assert bench.dist_max(3.0, 1, "cpu") == 3.0
    seeds = {bench.rank_seed(S.CONFIGS["c3"], r) for r in range(8)}
    assert len(seeds) == 8


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "c1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
