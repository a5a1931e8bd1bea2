"""Multi-rank host logic of bench.py on CPU: two ranks over gloo.

A job of N replicas reports the slowest rank's time and the tokens of all
ranks; each replica holds the same weights and its own token batch; with
--impl reference only rank 0 works and prints.  No GPU is involved.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from moe_inputs import WORKLOADS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(world, 1000, 4, job_ms)
        wl = WORKLOADS["tiny"]
        g = bench.rank_inputs(wl, 0, rank, "cpu")
        res = dict(job_ms=job_ms, value=value,
                   x_sum=float(g["x"].float().sum()), w13_sum=float(g["w13"].float().sum()))
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_inputs(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    for x in r:
        assert x["job_ms"] == 15.0                       # max over ranks, on every rank
        assert x["value"] == pytest.approx(2 * 1000 * 4 / 0.015)
    assert r[0]["w13_sum"] == r[1]["w13_sum"]            # replicated weights
    assert r[0]["x_sum"] != r[1]["x_sum"]                # each rank its own batch


def test_reference_arm_under_torchrun_prints_on_rank0_only(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "0.2"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
