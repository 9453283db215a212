"""Replica timing across ranks (the bench's multi-GPU path has no exchange
step: each rank runs an independent replica; the job's rate is every rank's
units over the slowest rank's time).  Two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 0.5 + rank                                   # rank r took 0.5 + r seconds
        t_max = bench.max_over_ranks(t, torch.device("cpu"))
        out[rank] = (t_max, bench.job_throughput(100, t_max, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: (1.5, 200 / 1.5), 1: (1.5, 200 / 1.5)}


def test_single_process_passes_through():
    assert bench.max_over_ranks(2.0, torch.device("cpu")) == 2.0
    assert bench.job_throughput(64, 2.0, 1) == 32.0


def test_bench_starts_its_own_ranks():
    """`bench.py --gpus 2` with no launcher around it starts two ranks under
    torch.distributed.run; here they run the CPU self-test of the rank
    plumbing (gloo), and rank 0 reports n_gpus = 2 and the job rate over the
    slowest rank."""
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"), "--gpus", "2",
                          "--rank-selftest"], capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    r = json.loads(lines[0])
    assert r["n_gpus"] == 2 and r["t_max"] == 0.5 and r["value"] == 400.0
