"""The bench's multi-rank logic on CPU (gloo, world size 2): every path shards
into independent replicas, so the only exchange is the timing reduction, and
under torchrun the reference arm runs on rank 0 alone."""
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


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    # rank r took 10 (r + 1) ms for 100 (r + 1) rows
    ms, rate = bench.job_rate(torch, 10.0 * (rank + 1), 100.0 * (rank + 1), world,
                              torch.device("cpu"))
    out[rank] = (ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_all_units():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, rate = res[r]
        assert ms == 20.0                       # the slower rank
        assert rate == pytest.approx(300.0 / 0.020)  # 100 + 200 rows in 20 ms


def test_job_rate_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench

    ms, rate = bench.job_rate(torch, 8.0, 64.0, 1, torch.device("cpu"))
    assert ms == 8.0 and rate == pytest.approx(8000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """Two ranks on 127.0.0.1: rank 0 times the oracle on a bounded sample and
    prints the only line; rank 1 exits without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
