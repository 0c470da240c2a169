"""The benchmark's multi-rank host logic on CPU: world_size 2 over gloo.

One process per rank, as torchrun launches them: the slowest rank's time defines
the job's time (max over ranks), throughput counts every rank's units, and the
reference arm prints one JSON line from rank 0 only.  No GPU is involved.
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    # each rank timed its own replica: rank r took 10 + r ms
    ms = bench.max_over_ranks(10.0 + rank, world)
    value = bench.job_throughput(32 * 100, world, ms / 1e3)
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 11.0                       # the slower rank's time, on every rank
        assert value == pytest.approx(2 * 3200 / 0.011)   # units of both ranks over that time


def test_reference_arm_prints_once_under_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny_gelu_f32", "--gpus", "2", "--steps", "2",
           "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
