"""The multi-rank (torchrun) path of the benchmark on CPU with the gloo
backend: the slowest rank's time is the job's time, the job's throughput sums
the ranks' work, and under torchrun exactly one rank prints the JSON line."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    values = [3.5, 7.25]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), values, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == max(values)


def test_single_process_and_throughput():
    assert bench.max_over_ranks(2.5, None, None) == 2.5
    # 4 ranks, 1e12 FLOP each, slowest rank 2 ms -> 2e15 FLOP/s for the job
    assert bench.job_throughput(4, 1e12, 2.0) == pytest.approx(2e15)


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks on CPU: rank 0 times the oracle and prints one JSON line,
    the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "C2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
