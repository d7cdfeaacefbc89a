"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the
job time is the maximum over ranks, and under torchrun the oracle arm prints
exactly one JSON line (rank 0) while every rank exits 0."""
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


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    sys.path.insert(0, ROOT)
    import bench
    got = bench._max_over_ranks([1.0 + rank, 5.0 - rank, 2.5], torch.device("cpu"))
    out[rank] = got
    dist.destroy_process_group()


def test_time_is_max_over_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
        assert out[0] == out[1] == [2.0, 5.0, 2.5]
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]  # single process


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny_f32_16x32"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    o = lines[0]
    assert o["impl"] == "reference" and o["n_gpus"] == 2 and o["value"] > 0
    assert o["cpu_baseline"]["kind"] == "oracle" and o["e2e"]["h2d_bytes_per_step"] == 0
    assert o["config"]["workload"] == "tiny_f32_16x32"
