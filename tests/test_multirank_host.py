"""The N > 1 path of bench.py on the CPU: two gloo ranks (one process each, spawned,
rendezvous on 127.0.0.1).  The GEMM path has no exchange step (replicas only), so the
only cross-rank operations are the barrier and the max over ranks of the step time."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.distributed.barrier()
        out[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    values = [1.25, 3.5]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, values, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == max(values)


def test_max_over_ranks_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_reference_arm_under_torchrun_prints_one_line():
    # rank 0 alone runs the oracle and prints; the other rank exits 0 without work
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
