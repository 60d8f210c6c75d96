"""The bench's multi-GPU path is replicas only: each rank decodes its own copy of the
workload, and the job's rate is world * steps / (slowest rank's time).  Checked here with
two gloo ranks on the CPU (the GPU runs of this build use one GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import importlib.util
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    rate, slowest = bench.job_rate(1.0 + rank, 10, world, "cpu")   # rank 1 is the slowest
    out[rank] = (rate, slowest)
    dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank():
    world = 2
    out = mp.get_context("spawn").Manager().dict()     # no fork of a threaded process
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        rate, slowest = out[rank]
        assert slowest == 2.0 and rate == world * 10 / 2.0


def test_reference_arm_prints_one_line_from_rank_zero():
    """`bench.py --impl reference` under torchrun with two ranks: rank 0 alone runs the oracle
    and prints the JSON line; the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--workload", "tiny_f32"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
