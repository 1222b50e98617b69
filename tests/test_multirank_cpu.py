"""The multi-process side of bench.py on CPU with the gloo backend (world size 2): every rank runs an
independent replica, the time is the maximum over ranks, the throughput is summed, and only rank 0
prints.  No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(2, _free_port(), [0.25, 0.75], out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == 0.75 and out[1] == 0.75


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(1.5, 1) == 1.5


def test_replica_throughput_is_weak_scaling():
    # two replicas of 2 TFLOP each, 3 steps, slowest rank 6 s: (2 * 2e12 * 3) / 6 / 1e12 = 2 TFLOP/s
    assert bench.replica_throughput(2e12, 3, 2, 6.0) == pytest.approx(2.0)
    assert bench.replica_throughput(2e12, 3, 1, 6.0) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_prints_once():
    """torchrun with two CPU ranks: rank 0 times the oracle and prints one JSON line, rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
