"""The N > 1 host logic on CPU with two gloo ranks (the operation has no exchange step: replicas only, each
rank runs its own batch-heads, and the job's time is the slowest rank's)."""
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


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        out[rank] = ms
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_value_counts_every_replica():
    import bench

    # two replicas of 1e12 FLOP each in 10 ms: 200 TFLOP/s for the job
    assert bench.whole_job_tflops(1e12, 2, 10.0) == pytest.approx(200.0)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_reference_arm_under_two_ranks_prints_one_line():
    """Launched the way the driver launches N > 1 runs; rank 0 alone times the oracle and prints."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
