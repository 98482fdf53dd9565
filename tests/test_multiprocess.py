"""The N > 1 host path of the benchmark, on CPU: two ranks over gloo.

Multi-GPU runs are replicas (each rank runs the whole step on its own GPU);
the only cross-rank steps are the barrier around the timed region and the
maximum of the per-rank times, from which rank 0 reports the whole job's
rate.  Those run here with the gloo backend on 127.0.0.1."""
import os
import socket
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        dist.barrier()
        # rank r was slower on the first timer and faster on the second
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], "cpu")
        rate = bench.whole_job_rate(1000, 10, world, times[0])
        out[rank] = (times, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_two_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        times, rate = out[r]
        assert times == [2.0, 5.0, 0.5]          # every rank sees the maximum
        assert rate == pytest.approx(1000 * 10 * 2 / 2.0)


def test_max_over_ranks_without_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 1.5], "cpu") == [3.0, 1.5]
    assert bench.whole_job_rate(10, 4, 1, 2.0) == 20.0


def test_reference_arm_on_a_non_zero_rank_prints_nothing():
    """Under torchrun only rank 0 runs the oracle arm; the others exit 0."""
    import subprocess

    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
