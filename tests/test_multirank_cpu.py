"""The bench's multi-rank logic on CPU: world_size-2 gloo process groups.

The path shards over the batch with no exchange (replicas); the only cross-rank
step is the max-over-ranks of the timed region, which these tests run with the
gloo backend on 127.0.0.1, plus the reference arm's rule that rank 0 alone runs."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 100.0 + 37.5 * rank            # rank 1 is the slower one
        t = bench.time_max_over_ranks(mine)
        v = bench.job_value(world, 10, 1000, t)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_time_is_the_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()   # no fork of a threaded process
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        t, v = out[r]
        assert t == pytest.approx(137.5)                      # every rank sees the slowest rank's time
        assert v == pytest.approx(world * 10 * 1000 / 0.1375)  # units of all ranks over that time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.time_max_over_ranks(12.5) == 12.5
    assert bench.job_value(1, 4, 100, 2.0) == pytest.approx(200000.0)


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""      # only rank 0 prints the line
