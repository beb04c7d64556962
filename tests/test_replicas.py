"""The multi-GPU path is replicas only (the single-GPU share has no exchange step): every rank runs
the whole step and the job's time is the slowest rank's.  This checks that aggregation, and the
reference arm's rank handling, with world-size-2 gloo process groups on the CPU."""
import os
import socket
import subprocess
import sys

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]
        ms_all = bench.max_over_ranks(ms, torch.device("cpu"))
        out[rank] = (ms_all, bench.job_value(1e12, world, ms_all))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms_all, value = out[rank]
        assert ms_all == 20.0
        assert abs(value - 2 * 1e12 / 20e-3 / 1e12) < 1e-9   # both replicas' work over the slower time


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(7.0, torch.device("cpu")) == 7.0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
