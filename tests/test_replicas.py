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


def test_kernel_summary_accounting():
    """The bench's per-kernel figures: GEMM FLOPs 2mnk and algorithmic bytes (A, B read once; C
    written, and read as well when accumulated), conversion 6 bytes per element, attention FLOPs
    from the visible pairs; the bound is the roofline whose time is longer."""
    import upipe_inputs as ui
    w = ui.workload("ulysses_1m")
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    S, d, Dh = w.S, w.d, w.Dh
    recs = [
        {"kind": "o_proj", "epilogue": 2, "split_k": 1, "chunk": 1, "m": S, "n": d, "k": Dh, "ms": 10.0},
        {"kind": "qkv_proj", "epilogue": 0, "split_k": 1, "chunk": 0, "m": S, "n": 3 * Dh, "k": d, "ms": 2.0},
        {"kind": "convert", "epilogue": 0, "split_k": 1, "chunk": 3, "m": S * d, "n": 1, "k": 1, "ms": 4.0},
        {"kind": "bwd_dkdv", "epilogue": 0, "split_k": 1, "chunk": 0, "m": S, "n": 1, "k": Dh, "ms": 500.0},
    ]
    out = {e["kernel"]: e for e in bench.summarize_kernels(recs, w, peaks, 4000.0)}
    acc = out["o_proj (fp32 C += A B^T)"]
    assert acc["bound"] == "hbm"                        # K = 128: the fp32 read-modify-write dominates
    assert acc["bytes_per_launch"] == 2 * S * Dh + 2 * d * Dh + 8 * S * d
    assert abs(acc["gbs"] - acc["bytes_per_launch"] / 1e-2 / 1e9) < 1e-6
    qkv = out["qkv_proj (store bf16)"]
    assert qkv["bound"] == "tensor" and abs(qkv["tflops"] - 2.0 * S * 3 * Dh * d / 2e-3 / 1e12) < 1e-9
    assert qkv["peak"] == 1500.0                        # a step of 4 s runs under the power cap: sustained
    assert out["convert"]["bytes_per_launch"] == 6 * S * d and out["convert"]["bound"] == "hbm"
    dkdv = out["bwd_dkdv"]
    assert abs(dkdv["tflops"] - 8 * Dh * S * (S + 1) // 2 / 0.5 / 1e12) < 1e-6
    assert list(out)[0] == "bwd_dkdv"                   # sorted by time
