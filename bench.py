"""Benchmark of the head-chunked attention layer (forward + backward) on GB300.

One step = upipe_attn_fwd + upipe_attn_bwd of the whole layer (tile table, per-chunk QKV
projection, attention forward, output-projection accumulation; recompute, attention backward,
input and weight gradients) on one batch of synthetic seeded inputs already resident in HBM.
The default workload is the single-GPU share of an 8-way Ulysses split at 1,048,576 tokens
(4 query heads, 1 KV head, head_dim 128, hidden 4096, causal) with 4 query heads per chunk,
swept over heads_per_chunk 1, 2 and 4; `--workload llama8b_32k` selects the Llama-3.1-8B-shaped
layer at 32,768 tokens (32 / 8 heads, 8 per chunk).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Multi-GPU runs are independent replicas (weak scaling): the
layer's single-GPU share has no exchange step.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd+bwd TFLOP/s (% bf16 peak) and peak HBM GB vs heads_per_chunk"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ulysses_1m")
    ap.add_argument("--hpc", type=int, default=None, help="query heads per chunk (default: the workload's largest "
                    "swept value, 4 at 1M tokens, 8 at 32K)")
    ap.add_argument("--accum-mode", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the step's kernels one by one instead of replaying "
                    "a CUDA graph of them")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-offload", action="store_true", help="skip the leg with X and dY in pinned host memory")
    ap.add_argument("--no-mlp", action="store_true", help="skip the sequence-tiled MLP leg")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sample-tokens", type=int, default=8192,
                    help="oracle sample length (CPU legs): the first tokens of the workload as one sequence, about "
                         "10 s of fp64 work on 16 cores")
    ap.add_argument("--kernel", default=None, choices=["fwd", "recompute", "dq", "dkdv", "lse_merge", "ring", "ring_bwd"],
                    help="time one attention kernel alone at the workload's chunk shapes (for profilers); "
                         "lse_merge: the ring merge of one block into fp32 accumulators; ring: the chunk's causal "
                         "attention as the steps of a zigzag ring of --ring-p devices (all devices' shards in one "
                         "launch per step) on this GPU, timed against the direct kernel")
    ap.add_argument("--ring-p", type=int, default=4)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--dkdv-window", type=int, default=0,
                    help="work items per dK/dV tensor-memory accumulation before it is added to fp32 sums "
                         "(upipe_attn_set_dkdv_window; 0: the library default)")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------------
# CPU legs: the fp64 oracle on a bounded sample of the workload
# ----------------------------------------------------------------------------------------------

def oracle_sample(w, sample_tokens, repeats=1):
    """Time the oracle's full forward + backward on the first `sample_tokens` tokens of the
    workload (same hidden size, heads and mask); returns (seconds per sample, FLOPs per sample,
    threads)."""
    import numpy as np

    import oracle as orc
    import upipe_inputs as ui

    S = min(sample_tokens, w.S)
    X = ui.normal_bf16(S * w.d, ui.TID_X).reshape(S, w.d)
    W = ui.normal_bf16((w.Hq + 2 * w.Hkv) * w.Dh * w.d, ui.TID_WQKV, ui.W_STD).reshape(-1, w.d)
    Wo = ui.normal_bf16(w.d * w.Hq * w.Dh, ui.TID_WO, ui.W_STD).reshape(w.d, -1)
    dY = ui.normal_bf16(S * w.d, ui.TID_DY).reshape(S, w.d)
    seg = None
    if w.seg_lengths is not None:
        seg = w.segments()[:S]
    sub = ui.Workload("sample", S, w.d, w.Hq, w.Hkv, w.Dh, (w.Hq,), w.causal,
                      None if seg is None else tuple(np.bincount(seg - seg[0]).tolist()))
    t0 = time.perf_counter()
    for _ in range(repeats):
        orc.layer_forward(X, W, Wo, seg, w.Hq, w.Hkv, w.Dh, w.causal)
        orc.layer_backward(X, W, Wo, seg, dY, w.Hq, w.Hkv, w.Dh, w.causal)
    dt = (time.perf_counter() - t0) / repeats
    threads = None
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 1) for i in threadpool_info()), default=None)
    except Exception:
        pass
    if threads is None:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dt, sub.flops_fwd_bwd(), threads, S


def max_over_ranks(ms: float, device) -> float:
    """The job's time per step is its slowest replica's: MAX over the ranks of the process group
    (any backend; a single process returns `ms`)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_step: float, world: int, ms_all: float) -> float:
    """Whole-job TFLOP/s: every replica runs the full step, the job takes the slowest one's time."""
    return flops_per_step * world / (ms_all * 1e-3) / 1e12


def run_reference(args):
    """The reference arm: the oracle as it stands, timed on the host cores (rank 0 only)."""
    import upipe_inputs as ui

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = ui.workload(args.workload)
    if args.hpc is None:
        args.hpc = max(w.hpc_sweep)
    for _ in range(args.warmup):
        oracle_sample(w, args.sample_tokens)
    times = []
    flops = threads = S = None
    for _ in range(args.steps):
        dt, flops, threads, S = oracle_sample(w, args.sample_tokens)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    sample = f"oracle fp64 forward+backward on the first {S} tokens of {w.name} (same hidden size, heads, mask)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "seq_len": w.S, "heads_per_chunk": args.hpc, "sample_tokens": S},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

def measured_traffic(kernel, workload, heads):
    """DRAM bytes per launch from a committed ncu capture of this kernel, or None when there is
    none for this launch shape or the kernel's source changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        recs = json.load(f)
    rec = next((r for k, r in recs.items() if isinstance(r, dict) and k.split("@")[0] == kernel
                and r.get("workload") == workload and r.get("heads") == heads), None)
    if rec is None:
        return None
    src = os.path.join(ROOT, rec["source"])
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != rec["sha256_16"]:
            return None
    return rec["bytes_per_launch"]


def attn_kernel_flops(w, nh, kernel):
    """MMA FLOPs one launch of an attention kernel does over the visible pairs of nh heads:
    fwd / recompute: Q K^T and P V (4 Dh per pair); dq: Q K^T, dO V^T, dS K (6 Dh);
    dkdv: Q K^T, dO V^T, P^T dO, dS^T Q (8 Dh)."""
    per_pair = {"fwd": 4, "recompute": 4, "dq": 6, "dkdv": 8}[kernel] * w.Dh
    return per_pair * w.visible_pairs() * nh


GEMM_KINDS = {"qkv_proj", "o_proj", "do_proj", "dwo", "dx_proj", "dwqkv"}
ATTN_PER_PAIR = {"attn_fwd": 4, "recompute": 4, "bwd_dq": 6, "bwd_dkdv": 8}   # MMA FLOPs per visible pair / Dh
EPI_NAMES = {0: "store bf16", 1: "store fp32", 2: "fp32 C += A B^T", 3: "bf16 C += A B^T"}


def gemm_bytes(r):
    """Algorithmic HBM bytes of one GEMM launch: A and B read once, C written (and read too when
    the epilogue accumulates); split-K partials are scratch, not counted."""
    m, n, k, epi = r["m"], r["n"], r["k"], r["epilogue"]
    c = {0: 2 * m * n, 1: 4 * m * n, 2: 8 * m * n, 3: 4 * m * n}[epi]
    return 2 * m * k + 2 * n * k + c


def summarize_kernels(recs, w, peaks, step_ms):
    """Per kernel class of one step: launches, device ms, executed FLOPs -> TFLOP/s, algorithmic
    HBM bytes -> GB/s, and the roofline that bounds it (tensor for the contractions, hbm for the
    conversion / zeroing passes and for GEMMs whose bytes take longer than their FLOPs)."""
    groups = {}
    for r in recs:
        key = r["kind"] if r["kind"] not in GEMM_KINDS else f'{r["kind"]} ({EPI_NAMES[r["epilogue"]]})'
        g = groups.setdefault(key, {"kernel": key, "launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0})
        g["launches"] += 1
        g["ms"] += r["ms"]
        if r["kind"] in GEMM_KINDS:
            g["flops"] += 2.0 * r["m"] * r["n"] * r["k"]
            g["bytes"] += gemm_bytes(r)
            g["shape"] = [r["m"], r["n"], r["k"]]
        elif r["kind"] in ATTN_PER_PAIR:
            g["flops"] += ATTN_PER_PAIR[r["kind"]] * w.Dh * w.visible_pairs() * r["n"]
        elif r["kind"] == "convert":
            g["bytes"] += 6.0 * r["m"]
        elif r["kind"] == "zero":
            g["bytes"] += 4.0 * r["m"]
        elif r["kind"] == "tile_table":
            g["bytes"] += 4.0 * r["m"]
        elif r["kind"] == "h2d":
            g["bytes"] += float(r["m"])
    sustained = step_ms > 500.0
    peak_t = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak_kind = f"measured bf16 {'sustained (inside a step of ' + format(step_ms / 1e3, '.1f') + ' s)' if sustained else 'burst'}"
    out = []
    for g in groups.values():
        sec = g["ms"] * 1e-3
        t_flops = g["flops"] / (peak_t * 1e12)
        t_bytes = g["bytes"] / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if g["flops"] and t_flops >= t_bytes else ("h2d" if g["kernel"] == "h2d" else "hbm")
        e = {"kernel": g["kernel"], "launches": g["launches"], "ms": round(g["ms"], 4),
             "share": round(g["ms"] / step_ms, 4), "bound": bound}
        if "shape" in g:
            e["mnk_last"] = g["shape"]
        if g["flops"]:
            e["tflops"] = g["flops"] / sec / 1e12 if sec > 0 else None
        if g["bytes"]:
            e["gbs"] = g["bytes"] / sec / 1e9 if sec > 0 else None
            e["bytes_per_launch"] = g["bytes"] / g["launches"]
        if bound == "tensor":
            e["peak"], e["peak_kind"] = peak_t, peak_kind
            e["frac"] = e["tflops"] / peak_t
        elif bound == "h2d":   # copies on the staging stream, overlapped with the kernels
            e["share"] = None
        else:
            e["peak"], e["peak_kind"] = peaks["hbm_gbs"], "measured HBM copy bandwidth"
            e["frac"] = e["gbs"] / peaks["hbm_gbs"] if e.get("gbs") else None
        out.append(e)
    out.sort(key=lambda e: -e["ms"])
    return out


MLP_S, MLP_D, MLP_F, MLP_TILE = 131072, 4096, 14336, 8192
MLP_KINDS = {"mlp_gate_up", "mlp_down", "mlp_dact", "mlp_dwd", "mlp_dx", "mlp_dwgu"}


def mlp_flops(S, d, F):
    """Algorithmic FLOPs of the SwiGLU MLP, forward + backward: 6 S d F forward (gate/up and down
    projections), 12 S d F backward (dA, dWd, dX, dWgu); the backward's recompute of the gate/up
    projection (4 S d F) is executed but not counted."""
    return 18.0 * S * d * F


def mlp_leg(up, torch, dev, peaks, time_steps):
    """The sequence-tiled feed-forward step beside the layer: the Llama-3.1-8B MLP (hidden 4096,
    ffn 14336) over 131,072 tokens, the per-GPU sequence shard of the 1M-token sequence under an
    8-way Ulysses layout, in tiles of 8192 rows against one untiled pass: time, device peak and
    the kernels of one instrumented tiled step."""
    import gc
    import upipe_inputs as ui
    S, d, F = MLP_S, MLP_D, MLP_F
    out = {"workload": f"llama3.1-8b-mlp_S{S}_d{d}_ffn{F}_swiglu", "flops_per_step": mlp_flops(S, d, F)}

    def fill(shape, tid, std):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        ui.fill_device_bf16(t.data_ptr(), t.numel(), tid, std)
        return t

    X, Wgu, Wd, dY = fill((S, d), ui.TID_X, 1.0), fill((2 * F, d), 6, ui.W_STD), fill((d, F), 7, ui.W_STD), \
        fill((S, d), ui.TID_DY, 1.0)
    runs = []
    for T in (MLP_TILE, 0):
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        before = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        desc = up.make_mlp_desc(S, d, F, T)
        ws = torch.empty(max(up.mlp_workspace_bytes(desc, 0), up.mlp_workspace_bytes(desc, 1)), dtype=torch.uint8,
                         device=dev)
        Y, dX = torch.empty_like(X), torch.empty_like(X)
        dW = torch.empty(Wgu.shape, dtype=torch.float32, device=dev)
        dD = torch.empty(Wd.shape, dtype=torch.float32, device=dev)

        def step():
            up.mlp_fwd(desc, X, Wgu, Wd, Y, ws)
            up.mlp_bwd(desc, X, Wgu, Wd, dY, dX, dW, dD, ws)

        step()
        ms = time_steps(step, 3)
        pk = torch.cuda.max_memory_allocated(dev)
        r = {"tile_rows": T if T else S, "ms_per_step": ms, "tflops": out["flops_per_step"] / (ms * 1e-3) / 1e12,
             "workspace_gb": round(ws.numel() / 1e9, 3), "layer_peak_gb": round((pk - before) / 1e9, 3)}
        if T:
            torch.cuda.synchronize()
            up.timing_records()
            up.timing_enable(True)
            try:
                step()
                torch.cuda.synchronize()
            finally:
                up.timing_enable(False)
            recs = up.timing_records()
            kern = {}
            for rec in recs:
                k = kern.setdefault(rec["kind"], {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0})
                k["launches"] += 1
                k["ms"] += rec["ms"]
                if rec["kind"] in MLP_KINDS:
                    k["flops"] += 2.0 * rec["m"] * rec["n"] * rec["k"]
                elif rec["kind"] == "mlp_act":
                    k["bytes"] += 6.0 * rec["m"]
                elif rec["kind"] == "mlp_act_bwd":
                    k["bytes"] += 12.0 * rec["m"]
            for name, k in kern.items():
                sec = k["ms"] * 1e-3
                if k["flops"]:
                    k["tflops"] = k["flops"] / sec / 1e12
                    k["frac"] = k["tflops"] / peaks["bf16_tflops"]
                if k["bytes"]:
                    k["gbs"] = k["bytes"] / sec / 1e9
                    k["frac"] = k["gbs"] / peaks["hbm_gbs"]
                    k["bound"] = "hbm"
                else:
                    k["bound"] = "tensor"
                del k["flops"], k["bytes"]
            r["kernels"] = kern
        runs.append(r)
        del ws, Y, dX, dW, dD, step
    out["runs"] = runs
    out["peak_ratio_untiled_over_tiled"] = runs[1]["layer_peak_gb"] / max(runs[0]["layer_peak_gb"], 1e-9)
    del X, Wgu, Wd, dY
    gc.collect()
    torch.cuda.empty_cache()
    return out


def instrumented_step(up, step, w, peaks, step_ms):
    """One eager step with the library's per-launch event timing on; per-kernel summary."""
    import torch
    torch.cuda.synchronize()
    up.timing_records()          # drop anything logged before
    up.timing_enable(True)
    try:
        step()
        torch.cuda.synchronize()
    finally:
        up.timing_enable(False)
    return summarize_kernels(up.timing_records(), w, peaks, step_ms)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return

    import numpy as np
    import torch

    import __graft_entry__

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    __graft_entry__.build()
    import long_context_attention_upipe_gb300 as up
    import upipe_inputs as ui

    up.set_dkdv_window(args.dkdv_window)
    window = args.dkdv_window or up.DKDV_WINDOW_DEFAULT
    w = ui.workload(args.workload)
    if args.hpc is None:
        args.hpc = max(w.hpc_sweep)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    S, d, Hq, Hkv, Dh = w.S, w.d, w.Hq, w.Hkv, w.Dh

    def fill(shape, tid, std):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        ui.fill_device_bf16(t.data_ptr(), t.numel(), tid, std, stream=stream.cuda_stream)
        return t

    X = fill((S, d), ui.TID_X, 1.0)
    W = fill(((Hq + 2 * Hkv) * Dh, d), ui.TID_WQKV, ui.W_STD)
    Wo = fill((d, Hq * Dh), ui.TID_WO, ui.W_STD)
    dY = fill((S, d), ui.TID_DY, 1.0)
    seg = w.segments()
    seg_t = torch.from_numpy(seg).to(dev) if seg is not None else None

    def make_layer(hpc):
        desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, w.causal, args.accum_mode)
        layer = up.Layer(desc, device=dev)
        Y = torch.empty_like(X)
        lse = torch.empty(Hq, S, dtype=torch.float32, device=dev)
        dX = torch.empty_like(X)
        dW = torch.empty(W.shape, dtype=torch.float32, device=dev)
        dWo = torch.empty(Wo.shape, dtype=torch.float32, device=dev)

        def fwd_on(s):
            up.fwd(desc, X, W, Wo, seg_t, Y, lse, layer.ws_fwd, s)

        def bwd_on(s):
            up.bwd(desc, X, W, Wo, seg_t, dY, lse, dX, dW, dWo, layer.ws_bwd, s)

        def step_on(s):
            fwd_on(s)
            bwd_on(s)

        step_on.fwd, step_on.bwd = fwd_on, bwd_on

        def step():
            step_on(stream)

        return desc, layer, step, (Y, lse, dX, dW, dWo), step_on

    def graph_of(step_on):
        """The step's kernel launches captured once in a CUDA graph (same kernels, same arguments,
        no per-kernel host launch cost); returns (replay, kernels per step) or (None, reason)."""
        try:
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            n0 = up.launch_count()
            with torch.cuda.graph(g):
                step_on(torch.cuda.current_stream())
            n = up.launch_count() - n0
            torch.cuda.synchronize()
            return g, n
        except Exception as ex:  # report and fall back to launching kernel by kernel
            return None, f"{type(ex).__name__}: {ex}"[:160]

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def time_local(step, n):
        """This rank's device time per call (no process-group barrier)."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def time_steps(step, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / n

    flops = w.flops_fwd_bwd()
    peaks, peak_kind = measured_peaks()

    def chunk_kernels(hpc):
        """The four attention kernels of one chunk (hpc query heads) on seeded Q/K/V/dO."""
        g = Hq // Hkv
        kvc = max(1, hpc // g)
        cdesc = up.make_desc(S, d, hpc, kvc, Dh, hpc, w.causal)
        q = fill((hpc, S, Dh), 10, 1.0)
        k = fill((kvc, S, Dh), 11, 1.0)
        v = fill((kvc, S, Dh), 12, 1.0)
        do = fill((hpc, S, Dh), 13, 1.0)
        o = torch.empty_like(q)
        lse_c = torch.empty(hpc, S, dtype=torch.float32, device=dev)
        Dt = torch.empty(2, hpc, -(-S // 128) * 128, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        table = torch.empty(up.tile_table_bytes(cdesc), dtype=torch.uint8, device=dev)
        up.build_tile_table(cdesc, seg_t, table, stream)
        up.core_fwd(cdesc, q, k, v, seg_t, table, o, lse_c, stream)
        up.core_recompute(cdesc, q, k, v, do, lse_c, seg_t, table, o, Dt, stream)
        # dK / dV as the layer launches it: into fp32 sums (flushed in windows) for a partial KV
        # group or once a key tile's work items exceed the window, else straight to bf16
        if hpc < g or min(hpc, g) * -(-S // 128) > window:
            dk_acc = torch.zeros(k.shape, dtype=torch.float32, device=dev)
            dv_acc = torch.zeros(v.shape, dtype=torch.float32, device=dev)
            dkdv = lambda: up.core_bwd_dkdv_acc(cdesc, q, k, v, do, lse_c, Dt, seg_t, table, dk_acc, dv_acc,
                                                stream=stream)
        else:
            dkdv = lambda: up.core_bwd_dkdv(cdesc, q, k, v, do, lse_c, Dt, seg_t, table, dk, dv, stream)
        return {
            "fwd": lambda: up.core_fwd(cdesc, q, k, v, seg_t, table, o, lse_c, stream),
            "recompute": lambda: up.core_recompute(cdesc, q, k, v, do, lse_c, seg_t, table, o, Dt, stream),
            "dq": lambda: up.core_bwd_dq(cdesc, q, k, v, do, lse_c, Dt, seg_t, table, dq, stream),
            "dkdv": dkdv,
        }

    if args.kernel in ("lse_merge", "ring", "ring_bwd"):
        g = Hq // Hkv
        kvc = max(1, args.hpc // g)
        if args.kernel == "lse_merge":
            o_b = fill((args.hpc, S, Dh), 13, 1.0)
            l_b = torch.zeros(args.hpc, S, dtype=torch.float32, device=dev)
            o_acc = torch.zeros(args.hpc, S, Dh, dtype=torch.float32, device=dev)
            l_acc = torch.zeros(args.hpc, S, dtype=torch.float32, device=dev)
            f = lambda: up.lse_merge(o_b, l_b, o_acc, l_acc, None, stream)
            f()
            ms_k = time_steps(f, args.reps)
            rows = args.hpc * S
            nbytes = rows * Dh * (2 + 4 + 4) + rows * 4 * 3   # O_b, O_acc read + write; lse_b, lse_acc read + write
            gbs = nbytes / (ms_k * 1e-3) / 1e9
            print(json.dumps({"kernel": "lse_merge", "workload": w.name, "heads": args.hpc, "ms": ms_k,
                              "bytes": nbytes, "gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"]}))
            return
        # the chunk's attention as a zigzag ring of P devices, all devices' shards batched in one
        # launch per step (tables built once, outside the timing, as for the direct kernels)
        P = args.ring_p
        if S % (2 * P):
            raise SystemExit(f"S = {S} is not a multiple of 2P = {2 * P}")
        C = S // (2 * P)
        qs = fill((P, args.hpc, 2 * C, Dh), 10, 1.0)
        ks = fill((P, kvc, 2 * C, Dh), 11, 1.0)
        vs = fill((P, kvc, 2 * C, Dh), 12, 1.0)
        ring = up.Ring(up.make_ring_desc(P, C, args.hpc, kvc, Dh, w.causal), seg_t, stream=stream)
        out = (torch.empty(qs.shape, dtype=torch.float32, device=dev),
               torch.empty(qs.shape[:3], dtype=torch.float32, device=dev), torch.empty_like(qs))
        direct = chunk_kernels(args.hpc)
        if args.kernel == "ring":
            f = lambda: ring.forward(qs, ks, vs, stream, out)
            fs = lambda: ring.forward(qs, ks, vs, stream, out, per_step=True)
            fd = direct["fwd"]
            fl = attn_kernel_flops(w, args.hpc, "fwd")
        else:  # dQ, dK, dV of the ring's steps (recompute-free: the forward's O and lse are given)
            dos = fill((P, args.hpc, 2 * C, Dh), 13, 1.0)
            o, lse_r = ring.forward(qs, ks, vs, stream, out)
            f = lambda: ring.backward(qs, ks, vs, o, lse_r, dos, stream)
            fs = lambda: ring.backward(qs, ks, vs, o, lse_r, dos, stream, per_step=True)
            fd = lambda: (direct["dq"](), direct["dkdv"]())
            fl = attn_kernel_flops(w, args.hpc, "dq") + attn_kernel_flops(w, args.hpc, "dkdv")
        for g_ in (f, fs, fd):
            g_()
        ms_k = time_steps(f, args.reps)
        ms_s = time_steps(fs, args.reps)
        ms_d = time_steps(fd, args.reps)
        print(json.dumps({"kernel": args.kernel, "ring_p": P, "workload": w.name, "heads": args.hpc, "ms": ms_k,
                          "tflops": fl / (ms_k * 1e-3) / 1e12, "ms_step_calls": ms_s, "direct_ms": ms_d,
                          "ratio_to_direct": ms_k / ms_d}))
        return
    if args.kernel:
        f = chunk_kernels(args.hpc)[args.kernel]
        f()
        ms_k = time_steps(f, args.reps)
        tf = attn_kernel_flops(w, args.hpc, args.kernel) / (ms_k * 1e-3) / 1e12
        print(json.dumps({"kernel": args.kernel, "workload": w.name, "heads": args.hpc, "ms": ms_k, "tflops": tf}))
        return

    # ---------------- hpc sweep first, on a clean device: speed and peak memory vs chunk size (plus
    # the HBM-bound kernels of the chunked schedule: the fp32 accumulating projections and the
    # fp32 -> bf16 pass)
    import gc
    sweep = []
    if not args.no_sweep:   # every rank runs it (its timing takes the job's barriers); rank 0 reports
        for h in w.hpc_sweep:
            gc.collect()
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            before = torch.cuda.memory_allocated(dev)      # the inputs X, Wqkv, Wo, dY (and segments)
            torch.cuda.reset_peak_memory_stats(dev)
            dsc, lay, stp, _, stp_on = make_layer(h)
            eager = stp
            gr = None if args.no_graph else graph_of(stp_on)[0]
            if gr is not None:
                stp = gr.replay
            stp()
            t = time_steps(stp, 3 if w.S < (1 << 19) else 2)
            pk = torch.cuda.max_memory_allocated(dev)
            kern = instrumented_step(up, eager, w, peaks, t)
            sweep.append({"heads_per_chunk": h, "ms_per_step": round(t, 3),
                          "tflops": round(flops / (t * 1e-3) / 1e12, 2),
                          "peak_hbm_gb": round(pk / 1e9, 3),
                          "layer_peak_gb": round((pk - before) / 1e9, 3),
                          "workspace_gb": round((up.workspace_bytes(dsc, 0) + up.workspace_bytes(dsc, 1)) / 1e9, 3),
                          "inputs_gb": round(before / 1e9, 3),
                          "hbm_kernels": [k for k in kern if k["bound"] == "hbm"]})
            del dsc, lay, stp, gr, stp_on, eager, _  # the graph and the step closures hold the layer's workspace
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    # ---------------- CPU offload of the layer's inputs: X and dY in pinned host memory, streamed in
    # 65,536-row blocks; throughput and device peak against the resident layer at the same chunking
    offload = None
    if not args.no_offload:
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        hX = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
        hdY = torch.empty(dY.shape, dtype=dY.dtype, pin_memory=True)
        hX.copy_(X)
        hdY.copy_(dY)
        before = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        odesc = up.make_desc(S, d, Hq, Hkv, Dh, args.hpc, w.causal, args.accum_mode)
        ows = torch.empty(max(up.workspace_bytes_offload(odesc, 0), up.workspace_bytes_offload(odesc, 1)),
                          dtype=torch.uint8, device=dev)
        oY, odX = torch.empty_like(X), torch.empty_like(X)
        olse = torch.empty(Hq, S, dtype=torch.float32, device=dev)
        odW = torch.empty(W.shape, dtype=torch.float32, device=dev)
        odWo = torch.empty(Wo.shape, dtype=torch.float32, device=dev)

        n_chunks = Hq // args.hpc
        xb = X.numel() * X.element_size()
        # host -> device copy bandwidth of this machine (pinned memory, one large copy)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dst = torch.empty_like(X)
        dst.copy_(hX, non_blocking=True)
        e0.record(stream)
        dst.copy_(hX, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = xb / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del dst
        offload = {"heads_per_chunk": args.hpc, "stage_rows": 65536, "h2d_gbs_measured": round(h2d_gbs, 1),
                   "what": "upipe_attn_fwd_offload / upipe_attn_bwd_offload: host tensors staged in row blocks by the "
                           "library; device peak excludes X (and dY when it is on the host)", "runs": []}
        for name, xa, dya, h2d in (("X on host, dY on device", hX, dY, 3 * n_chunks * xb),
                                   ("X and dY on host", hX, hdY, 5 * n_chunks * xb)):
            torch.cuda.synchronize()
            torch.cuda.reset_peak_memory_stats(dev)

            def ostep():
                up.fwd_offload(odesc, xa, W, Wo, seg_t, oY, olse, ows, 0, stream)
                up.bwd_offload(odesc, xa, W, Wo, seg_t, dya, olse, odX, odW, odWo, ows, 0, stream)

            ostep()
            t_off = max_over_ranks(time_steps(ostep, 2 if w.S >= (1 << 19) else 3), dev)
            pk = torch.cuda.max_memory_allocated(dev)
            off_dev = xb if dya is dY else 2 * xb      # the device copies of X (and dY) an offloading caller lacks
            run = {"placement": name, "ms_per_step": t_off, "tflops": job_value(flops, world, t_off),
                   "device_peak_gb": round((pk - off_dev) / 1e9, 3), "h2d_bytes_per_step": h2d}
            # where the offloaded step's time goes: its kernels, with the library's event timing
            t0 = time.perf_counter()
            kern = instrumented_step(up, ostep, w, peaks, t_off)
            run["host_s_instrumented_step"] = round(time.perf_counter() - t0, 3)
            run["kernel_ms"] = {k["kernel"]: round(k["ms"], 2) for k in kern}
            run["kernel_ms_total"] = round(sum(k["ms"] for k in kern), 2)
            offload["runs"].append(run)
        del ows, oY, odX, olse, odW, odWo, hX, hdY
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    mlp = None
    if not args.no_mlp and rank == 0:
        mlp = mlp_leg(up, torch, dev, peaks, time_local)

    # ---------------- main timed run
    torch.cuda.reset_peak_memory_stats(dev)
    desc, layer, step, outs, step_on = make_layer(args.hpc)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    launch_mode, graph, per_step = "eager", None, 0
    if not args.no_graph:
        graph, per_step = graph_of(step_on)
        if graph is not None:
            launch_mode = "cuda_graph"
            timed = graph.replay
            for _ in range(max(3, args.warmup)):
                timed()
            torch.cuda.synchronize()
        else:
            launch_mode = f"eager (graph capture failed: {per_step})"
    if graph is None:
        timed = step
    sampler = ClockSampler(local)
    sampler.start()
    launches_before = up.launch_count()
    ms = time_steps(timed, args.steps)
    # our kernels launched in the timed region (graph replays launch the kernels counted at capture)
    launches = per_step * args.steps if graph is not None else up.launch_count() - launches_before
    clocks = sampler.stop()
    peak_gb = torch.cuda.max_memory_allocated(dev) / 1e9
    ms_all = max_over_ranks(ms, dev)
    value = job_value(flops, world, ms_all)
    # one more step, launched kernel by kernel with the library's per-launch event timing on: the
    # same launches as a timed step, each bracketed by CUDA events on the step's stream
    step_kernels = instrumented_step(up, step, w, peaks, ms)

    # ---------------- end to end through the C-ABI with host buffers
    # Every step uploads its X, Wqkv, Wo and dY from pinned host memory and reads Y, dX, dWqkv
    # and dWo back, all inside the timed region.  The copies run on two copy streams beside
    # the compute: dY and the next step's X / Wqkv / Wo (double-buffered) upload while the
    # forward runs, Y downloads while the backward runs, and dX / dWqkv / dWo download while
    # the next step's forward runs.  Step 0 uploads its own inputs before its forward; the last
    # step prefetches nothing.
    e2e = None
    if not args.no_e2e:
        Y, lse, dX, dW, dWo = outs

        def pin(t):
            return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)

        hX, hW, hWo, hdY = pin(X), pin(W), pin(Wo), pin(dY)
        for h, t in ((hX, X), (hW, W), (hWo, Wo), (hdY, dY)):
            h.copy_(t)
        hY, hdX, hdW, hdWo = pin(Y), pin(dX), pin(dW), pin(dWo)
        ins = [(X, W, Wo), (torch.empty_like(X), torch.empty_like(W), torch.empty_like(Wo))]
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        dy_ready, fwd_done, bwd_done = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        y_done, out_done = torch.cuda.Event(), torch.cuda.Event()

        def upload(b):
            for dst, src in zip(ins[b], (hX, hW, hWo)):
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(cin)

        def e2e_run(n):
            """n steps; returns ms per step (CUDA events on the compute stream, which waits
            for the last download before the end event)."""
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bwd_done.record(stream)
            out_done.record(stream)
            y_done.record(stream)
            cin.wait_stream(stream)
            cout.wait_stream(stream)
            with torch.cuda.stream(cin):
                upload(0)
            for k in range(n):
                b = k & 1
                Xb, Wb, Wob = ins[b]
                stream.wait_event(in_ready[b])
                stream.wait_event(y_done)             # the previous step's Y has been read back
                up.fwd(desc, Xb, Wb, Wob, seg_t, Y, lse, layer.ws_fwd, stream)
                fwd_done.record(stream)
                with torch.cuda.stream(cin):
                    cin.wait_event(bwd_done)          # the previous backward read dY and ins[1 - b]
                    dY.copy_(hdY, non_blocking=True)
                    dy_ready.record(cin)
                    if k + 1 < n:
                        upload(1 - b)
                with torch.cuda.stream(cout):
                    cout.wait_event(fwd_done)
                    hY.copy_(Y, non_blocking=True)
                    y_done.record(cout)
                stream.wait_event(dy_ready)
                stream.wait_event(out_done)           # the previous results have been read back
                up.bwd(desc, Xb, Wb, Wob, seg_t, dY, lse, dX, dW, dWo, layer.ws_bwd, stream)
                bwd_done.record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(bwd_done)
                    hdX.copy_(dX, non_blocking=True)
                    hdW.copy_(dW, non_blocking=True)
                    hdWo.copy_(dWo, non_blocking=True)
                    out_done.record(cout)
            stream.wait_event(out_done)
            e1.record(stream)
            barrier()
            return e0.elapsed_time(e1) / n

        e2e_run(1 if ms > 2000 else 2)
        n_e2e = max(2, args.steps // 4) if ms > 2000 else max(3, args.steps // 2)
        t = max_over_ranks(e2e_run(n_e2e), dev)
        h2d = sum(x.numel() * x.element_size() for x in (hX, hW, hWo, hdY))
        d2h = sum(x.numel() * x.element_size() for x in (hY, hdX, hdW, hdWo))
        e2e = {"value": job_value(flops, world, t), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t, "steps": n_e2e,
               "overlap": "dY and the next step's inputs upload during the forward; Y downloads during the "
                          "backward; dX, dWqkv, dWo download during the next forward"}
        del ins

    result = {}
    if rank == 0:
        # ---------------- the dominant kernel of the step against its roofline
        dom = max((k for k in step_kernels if k["bound"] == "tensor"), key=lambda k: k["ms"])
        traffic = measured_traffic(dom["kernel"], args.workload, args.hpc)
        roofline = {"bound": "tensor", "kernel": dom["kernel"], "achieved": dom["tflops"], "peak": dom["peak"],
                    "unit": "TFLOP/s", "frac": dom["tflops"] / dom["peak"],
                    "traffic": None if traffic is None else traffic,
                    "peak_kind": dom["peak_kind"],
                    "how": "executed MMA FLOPs of its launches in one step / their CUDA-event durations inside "
                           "that step"}

        # ---------------- CPU baseline: the oracle on a bounded sample
        cpu = None
        if not args.no_cpu and world == 1:
            dt, fl, threads, Ssamp = oracle_sample(w, args.sample_tokens)
            cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"oracle fp64 forward+backward on the first {Ssamp} tokens of {w.name}; "
                             f"{dt:.2f} s for {fl / 1e12:.4f} TFLOP",
                   # labelled extrapolation: the whole step at the sample's FLOP rate
                   "extrapolated_step_s": flops / (fl / dt),
                   "extrapolated_how": "the workload's fwd+bwd FLOPs divided by the sample's FLOP rate "
                                       "(extrapolated, not timed)"}

        if offload is not None:
            for r in offload["runs"]:
                r["time_vs_resident"] = r["ms_per_step"] / ms_all
            res = next((e for e in sweep if e["heads_per_chunk"] == args.hpc), None)
            if res is not None:
                offload["resident_device_peak_gb"] = res["peak_hbm_gb"]
        sustained = ms > 500.0
        peak_step = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        x_mb = S * d * 2 / 1e6
        result = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_all, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "seq_len": S, "hidden": d, "n_q_heads": Hq, "n_kv_heads": Hkv,
                       "head_dim": Dh, "heads_per_chunk": args.hpc, "causal": bool(w.causal),
                       "accum_mode": args.accum_mode,
                       "l2": f"inputs larger than L2 (X and dY are {x_mb:.0f} MB each); no flush",
                       "flops_per_step": flops, "parallelism": f"replicas{world}"},
            "tokens_per_s": S * world / (ms_all * 1e-3),
            "pct_bf16_peak": 100.0 * (value / world) / peak_step,
            "pct_bf16_peak_of": (f"{peak_kind} bf16 {'sustained' if sustained else 'burst'} peak "
                                 f"{peak_step} TFLOP/s ({'steps of ' + format(ms / 1e3, '.1f') + ' s run under the power cap' if sustained else 'sub-second steps'})"),
            "pct_bf16_peak_burst": 100.0 * (value / world) / peaks["bf16_tflops"],
            "peak_hbm_gb": round(peak_gb, 3),
            "roofline": roofline,
            "step_kernels": step_kernels,
            "hpc_sweep": sweep,
            "offload": offload,
            "mlp_tiled": mlp,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "launch": launch_mode,
            "clocks": clocks,
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
