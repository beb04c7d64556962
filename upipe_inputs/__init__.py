"""Seeded synthetic inputs for the head-chunked attention layer.

This module is shared by the test oracle and the CUDA path and holds none of the layer's
arithmetic: it only produces the inputs (X, Wqkv, Wo, dY, segment ids) and describes the
workload shapes.  The generator is defined in ``gen.h``; ``gen_host.c`` fills host arrays and
``gen_dev.cu`` fills device buffers with the same bits.

Tensor ids of the generator: X=0, Wqkv=1, Wo=2, dY=4, segment lengths=5.
Distributions: X ~ N(0,1), Wqkv and Wo ~ N(0, 0.02), dY ~ N(0,1), all rounded to bf16.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libupipe_gen_host.so")
_DEV_SO = os.path.join(_HERE, "libupipe_gen_dev.so")

SEED = 0x5EED
TID_X, TID_WQKV, TID_WO, TID_DY, TID_SEG = 0, 1, 2, 4, 5
W_STD = 0.02


def build(device: bool = True) -> None:
    """Compile the host fill (gcc) and, if asked, the device fill (nvcc, sm_103a)."""
    srcs = [os.path.join(_HERE, f) for f in ("gen.h", "gen_host.c")]
    if _stale(_HOST_SO, srcs):
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
             os.path.join(_HERE, "gen_host.c"), "-o", _HOST_SO, "-lm"])
    if device:
        srcs = [os.path.join(_HERE, f) for f in ("gen.h", "gen_dev.cu")]
        if _stale(_DEV_SO, srcs):
            subprocess.check_call(
                ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-fmad=false",
                 "-Xcompiler", "-fPIC", "-shared", os.path.join(_HERE, "gen_dev.cu"), "-o", _DEV_SO])


def _stale(target, srcs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in srcs)


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        build(device=False)
        lib = ctypes.CDLL(_HOST_SO)
        lib.ug_fill_normal_bf16_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                                 ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                                 ctypes.c_double]
        lib.ug_fill_rows_normal_bf16_host.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                      ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                                      ctypes.c_double, ctypes.c_double]
        lib.ug_uniform_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64]
        lib.ug_log_host.argtypes = [ctypes.c_double]
        lib.ug_log_host.restype = ctypes.c_double
        lib.ug_bf16_rne_host.argtypes = [ctypes.c_double]
        lib.ug_bf16_rne_host.restype = ctypes.c_uint16
        lib.ug_mix64_host.argtypes = [ctypes.c_uint64]
        lib.ug_mix64_host.restype = ctypes.c_uint64
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            build(device=True)
        lib = ctypes.CDLL(_DEV_SO)
        lib.ug_fill_normal_bf16_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                                   ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                                   ctypes.c_double, ctypes.c_void_p]
        lib.ug_fill_normal_bf16_device.restype = ctypes.c_int
        _dev = lib
    return _dev


def normal_bf16(n: int, tid: int, std: float = 1.0, seed: int = SEED, first: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of elements first .. first+n-1 of tensor `tid`."""
    out = np.empty(n, dtype=np.uint16)
    _host_lib().ug_fill_normal_bf16_host(out.ctypes.data, n, seed, tid, first, 0.0, std)
    return out


def normal_bf16_rows(rows, cols: int, tid: int, std: float = 1.0, seed: int = SEED) -> np.ndarray:
    """Selected rows of a row-major [*, cols] seeded tensor, as uint16 [len(rows), cols]."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, cols), dtype=np.uint16)
    _host_lib().ug_fill_rows_normal_bf16_host(out.ctypes.data, rows.ctypes.data, rows.size, cols, seed,
                                              tid, 0.0, std)
    return out


def fill_device_bf16(ptr: int, n: int, tid: int, std: float = 1.0, seed: int = SEED, first: int = 0,
                     stream: int = 0) -> None:
    """Fill n bf16 elements at device address `ptr` with the same values `normal_bf16` gives."""
    rc = _dev_lib().ug_fill_normal_bf16_device(ptr, n, seed, tid, first, 0.0, std, stream)
    if rc != 0:
        raise RuntimeError(f"device fill failed with CUDA error {rc}")


def uniforms(n: int, tid: int, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _host_lib().ug_uniform_host(out.ctypes.data, n, seed, tid)
    return out


def bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# segment ids
# ----------------------------------------------------------------------------------------------

def segments_from_lengths(lengths) -> np.ndarray:
    """Non-decreasing int32 segment ids for contiguous packed segments of the given lengths."""
    lengths = [int(x) for x in lengths]
    return np.repeat(np.arange(len(lengths), dtype=np.int32), lengths)


def loguniform_lengths(S: int, lo: int = 1024, hi: int = 32768, seed: int = SEED) -> list:
    """Packed-sequence recipe: L_k = floor(lo * (hi/lo)^U_k), U_k the k-th uniform draw of
    tensor id 5, drawn until the total reaches S; the last segment is cut to fit."""
    ratio_log2 = math.log2(hi / lo)
    out, total, k = [], 0, 0
    while total < S:
        u = float(uniforms(k + 1, TID_SEG, seed)[k])
        L = int(math.floor(lo * 2.0 ** (u * ratio_log2)))
        L = max(1, min(L, S - total))
        out.append(L)
        total += L
        k += 1
    return out


# ----------------------------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int
    d: int
    Hq: int
    Hkv: int
    Dh: int
    hpc_sweep: tuple
    causal: bool = True
    seg_lengths: tuple | None = None  # None: one segment

    @property
    def g(self):
        return self.Hq // self.Hkv

    def segments(self):
        if self.seg_lengths is None:
            return None
        return segments_from_lengths(self.seg_lengths)

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask lets through, per head."""
        lens = self.seg_lengths if self.seg_lengths is not None else (self.S,)
        if self.causal:
            return sum(L * (L + 1) // 2 for L in lens)
        return sum(L * L for L in lens)

    def flops_fwd_bwd(self) -> float:
        """Algorithmic fwd+bwd FLOPs: attention 3.5 x 4*Dh*pairs per head, projections 3 x fwd."""
        attn = 3.5 * 4.0 * self.Dh * self.visible_pairs() * self.Hq
        proj_fwd = 2.0 * self.S * self.d * (self.Hq + 2 * self.Hkv) * self.Dh + 2.0 * self.S * self.Hq * self.Dh * self.d
        return attn + 3.0 * proj_fwd


def _c3_lengths():
    return tuple(loguniform_lengths(131072))


WORKLOADS = {
    "tiny": Workload("tiny_S512_d256_h4kv2_dh64_packed300+212", 512, 256, 4, 2, 64, (2,), True, (300, 212)),
    "llama8b_32k": Workload("llama3.1-8b-attn_S32768_d4096_h32kv8_dh128_causal", 32768, 4096, 32, 8, 128, (4, 8, 32)),
    "packed_131k": None,  # filled lazily (needs the host generator)
    "ulysses_1m": Workload("ulysses8-share_S1048576_d4096_h4kv1_dh128_causal", 1048576, 4096, 4, 1, 128, (1, 2, 4)),
    "share32b_5m": Workload("32b-share_S5000000_d5120_h8kv1_dh128_causal", 5000000, 5120, 8, 1, 128, (1, 2)),
}


def workload(key: str) -> Workload:
    if key == "packed_131k" and WORKLOADS[key] is None:
        WORKLOADS[key] = Workload("llama3.1-8b-attn_S131072_packed-loguniform1k-32k_h32kv8_dh128", 131072, 4096,
                                  32, 8, 128, (8,), True, _c3_lengths())
    return WORKLOADS[key]
