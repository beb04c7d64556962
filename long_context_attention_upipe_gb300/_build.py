"""In-tree build of the CUDA library (libupipe_attn.so) for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked with nvcc -shared.  No CMake.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libupipe_attn.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["api.cu", "tile_table.cu", "gemm_tc.cu", "attn_fwd_tc.cu", "attn_bwd_tc.cu", "tc_host.cu", "small.cu", "no_alloc.cu", "ring.cu", "wait_probe.cu", "mlp.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(INCLUDE, "upipe_attn.h"))
    return out


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(verbose: bool = False, extra_flags=None) -> str:
    """Compile the library if any source is newer than it; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])
    newest_src = _newest(_deps())
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= newest_src:
        return LIB
    objs = []
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = ["nvcc", *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    link = ["nvcc", "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", LIB + ".tmp", "-lcudart"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB)
