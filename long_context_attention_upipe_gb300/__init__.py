"""Python binding of the head-chunked attention library (libupipe_attn.so).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.  torch
is used for device memory and streams.  There is no fallback: if the library is missing, the
import raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libupipe_attn.so")

STATUS = {0: "UPIPE_OK", 1: "UPIPE_ERR_INVALID_ARG", 2: "UPIPE_ERR_UNSUPPORTED", 3: "UPIPE_ERR_ALIGNMENT",
          4: "UPIPE_ERR_WORKSPACE_TOO_SMALL", 5: "UPIPE_ERR_SEGMENTS_NOT_CONTIGUOUS", 6: "UPIPE_ERR_CUDA",
          7: "UPIPE_ERR_DEVICE_TIMEOUT"}
UPIPE_OK = 0

EXPORTS = ["upipe_attn_status_string", "upipe_attn_last_error_string", "upipe_attn_workspace_size", "upipe_attn_tile_table_size",
           "upipe_attn_build_tile_table", "upipe_attn_fwd", "upipe_attn_bwd", "upipe_attn_core_fwd",
           "upipe_attn_core_recompute", "upipe_attn_core_bwd_dq", "upipe_attn_core_bwd_dkdv", "upipe_attn_core_bwd_dkdv_acc", "upipe_attn_gemm_nt",
           "upipe_attn_device_status", "upipe_attn_fwd_no_alloc", "upipe_attn_launch_count", "upipe_attn_lse_merge",
           "upipe_attn_ring_bwd_prep", "upipe_attn_accumulate", "upipe_attn_last_device_error",
           "upipe_attn_no_alloc_device_status", "upipe_attn_timing_enable", "upipe_attn_timing_collect",
           "upipe_attn_workspace_size_offload", "upipe_attn_fwd_offload", "upipe_attn_bwd_offload",
           "upipe_attn_set_wait_limit_ns", "upipe_attn_set_dkdv_window", "upipe_attn_wait_probe", "upipe_mlp_workspace_size", "upipe_mlp_fwd",
           "upipe_mlp_bwd", "upipe_attn_ring_tables_size", "upipe_attn_ring_build_tables", "upipe_attn_ring_fwd_step",
           "upipe_attn_ring_bwd_step", "upipe_attn_ring_fwd", "upipe_attn_ring_bwd"]

# kinds of the per-launch timing records (upipe_attn_timing_collect)
KERNEL_KINDS = {0: "tile_table", 1: "qkv_proj", 2: "attn_fwd", 3: "o_proj", 4: "convert", 5: "do_proj",
                6: "recompute", 7: "dwo", 8: "bwd_dq", 9: "bwd_dkdv", 10: "dx_proj", 11: "dwqkv", 12: "zero",
                13: "mlp_gate_up", 14: "mlp_act", 15: "mlp_down", 16: "mlp_dact", 17: "mlp_act_bwd", 18: "mlp_dwd",
                19: "mlp_dx", 20: "mlp_dwgu", 21: "h2d", 22: "ring_fwd", 23: "ring_dq", 24: "ring_dkdv"}


class Desc(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int64), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("heads_per_chunk", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("accum_mode", ctypes.c_int32), ("softmax_scale", ctypes.c_float)]


class MlpDesc(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int64), ("hidden", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("tile_rows", ctypes.c_int64)]


def make_mlp_desc(S, d, F, tile_rows=0) -> MlpDesc:
    """Sequence-tiled SwiGLU MLP: tile_rows rows per tile (multiple of 128), 0 = one tile (untiled)."""
    return MlpDesc(int(S), int(d), int(F), int(tile_rows))


def make_desc(S, d, Hq, Hkv, Dh, hpc=None, causal=True, accum_mode=0, scale=0.0) -> Desc:
    return Desc(int(S), int(d), int(Hq), int(Hkv), int(Dh), int(hpc if hpc is not None else Hq), int(bool(causal)),
                int(accum_mode), float(scale))


class RingDesc(ctypes.Structure):
    _fields_ = [("ring_size", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("chunk_len", ctypes.c_int64), ("causal", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("dev_first", ctypes.c_int32), ("dev_count", ctypes.c_int32),
                ("kv_count", ctypes.c_int32)]


def make_ring_desc(P, C, Hq, Hkv, Dh, causal=True, scale=0.0, dev_first=0, dev_count=None, kv_count=None) -> RingDesc:
    """Zigzag ring of P devices over 2PC rows (chunks of C).  By default one call runs the shares of
    all P devices with every key/value shard held in device order (kv_count = P)."""
    dev_count = P if dev_count is None else dev_count
    kv_count = P if kv_count is None else kv_count
    return RingDesc(int(P), int(Hq), int(Hkv), int(Dh), int(C), int(bool(causal)), float(scale), int(dev_first),
                    int(dev_count), int(kv_count))


class TimingRec(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("ms", ctypes.c_float), ("start_ms", ctypes.c_float)]


class UpipeError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


_lib = None


def lib():
    """The loaded library.  Raises if it was not built (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libupipe_attn.so not found at {LIB_PATH}; run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(Desc)
        sig = {
            "upipe_attn_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "upipe_attn_last_error_string": ([], ctypes.c_char_p),
            "upipe_attn_workspace_size": ([D, ctypes.c_int, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_attn_tile_table_size": ([D, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_attn_build_tile_table": ([D, P, P, SZ, ctypes.POINTER(I64), P], ctypes.c_int),
            "upipe_attn_fwd": ([D, P, P, P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_attn_bwd": ([D, P, P, P, P, P, P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_attn_core_fwd": ([D, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_core_recompute": ([D, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_core_bwd_dq": ([D, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_core_bwd_dkdv": ([D, P, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_core_bwd_dkdv_acc": ([D, P, P, P, P, P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_gemm_nt": ([I64, I64, I64, P, I64, P, I64, P, I64, P], ctypes.c_int),
            "upipe_attn_device_status": ([P, ctypes.POINTER(ctypes.c_int32), P], ctypes.c_int),
            "upipe_attn_fwd_no_alloc": ([D, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_launch_count": ([], ctypes.c_uint64),
            "upipe_attn_lse_merge": ([I64, ctypes.c_int32, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_ring_bwd_prep": ([ctypes.c_int32, I64, ctypes.c_int32, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_accumulate": ([I64, P, P, P, P], ctypes.c_int),
            "upipe_attn_last_device_error": ([P, P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
            "upipe_attn_no_alloc_device_status": ([ctypes.POINTER(ctypes.c_int32), P], ctypes.c_int),
            "upipe_attn_timing_enable": ([ctypes.c_int32], ctypes.c_int),
            "upipe_attn_set_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_int),
            "upipe_attn_set_dkdv_window": ([ctypes.c_int32], ctypes.c_int),
            "upipe_mlp_workspace_size": ([ctypes.POINTER(MlpDesc), ctypes.c_int, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_mlp_fwd": ([ctypes.POINTER(MlpDesc), P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_mlp_bwd": ([ctypes.POINTER(MlpDesc), P, P, P, P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_attn_wait_probe": ([P, SZ, ctypes.c_int32, P], ctypes.c_int),
            "upipe_attn_workspace_size_offload": ([D, ctypes.c_int, I64, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_attn_fwd_offload": ([D, P, P, P, P, P, P, P, SZ, I64, P], ctypes.c_int),
            "upipe_attn_bwd_offload": ([D, P, P, P, P, P, P, P, P, P, P, SZ, I64, P], ctypes.c_int),
            "upipe_attn_timing_collect": ([ctypes.POINTER(TimingRec), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
                                          ctypes.c_int),
            "upipe_attn_ring_tables_size": ([ctypes.POINTER(RingDesc), ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_attn_ring_build_tables": ([ctypes.POINTER(RingDesc), P, P, SZ, P], ctypes.c_int),
            "upipe_attn_ring_fwd_step": ([ctypes.POINTER(RingDesc), ctypes.c_int32, P, P, P, P, P, P, P, P, P],
                                         ctypes.c_int),
            "upipe_attn_ring_bwd_step": ([ctypes.POINTER(RingDesc), ctypes.c_int32, P, P, P, P, P, P, P, P, P, P, P,
                                          P, P, P], ctypes.c_int),
            "upipe_attn_ring_fwd": ([ctypes.POINTER(RingDesc), P, P, P, P, P, P, P, P, P], ctypes.c_int),
            "upipe_attn_ring_bwd": ([ctypes.POINTER(RingDesc), P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P],
                                    ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(code, where):
    if code != UPIPE_OK:
        if code == 6:  # UPIPE_ERR_CUDA: name the CUDA error behind it
            where = f"{where} ({lib().upipe_attn_last_error_string().decode()})"
        raise UpipeError(code, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t):
    assert t.dtype == torch.bfloat16 and t.is_contiguous(), "bf16 contiguous tensor expected"
    return _ptr(t)


def workspace_bytes(desc: Desc, pass_: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().upipe_attn_workspace_size(ctypes.byref(desc), pass_, ctypes.byref(n)), "workspace_size")
    return n.value


def tile_table_bytes(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().upipe_attn_tile_table_size(ctypes.byref(desc), ctypes.byref(n)), "tile_table_size")
    return n.value


def build_tile_table(desc: Desc, seg, table, stream=None, counts=False):
    """Build the skip table into `table` (device uint8).  counts=True also returns the visited
    tile pairs per head (n_partial, n_full), read back by the library (synchronises the stream)."""
    out = (ctypes.c_int64 * 2)() if counts else None
    _check(lib().upipe_attn_build_tile_table(ctypes.byref(desc), _ptr(seg), _ptr(table), table.numel() * table.element_size(),
                                             out, _stream(stream)), "build_tile_table")
    return (int(out[0]), int(out[1])) if counts else None


def device_status(buf, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().upipe_attn_device_status(_ptr(buf), ctypes.byref(code), _stream(stream)), "device_status")
    return code.value


def last_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().upipe_attn_last_device_error(_ptr(ws), _stream(stream), ctypes.byref(code)), "last_device_error")
    return code.value


def no_alloc_device_status(stream=None) -> int:
    """Error word of the allocation-free forward's own workspace array (current device)."""
    code = ctypes.c_int32(0)
    _check(lib().upipe_attn_no_alloc_device_status(ctypes.byref(code), _stream(stream)), "no_alloc_device_status")
    return code.value


def timing_enable(on: bool = True):
    """Log every kernel launch of upipe_attn_fwd / _bwd with CUDA events (not during graph capture)."""
    _check(lib().upipe_attn_timing_enable(int(bool(on))), "timing_enable")


def timing_records(cap: int = 1 << 16):
    """Collect the logged launches (waits for them), clearing the log; returns a list of dicts."""
    buf = (TimingRec * cap)()
    n = ctypes.c_int32(0)
    _check(lib().upipe_attn_timing_collect(buf, cap, ctypes.byref(n)), "timing_collect")
    return [{"kind": KERNEL_KINDS.get(r.kind, r.kind), "epilogue": r.epilogue, "split_k": r.split_k,
             "chunk": r.chunk, "m": r.m, "n": r.n, "k": r.k, "ms": r.ms, "start_ms": r.start_ms}
            for r in buf[:min(n.value, cap)]]


def set_wait_limit_ns(ns: int):
    """Limit of the kernels' bounded device waits (0: the default 4 s)."""
    _check(lib().upipe_attn_set_wait_limit_ns(int(ns)), "set_wait_limit_ns")


DKDV_WINDOW_DEFAULT = 4096   # work items per dK / dV accumulation before a flush (upipe_attn_set_dkdv_window)


def set_dkdv_window(items: int):
    """Work items per dK/dV tensor-memory accumulation before it is added to fp32 sums (0: 4096)."""
    _check(lib().upipe_attn_set_dkdv_window(int(items)), "set_dkdv_window")


def wait_probe(buf, arrive: bool, stream=None):
    """One bounded wait on a barrier nothing completes (arrive=False) or one already completed."""
    _check(lib().upipe_attn_wait_probe(_ptr(buf), buf.numel() * buf.element_size(), int(bool(arrive)),
                                       _stream(stream)), "wait_probe")


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib().upipe_attn_launch_count())


def fwd(desc: Desc, X, Wqkv, Wo, seg, Y, lse, ws, stream=None):
    _check(lib().upipe_attn_fwd(ctypes.byref(desc), _bf16(X), _bf16(Wqkv), _bf16(Wo), _ptr(seg), _bf16(Y), _ptr(lse),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "fwd")


def bwd(desc: Desc, X, Wqkv, Wo, seg, dY, lse, dX, dWqkv, dWo, ws, stream=None):
    _check(lib().upipe_attn_bwd(ctypes.byref(desc), _bf16(X), _bf16(Wqkv), _bf16(Wo), _ptr(seg), _bf16(dY), _ptr(lse),
                                _bf16(dX), _ptr(dWqkv), _ptr(dWo), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(stream)), "bwd")


def workspace_bytes_offload(desc: Desc, pass_: int, stage_rows: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().upipe_attn_workspace_size_offload(ctypes.byref(desc), pass_, stage_rows, ctypes.byref(n)),
           "workspace_size_offload")
    return n.value


def _host_bf16(t):
    """A bf16 tensor the offloaded calls stage from pinned host memory, or read in place on the device."""
    assert t.dtype == torch.bfloat16 and t.is_contiguous() and (t.is_cuda or t.is_pinned()), \
        "pinned host or device bf16 contiguous tensor expected"
    return _ptr(t)


def fwd_offload(desc: Desc, X_host, Wqkv, Wo, seg, Y, lse, ws, stage_rows=0, stream=None):
    """Forward with X in pinned host memory (or on the device), staged stage_rows rows at a time."""
    _check(lib().upipe_attn_fwd_offload(ctypes.byref(desc), _host_bf16(X_host), _bf16(Wqkv), _bf16(Wo), _ptr(seg),
                                        _bf16(Y), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), stage_rows,
                                        _stream(stream)), "fwd_offload")


def bwd_offload(desc: Desc, X_host, Wqkv, Wo, seg, dY_host, lse, dX, dWqkv, dWo, ws, stage_rows=0, stream=None):
    """Backward with X and / or dY in pinned host memory (each may also be on the device)."""
    _check(lib().upipe_attn_bwd_offload(ctypes.byref(desc), _host_bf16(X_host), _bf16(Wqkv), _bf16(Wo), _ptr(seg),
                                        _host_bf16(dY_host), _ptr(lse), _bf16(dX), _ptr(dWqkv), _ptr(dWo), _ptr(ws),
                                        ws.numel() * ws.element_size(), stage_rows, _stream(stream)), "bwd_offload")


def mlp_workspace_bytes(desc: MlpDesc, pass_: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().upipe_mlp_workspace_size(ctypes.byref(desc), pass_, ctypes.byref(n)), "mlp_workspace_size")
    return n.value


def mlp_fwd(desc: MlpDesc, X, Wgu, Wd, Y, ws, stream=None):
    _check(lib().upipe_mlp_fwd(ctypes.byref(desc), _bf16(X), _bf16(Wgu), _bf16(Wd), _bf16(Y), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "mlp_fwd")


def mlp_bwd(desc: MlpDesc, X, Wgu, Wd, dY, dX, dWgu, dWd, ws, stream=None):
    _check(lib().upipe_mlp_bwd(ctypes.byref(desc), _bf16(X), _bf16(Wgu), _bf16(Wd), _bf16(dY), _bf16(dX), _ptr(dWgu),
                               _ptr(dWd), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "mlp_bwd")


def core_fwd(desc: Desc, q, k, v, seg, table, o, lse, stream=None):
    _check(lib().upipe_attn_core_fwd(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _ptr(seg), _ptr(table), _bf16(o),
                                     _ptr(lse), _stream(stream)), "core_fwd")


def core_recompute(desc: Desc, q, k, v, dO, lse, seg, table, o, D, stream=None):
    _check(lib().upipe_attn_core_recompute(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _bf16(dO), _ptr(lse),
                                           _ptr(seg), _ptr(table), _bf16(o), _ptr(D), _stream(stream)), "core_recompute")


def core_bwd_dq(desc: Desc, q, k, v, dO, lse, D, seg, table, dq, stream=None):
    _check(lib().upipe_attn_core_bwd_dq(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _bf16(dO), _ptr(lse), _ptr(D),
                                        _ptr(seg), _ptr(table), _bf16(dq), _stream(stream)), "core_bwd_dq")


def core_bwd_dkdv(desc: Desc, q, k, v, dO, lse, D, seg, table, dk, dv, stream=None):
    _check(lib().upipe_attn_core_bwd_dkdv(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _bf16(dO), _ptr(lse),
                                          _ptr(D), _ptr(seg), _ptr(table), _bf16(dk), _bf16(dv), _stream(stream)),
           "core_bwd_dkdv")


def core_bwd_dkdv_acc(desc: Desc, q, k, v, dO, lse, D, seg, table, dk_acc, dv_acc, dk=None, dv=None, stream=None):
    """dK, dV added to the fp32 sums dk_acc, dv_acc [Hkv, S, Dh] (flushed in windows); dk, dv: their
    bf16 rounding, or None."""
    _check(lib().upipe_attn_core_bwd_dkdv_acc(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _bf16(dO), _ptr(lse),
                                              _ptr(D), _ptr(seg), _ptr(table), _ptr(dk_acc), _ptr(dv_acc),
                                              None if dk is None else _bf16(dk), None if dv is None else _bf16(dv),
                                              _stream(stream)),
           "core_bwd_dkdv_acc")


def core_bwd(desc: Desc, q, k, v, dO, lse, seg, table, dq, dk, dv, stream=None):
    """recompute -> dq -> dkdv, with O and D in temporary torch buffers."""
    H, S = lse.shape
    o = torch.empty_like(q)
    D = torch.empty(2, H, -(-S // 128) * 128, dtype=torch.float32, device=q.device)
    core_recompute(desc, q, k, v, dO, lse, seg, table, o, D, stream)
    core_bwd_dq(desc, q, k, v, dO, lse, D, seg, table, dq, stream)
    core_bwd_dkdv(desc, q, k, v, dO, lse, D, seg, table, dk, dv, stream)
    return o, D


def gemm_nt(A, B, C, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check(lib().upipe_attn_gemm_nt(M, N, K, _bf16(A), A.stride(0), _bf16(B), B.stride(0), _ptr(C), C.stride(0),
                                    _stream(stream)), "gemm_nt")


def lse_merge(O_b, lse_b, O_acc, lse_acc, O_out=None, stream=None):
    """Fold a block's attention result (O_b bf16 [..., Dh], lse_b fp32 [...]) into the fp32
    accumulator (O_acc, lse_acc) in place; O_out (bf16, optional) receives the merged O."""
    Dh = O_b.shape[-1]
    rows = lse_b.numel()
    _check(lib().upipe_attn_lse_merge(rows, Dh, _bf16(O_b), _ptr(lse_b), _ptr(O_acc), _ptr(lse_acc),
                                      _bf16(O_out) if O_out is not None else None, _stream(stream)), "lse_merge")


# ------------------------------------------------------------------------------------------------
# Ring (P2P) context parallelism, single-GPU share: one C-ABI call per ring step
# ------------------------------------------------------------------------------------------------

def zigzag_chunks(P: int):
    """Causal load balancing for a ring of P devices: the sequence is cut into 2P equal chunks
    and device r holds chunks r and 2P - 1 - r, so every device owns one early and one late chunk
    and does the same number of block computations (the ring strategy needs explicit load
    balancing because later positions look back over more keys)."""
    return [(r, 2 * P - 1 - r) for r in range(P)]


def ring_block_schedule(P: int):
    """For each device r and ring step s (the key/value chunks of device (r - s) mod P visit r):
    the blocks (query chunk, key chunk, "causal" | "full") that r computes; key chunks after the
    query chunk are skipped."""
    chunks = zigzag_chunks(P)
    sched = []
    for r in range(P):
        steps = []
        for s in range(P):
            src = (r - s) % P
            blocks = []
            for qc in chunks[r]:
                for kc in chunks[src]:
                    if kc < qc:
                        blocks.append((qc, kc, "full"))
                    elif kc == qc:
                        blocks.append((qc, kc, "causal"))
            steps.append(blocks)
        sched.append(steps)
    return sched


def zigzag_positions(P: int, C: int, r: int) -> torch.Tensor:
    """Sequence positions of the 2C local rows of ring device r (its chunks r and 2P - 1 - r)."""
    a, b = zigzag_chunks(P)[r]
    return torch.cat([torch.arange(a * C, (a + 1) * C), torch.arange(b * C, (b + 1) * C)])


def to_zigzag(x, P: int):
    """[H, S, ...] in sequence order -> [P, H, 2S/(2P), ...] device shards (the data loader's
    one-time reordering for causal load balancing; not part of the ring steps)."""
    C = x.shape[1] // (2 * P)
    idx = torch.stack([zigzag_positions(P, C, r) for r in range(P)]).to(x.device)
    return torch.stack([x.index_select(1, idx[r]) for r in range(P)])


def from_zigzag(xs, P: int):
    """Inverse of to_zigzag: [P, H, 2C, ...] shards -> [H, 2PC, ...] in sequence order."""
    C = xs.shape[2] // 2
    out = torch.empty((xs.shape[1], 2 * P * C) + tuple(xs.shape[3:]), dtype=xs.dtype, device=xs.device)
    for r in range(P):
        out[:, zigzag_positions(P, C, r).to(xs.device)] = xs[r]
    return out


def ring_tables_bytes(desc: RingDesc) -> int:
    n = ctypes.c_size_t()
    _check(lib().upipe_attn_ring_tables_size(ctypes.byref(desc), ctypes.byref(n)), "ring_tables_size")
    return n.value


def ring_build_tables(desc: RingDesc, seg, tables, stream=None):
    """The P per-step tile tables (seg: None or int32 [2PC] in sequence order)."""
    _check(lib().upipe_attn_ring_build_tables(ctypes.byref(desc), _ptr(seg), _ptr(tables), tables.numel(),
                                              _stream(stream)), "ring_build_tables")


def ring_fwd_step(desc: RingDesc, step: int, q, k, v, seg, tables, o_acc, lse, o=None, stream=None):
    """One forward ring step (upipe_attn_ring_fwd_step): q [dev_count, Hq, 2C, Dh], k, v [kv_count,
    Hkv, 2C, Dh] bf16; o_acc fp32 like q, lse fp32 [dev_count, Hq, 2C]; o bf16 like q or None."""
    _check(lib().upipe_attn_ring_fwd_step(ctypes.byref(desc), int(step), _bf16(q), _bf16(k), _bf16(v), _ptr(seg),
                                          _ptr(tables), _ptr(o_acc), _ptr(lse), _bf16(o) if o is not None else None,
                                          _stream(stream)), "ring_fwd_step")


def ring_bwd_step(desc: RingDesc, step: int, q, k, v, dO, D, seg, tables, dq_acc, dk_acc, dv_acc, dq=None, dk=None,
                  dv=None, stream=None):
    """One backward ring step (upipe_attn_ring_bwd_step): dQ, dK, dV of the step's blocks folded
    into the fp32 sums (dq_acc like q, dk_acc / dv_acc like k); dq, dk, dv bf16 or None."""
    opt = lambda t: _bf16(t) if t is not None else None
    _check(lib().upipe_attn_ring_bwd_step(ctypes.byref(desc), int(step), _bf16(q), _bf16(k), _bf16(v), _bf16(dO),
                                          _ptr(D), _ptr(seg), _ptr(tables), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc),
                                          opt(dq), opt(dk), opt(dv), _stream(stream)), "ring_bwd_step")


def ring_fwd(desc: RingDesc, q, k, v, seg, tables, o_acc, lse, o=None, stream=None):
    """All P forward steps in one call (upipe_attn_ring_fwd: consecutive steps overlap)."""
    _check(lib().upipe_attn_ring_fwd(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _ptr(seg), _ptr(tables),
                                     _ptr(o_acc), _ptr(lse), _bf16(o) if o is not None else None, _stream(stream)),
           "ring_fwd")


def ring_bwd(desc: RingDesc, q, k, v, o, dO, lse, seg, tables, D, dq_acc, dk_acc, dv_acc, dq=None, dk=None, dv=None,
             stream=None):
    """D from the final o, dO, lse, then all P backward steps (upipe_attn_ring_bwd)."""
    opt = lambda t: _bf16(t) if t is not None else None
    _check(lib().upipe_attn_ring_bwd(ctypes.byref(desc), _bf16(q), _bf16(k), _bf16(v), _bf16(o), _bf16(dO), _ptr(lse),
                                     _ptr(seg), _ptr(tables), _ptr(D), _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc),
                                     opt(dq), opt(dk), opt(dv), _stream(stream)), "ring_bwd")


def ring_bwd_prep(O, dO, lse, D, stream=None):
    """D buffer [2][H][Sp] of the backward kernels from the final O, dO [H, S, Dh] and lse [H, S]."""
    H, S, Dh = O.shape
    _check(lib().upipe_attn_ring_bwd_prep(H, S, Dh, _bf16(O), _bf16(dO), _ptr(lse), _ptr(D), _stream(stream)),
           "ring_bwd_prep")


def accumulate(src, acc, out=None, stream=None):
    """acc += src (bf16 into fp32, in place); out (bf16, optional) = the rounded sum."""
    _check(lib().upipe_attn_accumulate(src.numel(), _bf16(src), _ptr(acc), _bf16(out) if out is not None else None,
                                       _stream(stream)), "accumulate")


class Ring:
    """The single-GPU share of a zigzag ring: the descriptor, its per-step tables (built once per
    segment layout) and the P forward / backward step calls.  Shards: q [dev_count, Hq, 2C, Dh],
    k, v [kv_count, Hkv, 2C, Dh] bf16 (to_zigzag gives them from sequence order)."""

    def __init__(self, desc: RingDesc, seg=None, device="cuda", stream=None):
        self.desc = desc
        self.seg = seg
        self.tables = torch.empty(ring_tables_bytes(desc), dtype=torch.uint8, device=device)
        ring_build_tables(desc, seg, self.tables, stream)

    def forward(self, q, k, v, stream=None, out=None, per_step=False):
        """All P steps (one call, consecutive steps overlapping; per_step: P separate step calls);
        returns (o bf16 like q, lse fp32 [dev_count, Hq, 2C])."""
        d = self.desc
        n, S = d.dev_count, 2 * d.chunk_len
        if out is None:
            out = (torch.empty(n, d.n_q_heads, S, d.head_dim, dtype=torch.float32, device=q.device),
                   torch.empty(n, d.n_q_heads, S, dtype=torch.float32, device=q.device), torch.empty_like(q))
        o_acc, lse, o = out
        if per_step:
            for s in range(d.ring_size):
                ring_fwd_step(d, s, q, k, v, self.seg, self.tables, o_acc, lse, o, stream)
        else:
            ring_fwd(d, q, k, v, self.seg, self.tables, o_acc, lse, o, stream)
        return o, lse

    def backward(self, q, k, v, o, lse, dO, stream=None, per_step=False):
        """D from the final o, dO, lse, then the P steps (one call, or P step calls with per_step);
        returns dq, dk, dv (bf16)."""
        d = self.desc
        n, S, Dh = d.dev_count, 2 * d.chunk_len, d.head_dim
        H = n * d.n_q_heads
        sp = -(-S // 128) * 128
        D = torch.empty(2, H, sp, dtype=torch.float32, device=q.device)
        dq_acc = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        dk_acc = torch.empty(k.shape, dtype=torch.float32, device=q.device)
        dv_acc = torch.empty(v.shape, dtype=torch.float32, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if per_step:
            ring_bwd_prep(o.view(H, S, Dh), dO.view(H, S, Dh), lse.view(H, S), D, stream)
            for s in range(d.ring_size):
                ring_bwd_step(d, s, q, k, v, dO, D, self.seg, self.tables, dq_acc, dk_acc, dv_acc, dq, dk, dv, stream)
        else:
            ring_bwd(d, q, k, v, o, dO, lse, self.seg, self.tables, D, dq_acc, dk_acc, dv_acc, dq, dk, dv, stream)
        return dq, dk, dv


class Layer:
    """Convenience wrapper: owns the workspaces for one descriptor (allocated with torch)."""

    def __init__(self, desc: Desc, device="cuda"):
        self.desc = desc
        self.ws_fwd = torch.empty(workspace_bytes(desc, 0), dtype=torch.uint8, device=device)
        self.ws_bwd = torch.empty(workspace_bytes(desc, 1), dtype=torch.uint8, device=device)

    def forward(self, X, Wqkv, Wo, seg=None):
        S, d = X.shape
        Y = torch.empty_like(X)
        lse = torch.empty(self.desc.n_q_heads, S, dtype=torch.float32, device=X.device)
        fwd(self.desc, X, Wqkv, Wo, seg, Y, lse, self.ws_fwd)
        return Y, lse

    def backward(self, X, Wqkv, Wo, seg, dY, lse):
        dX = torch.empty_like(X)
        dWqkv = torch.empty(Wqkv.shape, dtype=torch.float32, device=X.device)
        dWo = torch.empty(Wo.shape, dtype=torch.float32, device=X.device)
        bwd(self.desc, X, Wqkv, Wo, seg, dY, lse, dX, dWqkv, dWo, self.ws_bwd)
        return dX, dWqkv, dWo
