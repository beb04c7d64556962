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
           "upipe_attn_core_recompute", "upipe_attn_core_bwd_dq", "upipe_attn_core_bwd_dkdv", "upipe_attn_gemm_nt",
           "upipe_attn_device_status", "upipe_attn_fwd_no_alloc", "upipe_attn_launch_count", "upipe_attn_lse_merge",
           "upipe_attn_ring_bwd_prep", "upipe_attn_accumulate", "upipe_attn_last_device_error",
           "upipe_attn_no_alloc_device_status", "upipe_attn_timing_enable", "upipe_attn_timing_collect",
           "upipe_attn_workspace_size_offload", "upipe_attn_fwd_offload", "upipe_attn_bwd_offload",
           "upipe_attn_set_wait_limit_ns", "upipe_attn_wait_probe", "upipe_mlp_workspace_size", "upipe_mlp_fwd",
           "upipe_mlp_bwd"]

# kinds of the per-launch timing records (upipe_attn_timing_collect)
KERNEL_KINDS = {0: "tile_table", 1: "qkv_proj", 2: "attn_fwd", 3: "o_proj", 4: "convert", 5: "do_proj",
                6: "recompute", 7: "dwo", 8: "bwd_dq", 9: "bwd_dkdv", 10: "dx_proj", 11: "dwqkv", 12: "zero",
                13: "mlp_gate_up", 14: "mlp_act", 15: "mlp_down", 16: "mlp_dact", 17: "mlp_act_bwd", 18: "mlp_dwd",
                19: "mlp_dx", 20: "mlp_dwgu", 21: "h2d"}


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
            "upipe_mlp_workspace_size": ([ctypes.POINTER(MlpDesc), ctypes.c_int, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_mlp_fwd": ([ctypes.POINTER(MlpDesc), P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_mlp_bwd": ([ctypes.POINTER(MlpDesc), P, P, P, P, P, P, P, P, SZ, P], ctypes.c_int),
            "upipe_attn_wait_probe": ([P, SZ, ctypes.c_int32, P], ctypes.c_int),
            "upipe_attn_workspace_size_offload": ([D, ctypes.c_int, I64, ctypes.POINTER(SZ)], ctypes.c_int),
            "upipe_attn_fwd_offload": ([D, P, P, P, P, P, P, P, SZ, I64, P], ctypes.c_int),
            "upipe_attn_bwd_offload": ([D, P, P, P, P, P, P, P, P, P, P, SZ, I64, P], ctypes.c_int),
            "upipe_attn_timing_collect": ([ctypes.POINTER(TimingRec), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
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
# Ring (P2P) context parallelism, single-GPU share: the host schedule and a one-GPU run of it
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


def _check_ring_inputs(q, k, v, P):
    if P < 1:
        raise ValueError("P must be at least 1")
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("q must be [Hq, S, Dh] and k, v [Hkv, S, Dh]")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bf16")
    Hq, S, Dh = q.shape
    Hkv = k.shape[0]
    if k.shape[1] != S or k.shape[2] != Dh or Hq % Hkv:
        raise ValueError("k, v must cover the same positions and head_dim as q, with Hq a multiple of Hkv")
    if Dh not in (64, 128):
        raise ValueError("head_dim must be 64 or 128")
    if S % (2 * P):
        raise ValueError("S must be a multiple of 2P")


def ring_attention_share(q, k, v, P: int, softmax_scale: float = 0.0, stream=None):
    """Causal attention of q [Hq, S, Dh] over k, v [Hkv, S, Dh] computed block by block as the P
    devices of a zigzag ring would, each block with upipe_attn_core_fwd on contiguous chunk copies
    and folded into per-chunk fp32 accumulators with upipe_attn_lse_merge, in ring-step order.
    One GPU runs every device's blocks in turn (there is no exchange to make).  Returns O bf16
    [Hq, S, Dh] and lse fp32 [Hq, S].  softmax_scale 0 means 1/sqrt(Dh)."""
    _check_ring_inputs(q, k, v, P)
    Hq, S, Dh = q.shape
    Hkv = k.shape[0]
    n = 2 * P
    C = S // n
    descs = {kind: make_desc(C, 64, Hq, Hkv, Dh, Hq, kind == "causal", 0, softmax_scale) for kind in ("causal", "full")}
    tables = {}
    for kind, dsc in descs.items():
        t = torch.empty(tile_table_bytes(dsc), dtype=torch.uint8, device=q.device)
        build_tile_table(dsc, None, t, stream)
        tables[kind] = t
    # each chunk once as a dense [heads, C, Dh] block: a device holds its own query chunks, and the
    # ring delivers the key/value chunks of the others in this form
    qs, ks, vs = ([x[:, c * C:(c + 1) * C].contiguous() for c in range(n)] for x in (q, k, v))
    o_acc = {c: torch.zeros(Hq, C, Dh, dtype=torch.float32, device=q.device) for c in range(n)}
    l_acc = {c: torch.full((Hq, C), float("-inf"), dtype=torch.float32, device=q.device) for c in range(n)}
    o_b = torch.empty(Hq, C, Dh, dtype=torch.bfloat16, device=q.device)
    l_b = torch.empty(Hq, C, dtype=torch.float32, device=q.device)
    o_out = {c: torch.empty(Hq, C, Dh, dtype=torch.bfloat16, device=q.device) for c in range(n)}
    order = [blk for steps in ring_block_schedule(P) for blocks in steps for blk in blocks]
    last = {qc: i for i, (qc, _, _) in enumerate(order)}   # the merge that also writes the bf16 output
    for i, (qc, kc, kind) in enumerate(order):
        core_fwd(descs[kind], qs[qc], ks[kc], vs[kc], None, tables[kind], o_b, l_b, stream)
        lse_merge(o_b, l_b, o_acc[qc], l_acc[qc], o_out[qc] if last[qc] == i else None, stream)
    O = torch.empty_like(q)
    lse = torch.empty(Hq, S, dtype=torch.float32, device=q.device)
    for c in range(n):  # placement only
        O[:, c * C:(c + 1) * C] = o_out[c]
        lse[:, c * C:(c + 1) * C] = l_acc[c]
    return O, lse


def ring_bwd_prep(O, dO, lse, D, stream=None):
    """D buffer [2][H][Sp] of the backward kernels from a chunk's final O, dO [H, S, Dh] and lse."""
    H, S, Dh = O.shape
    _check(lib().upipe_attn_ring_bwd_prep(H, S, Dh, _bf16(O), _bf16(dO), _ptr(lse), _ptr(D), _stream(stream)),
           "ring_bwd_prep")


def accumulate(src, acc, out=None, stream=None):
    """acc += src (bf16 into fp32, in place); out (bf16, optional) = the rounded sum."""
    _check(lib().upipe_attn_accumulate(src.numel(), _bf16(src), _ptr(acc), _bf16(out) if out is not None else None,
                                       _stream(stream)), "accumulate")


def ring_attention_share_backward(q, k, v, O, lse, dO, P: int, softmax_scale: float = 0.0, stream=None):
    """Gradients of causal attention (dQ [Hq, S, Dh], dK, dV [Hkv, S, Dh], bf16) computed block by
    block as the zigzag ring's devices would: each block runs upipe_attn_core_bwd_dq and _dkdv with
    its query chunk's final log-sum-exp and D = rowsum(dO * O) (upipe_attn_ring_bwd_prep), and the
    blocks' contributions are summed in fp32 per chunk (upipe_attn_accumulate), rounded once.
    O, lse: the forward's result over the whole sequence (ring_attention_share)."""
    _check_ring_inputs(q, k, v, P)
    if O.shape != q.shape or dO.shape != q.shape or tuple(lse.shape) != tuple(q.shape[:2]):
        raise ValueError("O and dO must be shaped like q, lse [Hq, S]")
    Hq, S, Dh = q.shape
    Hkv = k.shape[0]
    n = 2 * P
    C = S // n
    dev = q.device
    descs = {kind: make_desc(C, 64, Hq, Hkv, Dh, Hq, kind == "causal", 0, softmax_scale) for kind in ("causal", "full")}
    tables = {}
    for kind, dsc in descs.items():
        t = torch.empty(tile_table_bytes(dsc), dtype=torch.uint8, device=dev)
        build_tile_table(dsc, None, t, stream)
        tables[kind] = t
    cut = lambda x: [x[:, c * C:(c + 1) * C].contiguous() for c in range(n)]
    qs, ks, vs, os_, dos, ls = cut(q), cut(k), cut(v), cut(O), cut(dO), cut(lse)
    sp = -(-C // 128) * 128
    Ds = [torch.empty(2, Hq, sp, dtype=torch.float32, device=dev) for _ in range(n)]
    for c in range(n):
        ring_bwd_prep(os_[c], dos[c], ls[c], Ds[c], stream)
    f32 = lambda H: [torch.zeros(H, C, Dh, dtype=torch.float32, device=dev) for _ in range(n)]
    b16 = lambda H: [torch.empty(H, C, Dh, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    dq_acc, dk_acc, dv_acc = f32(Hq), f32(Hkv), f32(Hkv)
    dq_out, dk_out, dv_out = b16(Hq), b16(Hkv), b16(Hkv)
    dq_b = torch.empty(Hq, C, Dh, dtype=torch.bfloat16, device=dev)
    dk_b = torch.empty(Hkv, C, Dh, dtype=torch.bfloat16, device=dev)
    dv_b = torch.empty(Hkv, C, Dh, dtype=torch.bfloat16, device=dev)
    order = [blk for steps in ring_block_schedule(P) for blocks in steps for blk in blocks]
    last_q = {qc: i for i, (qc, _, _) in enumerate(order)}
    last_k = {kc: i for i, (_, kc, _) in enumerate(order)}
    for i, (qc, kc, kind) in enumerate(order):
        d, t = descs[kind], tables[kind]
        core_bwd_dq(d, qs[qc], ks[kc], vs[kc], dos[qc], ls[qc], Ds[qc], None, t, dq_b, stream)
        accumulate(dq_b, dq_acc[qc], dq_out[qc] if last_q[qc] == i else None, stream)
        core_bwd_dkdv(d, qs[qc], ks[kc], vs[kc], dos[qc], ls[qc], Ds[qc], None, t, dk_b, dv_b, stream)
        accumulate(dk_b, dk_acc[kc], dk_out[kc] if last_k[kc] == i else None, stream)
        accumulate(dv_b, dv_acc[kc], dv_out[kc] if last_k[kc] == i else None, stream)
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for c in range(n):  # placement only
        dQ[:, c * C:(c + 1) * C] = dq_out[c]
        dK[:, c * C:(c + 1) * C] = dk_out[c]
        dV[:, c * C:(c + 1) * C] = dv_out[c]
    return dQ, dK, dV


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
