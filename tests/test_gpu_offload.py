"""CPU offload of the layer's inputs: X and dY in pinned host memory, staged in row blocks.

The offloaded calls must give the regular calls' Y, lse and dX bit for bit (the same kernels see
the same values; only the Q/K/V and dO projections run block by block over the rows), and the
weight gradients to rounding (their sums over the sequence are cut at the blocks), and both must
match the oracle at the parity bar.  Small stage_rows force many blocks, including a ragged
last block, so the double-buffered copy pipeline turns over several times per pass."""
import numpy as np
import pytest
import torch

import long_context_attention_upipe_gb300 as up
import oracle as orc
import upipe_inputs as ui
from helpers import GRAD_REL_FRO, OUT_MAX_ABS, OUT_REL_FRO, bf16_tensor, layer_inputs, max_abs, max_abs_bf16_out, rel_fro, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()
    ui.build(device=True)


def pinned(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


CASES = [
    # S, d, Hq, Hkv, Dh, segment lengths, hpc, accum_mode, stage_rows
    (1000, 256, 8, 2, 128, [250, 1, 600, 149], 4, 0, 128),   # 8 blocks, the last of 104 rows
    (1000, 256, 8, 2, 128, [250, 1, 600, 149], 1, 0, 256),   # partial KV groups: dK/dV summed over chunks
    (1000, 256, 8, 2, 128, [250, 1, 600, 149], 2, 1, 384),   # bf16 in-place sums
    (512, 256, 4, 2, 64, [300, 212], 2, 0, 0),                # the default stage: one block
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c[0]}_hpc{c[6]}_acc{c[7]}_rows{c[8]}")
def test_offload_matches_regular_and_oracle(case):
    S, d, Hq, Hkv, Dh, segs, hpc, accum, stage_rows = case
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs)
    seg_t = torch.from_numpy(seg).cuda()
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, True, accum)
    layer = up.Layer(desc)
    Y_ref, lse_ref = layer.forward(Xt, Wt, Wot, seg_t)
    dX_ref, dW_ref, dWo_ref = layer.backward(Xt, Wt, Wot, seg_t, dYt, lse_ref)

    hX, hdY = pinned(Xt.cpu()), pinned(dYt.cpu())
    ws = torch.empty(max(up.workspace_bytes_offload(desc, 0, stage_rows), up.workspace_bytes_offload(desc, 1, stage_rows)),
                     dtype=torch.uint8, device="cuda")
    Y = torch.full_like(Xt, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    up.fwd_offload(desc, hX, Wt, Wot, seg_t, Y, lse, ws, stage_rows)
    assert up.device_status(ws) == 0
    dX = torch.full_like(Xt, float("nan"))
    dW = torch.full_like(dW_ref, float("nan"))
    dWo = torch.full_like(dWo_ref, float("nan"))
    up.bwd_offload(desc, hX, Wt, Wot, seg_t, hdY, lse, dX, dW, dWo, ws, stage_rows)
    torch.cuda.synchronize()
    assert up.device_status(ws) == 0
    assert torch.equal(Y, Y_ref) and torch.equal(lse, lse_ref) and torch.equal(dX, dX_ref)
    assert rel_fro(to_f64(dW), to_f64(dW_ref)) <= 1e-5
    assert rel_fro(to_f64(dWo), to_f64(dWo_ref)) <= 1e-5
    # and against the oracle
    Yo, Lo = orc.layer_forward(X, W, Wo, seg, Hq, Hkv, Dh, True)
    dXo, dWq, dWoo = orc.layer_backward(X, W, Wo, seg, dY, Hq, Hkv, Dh, True)
    assert max_abs_bf16_out(to_f64(Y), Yo) <= OUT_MAX_ABS and rel_fro(to_f64(Y), Yo) <= OUT_REL_FRO
    assert max_abs(to_f64(lse), Lo) <= 1e-3
    assert rel_fro(to_f64(dX), dXo) <= GRAD_REL_FRO
    assert rel_fro(to_f64(dW), dWq) <= GRAD_REL_FRO and rel_fro(to_f64(dWo), dWoo) <= GRAD_REL_FRO


@pytest.mark.parametrize("x_host,dy_host", [(True, False), (False, True)])
def test_offload_with_one_tensor_on_the_device(x_host, dy_host):
    """A training stack offloads the block input X while dY, produced during the backward, stays
    on the device: each tensor is staged only if it is in host memory."""
    S, d, Hq, Hkv, Dh, hpc, stage_rows = 1000, 256, 8, 2, 128, 2, 256
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, True)
    layer = up.Layer(desc)
    Y_ref, lse_ref = layer.forward(Xt, Wt, Wot)
    dX_ref, dW_ref, dWo_ref = layer.backward(Xt, Wt, Wot, None, dYt, lse_ref)
    Xa = pinned(Xt.cpu()) if x_host else Xt
    dYa = pinned(dYt.cpu()) if dy_host else dYt
    ws = torch.empty(up.workspace_bytes_offload(desc, 1, stage_rows), dtype=torch.uint8, device="cuda")
    Y = torch.empty_like(Xt); lse = torch.empty_like(lse_ref)
    up.fwd_offload(desc, Xa, Wt, Wot, None, Y, lse, ws, stage_rows)
    dX = torch.empty_like(Xt); dW = torch.empty_like(dW_ref); dWo = torch.empty_like(dWo_ref)
    up.bwd_offload(desc, Xa, Wt, Wot, None, dYa, lse, dX, dW, dWo, ws, stage_rows)
    torch.cuda.synchronize()
    assert up.device_status(ws) == 0
    assert torch.equal(Y, Y_ref) and torch.equal(lse, lse_ref) and torch.equal(dX, dX_ref)
    assert rel_fro(to_f64(dW), to_f64(dW_ref)) <= 1e-5 and rel_fro(to_f64(dWo), to_f64(dWo_ref)) <= 1e-5


def test_offload_rejects_pageable_host_memory():
    S, d, Hq, Hkv, Dh = 256, 128, 2, 1, 64
    X, W, Wo, _ = layer_inputs(S, d, Hq, Hkv, Dh, dy=False)
    desc = up.make_desc(S, d, Hq, Hkv, Dh, 1, True)
    Xh = bf16_tensor(X, device="cpu")                  # pageable
    ws = torch.empty(up.workspace_bytes_offload(desc, 0), dtype=torch.uint8, device="cuda")
    Y = torch.empty(S, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    n0 = up.launch_count()
    rc = up.lib().upipe_attn_fwd_offload(up.ctypes.byref(desc), up._ptr(Xh), up._ptr(bf16_tensor(W)), up._ptr(bf16_tensor(Wo)),
                                         None, up._ptr(Y), up._ptr(lse), up._ptr(ws), ws.numel(), 0, None)
    assert rc == 1 and up.launch_count() == n0


def test_offload_step_overlaps_and_replays_from_a_cuda_graph():
    """The copy stream forks from and joins the caller's stream with events, so an offloaded step
    can be captured in a CUDA graph; its replays reproduce the eager results bit for bit."""
    S, d, Hq, Hkv, Dh, hpc, stage_rows = 768, 256, 4, 1, 128, 2, 128
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    hX, hdY = pinned(Xt.cpu()), pinned(dYt.cpu())
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, True)
    ws = torch.empty(up.workspace_bytes_offload(desc, 1, stage_rows), dtype=torch.uint8, device="cuda")
    Y = torch.empty_like(Xt); lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    dX = torch.empty_like(Xt); dW = torch.empty(Wt.shape, dtype=torch.float32, device="cuda")
    dWo = torch.empty(Wot.shape, dtype=torch.float32, device="cuda")

    def step(s):
        up.fwd_offload(desc, hX, Wt, Wot, None, Y, lse, ws, stage_rows, s)
        up.bwd_offload(desc, hX, Wt, Wot, None, hdY, lse, dX, dW, dWo, ws, stage_rows, s)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [t.clone() for t in (Y, lse, dX, dW, dWo)]
    for t in (Y, lse, dX, dW, dWo):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for got, want in zip((Y, lse, dX, dW, dWo), eager):
        assert torch.equal(got, want)
