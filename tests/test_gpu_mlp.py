"""The sequence-tiled SwiGLU MLP (the feed-forward step beside the layer, computed a tile of rows at a
time) against the fp64 oracle, and tiled against untiled.

Rows of an MLP are independent, so tiling changes only where the weight-gradient sums over the
sequence are cut: Y and dX must be bit-identical between tilings, dWgu and dWd equal to
rounding, and all of them within the parity bar of the oracle."""
import numpy as np
import pytest
import torch

import long_context_attention_upipe_gb300 as up
import oracle as orc
import upipe_inputs as ui
from helpers import FULL_MLP_OUT_MAX_ABS, GRAD_REL_FRO, OUT_MAX_ABS, OUT_REL_FRO, bf16_tensor, max_abs_bf16_out, rel_fro, to_f64

pytestmark = pytest.mark.gpu

TID_WGU, TID_WD = 6, 7


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()
    ui.build(device=True)


def mlp_inputs(S, d, F):
    X = ui.normal_bf16(S * d, ui.TID_X).reshape(S, d)
    Wgu = ui.normal_bf16(2 * F * d, TID_WGU, ui.W_STD).reshape(2 * F, d)
    Wd = ui.normal_bf16(d * F, TID_WD, ui.W_STD).reshape(d, F)
    dY = ui.normal_bf16(S * d, ui.TID_DY).reshape(S, d)
    return X, Wgu, Wd, dY


def run_mlp(desc, Xt, Wt, Dt, dYt):
    ws = torch.empty(max(up.mlp_workspace_bytes(desc, 0), up.mlp_workspace_bytes(desc, 1)), dtype=torch.uint8,
                     device="cuda")
    Y = torch.full_like(Xt, float("nan"))
    up.mlp_fwd(desc, Xt, Wt, Dt, Y, ws)
    dX = torch.full_like(Xt, float("nan"))
    dW = torch.full(Wt.shape, float("nan"), dtype=torch.float32, device="cuda")
    dD = torch.full(Dt.shape, float("nan"), dtype=torch.float32, device="cuda")
    up.mlp_bwd(desc, Xt, Wt, Dt, dYt, dX, dW, dD, ws)
    torch.cuda.synchronize()
    return Y, dX, dW, dD


@pytest.mark.parametrize("S,d,F,tiles", [(1000, 256, 512, (0, 128, 384)), (640, 128, 192, (0, 256)),
                                         (1, 64, 64, (0, 128))])
def test_mlp_matches_oracle_and_tilings_agree(S, d, F, tiles):
    X, Wgu, Wd, dY = mlp_inputs(S, d, F)
    Xt, Wt, Dt, dYt = (bf16_tensor(a) for a in (X, Wgu, Wd, dY))
    Y_ref = orc.mlp_forward(X, Wgu, Wd)
    dX_ref, dW_ref, dD_ref = orc.mlp_backward(X, Wgu, Wd, dY)
    first = None
    for T in tiles:
        Y, dX, dW, dD = run_mlp(up.make_mlp_desc(S, d, F, T), Xt, Wt, Dt, dYt)
        y = to_f64(Y)
        assert max_abs_bf16_out(y, Y_ref) <= OUT_MAX_ABS, (T, max_abs_bf16_out(y, Y_ref))
        assert rel_fro(y, Y_ref) <= OUT_REL_FRO, (T, rel_fro(y, Y_ref))
        assert rel_fro(to_f64(dX), dX_ref) <= GRAD_REL_FRO, (T, rel_fro(to_f64(dX), dX_ref))
        assert rel_fro(to_f64(dW), dW_ref) <= GRAD_REL_FRO, (T, rel_fro(to_f64(dW), dW_ref))
        assert rel_fro(to_f64(dD), dD_ref) <= GRAD_REL_FRO, (T, rel_fro(to_f64(dD), dD_ref))
        if first is None:
            first = (Y, dX, dW, dD)
        else:
            assert torch.equal(Y, first[0]) and torch.equal(dX, first[1])
            assert rel_fro(to_f64(dW), to_f64(first[2])) <= 1e-5 and rel_fro(to_f64(dD), to_f64(first[3])) <= 1e-5


def test_mlp_full_shape_tiled_against_oracle_and_memory():
    """The Llama-3.1-8B feed-forward shape (hidden 4096, ffn 14336) over 32,768 tokens in tiles of
    4096 rows.  Forward rows (first, tile edges, last) against the oracle; backward with dY non-zero
    on the first P rows only, so dX rows >= P are exactly zero and every gradient equals the
    oracle's on P rows.  The tiled run's device peak stays far below the untiled workspace."""
    S, d, F, T, P = 32768, 4096, 14336, 4096, 256
    dev = torch.device("cuda")

    def fill(shape, tid, std, n=None):
        t = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        ui.fill_device_bf16(t.data_ptr(), t.numel() if n is None else n, tid, std)
        return t

    Xt = fill((S, d), ui.TID_X, 1.0)
    Wt = fill((2 * F, d), TID_WGU, ui.W_STD)
    Dt = fill((d, F), TID_WD, ui.W_STD)
    dYt = fill((S, d), ui.TID_DY, 1.0, P * d)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    desc = up.make_mlp_desc(S, d, F, T)
    Y, dX, dW, dD = run_mlp(desc, Xt, Wt, Dt, dYt)
    held = torch.cuda.max_memory_allocated() - before
    untiled = up.mlp_workspace_bytes(up.make_mlp_desc(S, d, F, 0), 1)
    tiled = up.mlp_workspace_bytes(desc, 1)
    assert held <= tiled + 2 * S * d * 2 + (2 * F * d + d * F) * 4 + (64 << 20), held
    assert untiled > 7 * tiled
    rows = np.array([0, 1, T - 1, T, 2 * T + 5, S // 2, S - T - 1, S - T, S - 2, S - 1])
    Wgu = ui.normal_bf16(2 * F * d, TID_WGU, ui.W_STD).reshape(2 * F, d)
    Wd = ui.normal_bf16(d * F, TID_WD, ui.W_STD).reshape(d, F)
    Y_ref = orc.mlp_forward(ui.normal_bf16_rows(rows, d, ui.TID_X), Wgu, Wd)
    y = to_f64(Y[torch.from_numpy(rows).cuda()])
    assert rel_fro(y, Y_ref) <= OUT_REL_FRO, rel_fro(y, Y_ref)
    # the bf16-stored gate/up output and A of an exact implementation already give 0.029 here
    # (tests/test_error_budget.py)
    assert max_abs_bf16_out(y, Y_ref) <= FULL_MLP_OUT_MAX_ABS, max_abs_bf16_out(y, Y_ref)
    Xp = ui.normal_bf16_rows(np.arange(P), d, ui.TID_X)
    dYp = ui.normal_bf16(P * d, ui.TID_DY).reshape(P, d)
    dX_ref, dW_ref, dD_ref = orc.mlp_backward(Xp, Wgu, Wd, dYp)
    assert rel_fro(to_f64(dX[:P]), dX_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dX[:P]), dX_ref)
    assert not bool((dX[P:] != 0).any())
    assert rel_fro(to_f64(dW), dW_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dW), dW_ref)
    assert rel_fro(to_f64(dD), dD_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dD), dD_ref)
