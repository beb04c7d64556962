"""Ring (P2P) context parallelism, single-GPU share: the log-sum-exp merge kernel against the
oracle's merge, and the zigzag ring's blocks (upipe_attn_core_fwd per block, merged in ring order)
against causal attention over the whole sequence."""
import numpy as np
import pytest
import torch

import long_context_attention_upipe_gb300 as up
import oracle as orc
import upipe_inputs as ui
from helpers import (GRAD_REL_FRO, OUT_MAX_ABS, OUT_REL_FRO, bf16_tensor, max_abs, max_abs_bf16_out, qkv_inputs, rel_fro,
                     to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()
    ui.build(device=True)


@pytest.mark.parametrize("rows,Dh", [(1, 64), (1000, 128), (4097, 64), (8 * 4096, 128)])
def test_lse_merge_kernel_matches_oracle(rows, Dh):
    Oa = ui.bf16_to_f64(ui.normal_bf16(rows * Dh, 40)).reshape(rows, Dh)            # fp32-exact values
    La = ui.bf16_to_f64(ui.normal_bf16(rows, 41, 3.0))
    Ob_bits = ui.normal_bf16(rows * Dh, 42).reshape(rows, Dh)
    Lb = ui.bf16_to_f64(ui.normal_bf16(rows, 43, 3.0))
    La[::7] = -np.inf          # accumulator that has seen no key yet
    Lb[3::11] = -np.inf        # block row that sees no key
    Oa_dev = torch.from_numpy(Oa.astype(np.float32)).cuda()
    La_dev = torch.from_numpy(La.astype(np.float32)).cuda()
    Ob_dev = bf16_tensor(Ob_bits)
    Lb_dev = torch.from_numpy(Lb.astype(np.float32)).cuda()
    out = torch.empty(rows, Dh, dtype=torch.bfloat16, device="cuda")
    up.lse_merge(Ob_dev, Lb_dev, Oa_dev, La_dev, out)
    torch.cuda.synchronize()
    O_ref, L_ref = orc.lse_merge(Oa, La, ui.bf16_to_f64(Ob_bits), Lb)
    got_L = La_dev.cpu().double().numpy()
    np.testing.assert_array_equal(np.isneginf(got_L), np.isneginf(L_ref))
    fin = np.isfinite(L_ref)
    assert max_abs(got_L[fin], L_ref[fin]) <= 1e-5 * max(1.0, np.abs(L_ref[fin]).max())
    got_O = Oa_dev.cpu().double().numpy()
    assert max_abs(got_O, O_ref) <= 1e-5 * max(1.0, np.abs(O_ref).max())
    assert not np.any(got_O[~fin])
    # the bf16 output is the merged fp32 value rounded to nearest even, bit for bit
    assert torch.equal(out.view(torch.int16), Oa_dev.to(torch.bfloat16).view(torch.int16))


RING_CASES = [
    # P (devices), C (chunk length), Hq, Hkv, Dh
    (2, 256, 4, 2, 128),
    (3, 200, 2, 1, 64),
    (4, 128, 8, 2, 128),
]


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: f"P{c[0]}_C{c[1]}_hq{c[2]}_hkv{c[3]}_dh{c[4]}")
def test_zigzag_ring_share_matches_causal_attention(case):
    P, C, Hq, Hkv, Dh = case
    S = 2 * P * C
    q, k, v, _ = qkv_inputs(S, Hq, Hkv, Dh)
    qt, kt, vt = (bf16_tensor(x) for x in (q, k, v))
    n0 = up.launch_count()
    O, lse = up.ring_attention_share(qt, kt, vt, P)
    torch.cuda.synchronize()
    n_blocks = P * (2 * P + 1)
    assert up.launch_count() - n0 == 2 * 4 + 2 * n_blocks   # two tables, then one attention + one merge per block
    Q, K, V = (ui.bf16_to_f64(x) for x in (q, k, v))
    O_ref, L_ref = orc.attention_forward(Q, K, V, None, True, orc.default_scale(Dh))
    o = to_f64(O)
    assert max_abs_bf16_out(o, O_ref) <= OUT_MAX_ABS, max_abs_bf16_out(o, O_ref)
    assert rel_fro(o, O_ref) <= OUT_REL_FRO, rel_fro(o, O_ref)
    assert max_abs(to_f64(lse), L_ref) <= 1e-3


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: f"P{c[0]}_C{c[1]}_hq{c[2]}_hkv{c[3]}_dh{c[4]}")
def test_zigzag_ring_share_backward_matches_causal_gradients(case):
    P, C, Hq, Hkv, Dh = case
    S = 2 * P * C
    q, k, v, do = qkv_inputs(S, Hq, Hkv, Dh)
    qt, kt, vt, dot = (bf16_tensor(x) for x in (q, k, v, do))
    O, lse = up.ring_attention_share(qt, kt, vt, P)
    n0 = up.launch_count()
    dq, dk, dv = up.ring_attention_share_backward(qt, kt, vt, O, lse, dot, P)
    torch.cuda.synchronize()
    n_blocks = P * (2 * P + 1)
    # two tables, one D buffer per chunk, then per block dQ, dK/dV and three accumulations
    assert up.launch_count() - n0 == 2 * 4 + 2 * P + 5 * n_blocks
    Q, K, V, dO = (ui.bf16_to_f64(x) for x in (q, k, v, do))
    dQ, dK, dV = orc.attention_backward(Q, K, V, dO, None, True, orc.default_scale(Dh))
    assert rel_fro(to_f64(dq), dQ) <= GRAD_REL_FRO, rel_fro(to_f64(dq), dQ)
    assert rel_fro(to_f64(dk), dK) <= GRAD_REL_FRO, rel_fro(to_f64(dk), dK)
    assert rel_fro(to_f64(dv), dV) <= GRAD_REL_FRO, rel_fro(to_f64(dv), dV)


@pytest.mark.parametrize("S,H,Dh", [(1, 1, 64), (200, 3, 64), (1000, 4, 128)])
def test_ring_bwd_prep_matches_definition(S, H, Dh):
    o = ui.normal_bf16(H * S * Dh, 44).reshape(H, S, Dh)
    g = ui.normal_bf16(H * S * Dh, 45).reshape(H, S, Dh)
    L = ui.bf16_to_f64(ui.normal_bf16(H * S, 46, 3.0)).reshape(H, S)
    sp = -(-S // 128) * 128
    D = torch.full((2, H, sp), 7.0, dtype=torch.float32, device="cuda")
    up.ring_bwd_prep(bf16_tensor(o), bf16_tensor(g), torch.from_numpy(L.astype(np.float32)).cuda(), D)
    torch.cuda.synchronize()
    got = D.cpu().double().numpy()
    want = (ui.bf16_to_f64(o) * ui.bf16_to_f64(g)).sum(axis=2)
    assert max_abs(got[0, :, :S], want) <= 1e-5 * max(1.0, np.abs(want).max())
    assert max_abs(got[1, :, :S], L * np.log2(np.e)) <= 1e-5 * max(1.0, np.abs(L).max())
    assert not np.any(got[:, :, S:])


@pytest.mark.parametrize("n", [1, 7, 4096 + 3])
def test_accumulate_sums_in_fp32_and_rounds_once(n):
    src = ui.normal_bf16(n, 47)
    acc0 = ui.bf16_to_f64(ui.normal_bf16(n, 48)).astype(np.float32)
    acc = torch.from_numpy(acc0.copy()).cuda()
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    up.accumulate(bf16_tensor(src), acc, out)
    torch.cuda.synchronize()
    want = acc0 + ui.bf16_to_f64(src).astype(np.float32)   # one fp32 addition per element
    np.testing.assert_array_equal(acc.cpu().numpy(), want)
    assert torch.equal(out.view(torch.int16), acc.to(torch.bfloat16).view(torch.int16))
