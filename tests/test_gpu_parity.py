"""GPU parity: the CUDA path through the C-ABI against the fp64 oracle on the same seeded inputs.

Bar: tile tables and visited counts bit-exact; outputs max-abs <= 1e-2 and relative Frobenius
<= 5e-3; gradients relative Frobenius <= 1e-2."""
import numpy as np
import pytest
import torch

import long_context_attention_upipe_gb300 as up
import oracle as orc
import upipe_inputs as ui
from helpers import (GRAD_REL_FRO, OUT_MAX_ABS, OUT_REL_FRO, bf16_tensor, layer_inputs, max_abs, max_abs_bf16_out, qkv_inputs, rel_fro,
                     to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()
    ui.build(device=True)


def gpu_table(S, seg_np, causal):
    desc = up.make_desc(S, 64, 1, 1, 64, 1, causal)
    table = torch.empty(up.tile_table_bytes(desc), dtype=torch.uint8, device="cuda")
    seg = torch.from_numpy(seg_np).cuda() if seg_np is not None else None
    host_counts = up.build_tile_table(desc, seg, table, counts=True)   # read back by the library
    torch.cuda.synchronize()
    t = table.cpu().numpy()
    nt = -(-S // 128)
    head = t[:32]
    counts = head[:16].view(np.int64)
    assert list(host_counts) == counts.tolist()
    err = int(head[16:20].view(np.int32)[0])
    q_rows = t[32:32 + 16 * nt].view(np.int32).reshape(nt, 4)
    kv_rows = t[32 + 16 * nt:32 + 32 * nt].view(np.int32).reshape(nt, 4)
    return q_rows, kv_rows, counts, err, table


def gpu_orders(table, S):
    """The table's dispatch orders: query-tile pairs, then key tiles (int32, after the ranges)."""
    t = table.cpu().numpy()
    nt = -(-S // 128)
    np_ = (nt + 1) // 2
    o = 32 + 32 * nt
    return t[o:o + 4 * np_].view(np.int32), t[o + 4 * np_:o + 4 * np_ + 4 * nt].view(np.int32)


def expected_orders(q_rows, kv_rows):
    """Pairs (2p, 2p + 1) by non-increasing number of non-empty key tiles, ties later pair first;
    key tiles by non-increasing number of non-empty query tiles, ties earlier tile first."""
    nt = len(q_rows)
    wq = (q_rows[:, 3] - q_rows[:, 0]).astype(np.int64)
    wq = np.append(wq, 0) if nt % 2 else wq
    wp = wq[0::2] + wq[1::2]
    pairs = np.arange(len(wp))
    q_order = np.lexsort((-pairs, -wp))
    wk = (kv_rows[:, 3] - kv_rows[:, 0]).astype(np.int64)
    kv_order = np.lexsort((np.arange(nt), -wk))
    return q_order.astype(np.int32), kv_order.astype(np.int32)


def random_segments(S, rng, max_segs=8):
    k = int(rng.integers(1, max_segs + 1))
    if S < 2 or k == 1:
        return ui.segments_from_lengths([S])
    cuts = np.sort(rng.choice(np.arange(1, S), size=min(k - 1, S - 1), replace=False))
    return ui.segments_from_lengths(np.diff(np.concatenate([[0], cuts, [S]])))


# ----------------------------------------------------------------------------------------------
# tile-skip table: bit-exact
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 7, 128, 129, 300, 512, 1000, 5000, 70000])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_table_bit_exact(S, causal):
    rng = np.random.default_rng(S * 3 + causal)
    for trial in range(3):
        seg = None if trial == 0 else random_segments(S, rng, 8 if trial == 1 else 40)
        want_q, want_kv, want_tot = orc.tile_table(S, seg, causal)
        q, kv, counts, err, table = gpu_table(S, seg, causal)
        assert err == 0
        np.testing.assert_array_equal(q, want_q)
        np.testing.assert_array_equal(kv, want_kv)
        np.testing.assert_array_equal(counts, want_tot)
        for got, want in zip(gpu_orders(table, S), expected_orders(want_q, want_kv)):
            np.testing.assert_array_equal(got, want)


def test_tile_table_packed_131k():
    w = ui.workload("packed_131k")
    seg = w.segments()
    want_q, want_kv, want_tot = orc.tile_table(w.S, seg, True)
    q, kv, counts, err, table = gpu_table(w.S, seg, True)
    assert err == 0
    np.testing.assert_array_equal(q, want_q)
    np.testing.assert_array_equal(kv, want_kv)
    np.testing.assert_array_equal(counts, want_tot)
    for got, want in zip(gpu_orders(table, w.S), expected_orders(want_q, want_kv)):
        np.testing.assert_array_equal(got, want)


def test_tile_table_5m_sampled_and_closed_form():
    S = 5_000_000
    n = -(-S // 128)
    q, kv, counts, err, table = gpu_table(S, None, True)
    assert err == 0
    assert counts.tolist() == [n, n * (n - 1) // 2]  # diagonal partial, the rest of the triangle full
    # one causal segment: query tile i sees i + 1 key tiles, key tile j is seen by n - j query tiles
    i = np.arange(n)
    closed_q = np.stack([0 * i, 0 * i, i, i + 1], 1)
    closed_kv = np.stack([i, i, 0 * i + n, 0 * i + n], 1)
    for got, want in zip(gpu_orders(table, S), expected_orders(closed_q, closed_kv)):
        np.testing.assert_array_equal(got, want)
    sel = np.array([0, 1, 2, 777, n // 2, n - 2, n - 1])
    want_q, want_kv, _ = orc.tile_table(S, None, True, q_tiles=sel, kv_tiles=sel)
    np.testing.assert_array_equal(q[sel], want_q)
    np.testing.assert_array_equal(kv[sel], want_kv)


def test_tile_table_rejects_unsorted_segments():
    seg = np.array([0] * 100 + [1] * 100 + [0] * 56, dtype=np.int32)
    *_, err, table = gpu_table(256, seg, True)
    assert err == 5
    assert up.device_status(table) == 5
    assert up.last_device_error(table) == 5


# ----------------------------------------------------------------------------------------------
# GEMM alone
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (300, 128, 64), (1000, 384, 256), (4096, 1024, 4096)])
def test_gemm_nt_matches_fp64(M, N, K):
    A = ui.normal_bf16(M * K, 20).reshape(M, K)
    B = ui.normal_bf16(N * K, 21, 0.05).reshape(N, K)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    a, b = bf16_tensor(A), bf16_tensor(B)
    n0 = up.launch_count()
    up.gemm_nt(a, b, C)
    assert up.launch_count() - n0 == 1  # one tensor-core GEMM kernel, no split-K reduce
    torch.cuda.synchronize()
    want = ui.bf16_to_f64(A) @ ui.bf16_to_f64(B).T
    got = C.cpu().double().numpy()
    assert rel_fro(got, want) < 1e-5
    assert max_abs(got, want) < 1e-3 * max(1.0, np.abs(want).max())


# ----------------------------------------------------------------------------------------------
# attention core alone (Q, K, V given directly)
# ----------------------------------------------------------------------------------------------

CORE_CASES = [
    # S, Hq, Hkv, Dh, segment lengths, causal
    (1, 1, 1, 64, None, True),
    (300, 4, 2, 64, [100, 200], True),
    (700, 2, 1, 128, [300, 1, 399], True),
    (512, 4, 4, 128, None, False),
    (1000, 4, 1, 128, [129, 500, 371], False),
    (2048, 2, 1, 128, None, True),
]


def run_core(S, Hq, Hkv, Dh, segs, causal):
    q, k, v, do = qkv_inputs(S, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs) if segs else None
    desc = up.make_desc(S, 64, Hq, Hkv, Dh, Hq, causal)
    table = torch.empty(up.tile_table_bytes(desc), dtype=torch.uint8, device="cuda")
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    up.build_tile_table(desc, seg_t, table)
    qt, kt, vt, dot = (bf16_tensor(x) for x in (q, k, v, do))
    o = torch.empty_like(qt)
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    up.core_fwd(desc, qt, kt, vt, seg_t, table, o, lse)
    dq, dk, dv = torch.empty_like(qt), torch.empty_like(kt), torch.empty_like(vt)
    up.core_bwd(desc, qt, kt, vt, dot, lse, seg_t, table, dq, dk, dv)
    torch.cuda.synchronize()
    return (q, k, v, do, seg), (to_f64(o), to_f64(lse), to_f64(dq), to_f64(dk), to_f64(dv))


@pytest.mark.parametrize("case", CORE_CASES, ids=lambda c: f"S{c[0]}_hq{c[1]}_hkv{c[2]}_dh{c[3]}_c{int(c[5])}")
def test_core_fwd_bwd_match_oracle(case):
    S, Hq, Hkv, Dh, segs, causal = case
    (q, k, v, do, seg), (o, lse, dq, dk, dv) = run_core(*case)
    Q, K, V, dO = (ui.bf16_to_f64(x) for x in (q, k, v, do))
    scale = orc.default_scale(Dh)
    O_ref, L_ref = orc.attention_forward(Q, K, V, seg, causal, scale)
    assert max_abs_bf16_out(o, O_ref) <= OUT_MAX_ABS
    assert rel_fro(o, O_ref) <= OUT_REL_FRO
    assert max_abs(lse, L_ref) <= 1e-3
    dQ, dK, dV = orc.attention_backward(Q, K, V, dO, seg, causal, scale)
    assert rel_fro(dq, dQ) <= GRAD_REL_FRO, rel_fro(dq, dQ)
    assert rel_fro(dk, dK) <= GRAD_REL_FRO, rel_fro(dk, dK)
    assert rel_fro(dv, dV) <= GRAD_REL_FRO, rel_fro(dv, dV)


@pytest.mark.parametrize("window", [2, 4, 1 << 24])
@pytest.mark.parametrize("case", [CORE_CASES[2], CORE_CASES[4], CORE_CASES[5]],
                         ids=lambda c: f"S{c[0]}_hq{c[1]}_hkv{c[2]}_dh{c[3]}_c{int(c[5])}")
def test_core_dkdv_into_fp32_sums_flushed_in_windows(case, window):
    # dK / dV added to fp32 sums that already hold values, the tensor-memory accumulators flushed
    # every `window` work items (2: after every item pair; 2^24: never)
    S, Hq, Hkv, Dh, segs, causal = case
    q, k, v, do = qkv_inputs(S, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs) if segs else None
    desc = up.make_desc(S, 64, Hq, Hkv, Dh, Hq, causal)
    table = torch.empty(up.tile_table_bytes(desc), dtype=torch.uint8, device="cuda")
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    up.build_tile_table(desc, seg_t, table)
    qt, kt, vt, dot = (bf16_tensor(x) for x in (q, k, v, do))
    o = torch.empty_like(qt)
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    up.core_fwd(desc, qt, kt, vt, seg_t, table, o, lse)
    D = torch.empty(2, Hq, -(-S // 128) * 128, dtype=torch.float32, device="cuda")
    up.core_recompute(desc, qt, kt, vt, dot, lse, seg_t, table, o, D)
    rng = np.random.default_rng(7)
    init_k = rng.standard_normal((Hkv, S, Dh))
    init_v = rng.standard_normal((Hkv, S, Dh))
    dk_acc = torch.from_numpy(init_k.astype(np.float32)).cuda()
    dv_acc = torch.from_numpy(init_v.astype(np.float32)).cuda()
    dk, dv = torch.empty_like(kt), torch.empty_like(vt)
    try:
        up.set_dkdv_window(window)
        up.core_bwd_dkdv_acc(desc, qt, kt, vt, dot, lse, D, seg_t, table, dk_acc, dv_acc, dk, dv)
        torch.cuda.synchronize()
    finally:
        up.set_dkdv_window(0)
    assert up.device_status(table) == 0
    Q, K, V, dO = (ui.bf16_to_f64(x) for x in (q, k, v, do))
    _, dK, dV = orc.attention_backward(Q, K, V, dO, seg, causal, orc.default_scale(Dh))
    sk, sv = dk_acc.double().cpu().numpy() - init_k, dv_acc.double().cpu().numpy() - init_v
    assert rel_fro(sk, dK) <= GRAD_REL_FRO, rel_fro(sk, dK)
    assert rel_fro(sv, dV) <= GRAD_REL_FRO, rel_fro(sv, dV)
    # the bf16 outputs are the sums rounded (to the nearest bf16: within half a bf16 unit)
    for out, acc in ((dk, dk_acc), (dv, dv_acc)):
        a = acc.double().cpu().numpy()
        assert np.all(np.abs(to_f64(out) - a) <= np.abs(a) * 2.0 ** -8 + 1e-30)


def grow_keys(k, S, every=384):
    """K with its magnitude doubled every `every` positions (an exact bf16 exponent shift), so the
    scores of late key tiles outgrow those of the first tile by far more than 2^16 in exp2 units."""
    e = (np.arange(S) // every).astype(np.uint16)
    bits = k.astype(np.uint16)
    grown = bits + (e[None, :, None] << 7).astype(np.uint16)
    return np.where((bits & 0x7F80) != 0, grown, bits).astype(np.uint16)


@pytest.mark.parametrize("segs", [None, [700, 1348]])
def test_forward_offset_moves_when_scores_outgrow_it(segs):
    """The forward's optimistic softmax offset: keys whose magnitude doubles every 384 positions
    make later tiles' scores exceed the first visible tile's maximum by more than 2^16, so the
    forward has to move the offset, rescale O and l and redo the tile's P; results at the bar."""
    S, Hq, Hkv, Dh = 2048, 2, 1, 128
    q, k, v, do = qkv_inputs(S, Hq, Hkv, Dh)
    k = grow_keys(k, S)
    seg = ui.segments_from_lengths(segs) if segs else None
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    desc = up.make_desc(S, 64, Hq, Hkv, Dh, Hq, True)
    table = torch.empty(up.tile_table_bytes(desc), dtype=torch.uint8, device="cuda")
    up.build_tile_table(desc, seg_t, table)
    qt, kt, vt, dot = (bf16_tensor(x) for x in (q, k, v, do))
    o = torch.empty_like(qt)
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    up.core_fwd(desc, qt, kt, vt, seg_t, table, o, lse)
    dq, dk, dv = torch.empty_like(qt), torch.empty_like(kt), torch.empty_like(vt)
    up.core_bwd(desc, qt, kt, vt, dot, lse, seg_t, table, dq, dk, dv)
    torch.cuda.synchronize()
    assert up.device_status(table) == 0
    Q, K, V, dO = (ui.bf16_to_f64(x) for x in (q, k, v, do))
    scale = orc.default_scale(Dh)
    O_ref, L_ref = orc.attention_forward(Q, K, V, seg, True, scale)
    if seg is None:  # the scores really do outgrow the first tile's maximum by more than 16 in exp2 units
        s0 = (Q[:, 1500] @ K[0, :128].T).max(axis=-1) * scale * np.log2(np.e)
        assert np.all(L_ref[:, 1500] * np.log2(np.e) - s0 > 16)
    assert max_abs_bf16_out(to_f64(o), O_ref) <= OUT_MAX_ABS
    assert rel_fro(to_f64(o), O_ref) <= OUT_REL_FRO
    assert max_abs(to_f64(lse), L_ref) <= 1e-3 * max(1.0, np.abs(L_ref).max())
    dQ, dK, dV = orc.attention_backward(Q, K, V, dO, seg, True, scale)
    assert rel_fro(to_f64(dq), dQ) <= GRAD_REL_FRO
    assert rel_fro(to_f64(dk), dK) <= GRAD_REL_FRO
    assert rel_fro(to_f64(dv), dV) <= GRAD_REL_FRO


# ----------------------------------------------------------------------------------------------
# the whole layer, chunked
# ----------------------------------------------------------------------------------------------

LAYER_CASES = [
    # S, d, Hq, Hkv, Dh, segment lengths, causal, hpc, accum_mode
    (512, 256, 4, 2, 64, [300, 212], True, 2, 0),   # the tiny workload
    (512, 256, 4, 2, 64, [300, 212], True, 1, 0),
    (512, 256, 4, 2, 64, [300, 212], True, 4, 0),
    (512, 256, 4, 2, 64, [300, 212], True, 1, 1),
    (300, 128, 4, 1, 128, None, True, 1, 0),        # partial KV groups, ragged S
    (300, 128, 4, 1, 128, None, False, 2, 0),
    (1000, 256, 8, 2, 128, [250, 1, 600, 149], True, 4, 0),
    (1000, 256, 8, 2, 128, [250, 1, 600, 149], True, 8, 1),
]


@pytest.mark.parametrize("case", LAYER_CASES,
                         ids=lambda c: f"S{c[0]}_d{c[1]}_hq{c[2]}_hkv{c[3]}_dh{c[4]}_c{int(c[6])}_hpc{c[7]}_acc{c[8]}")
def test_layer_fwd_bwd_match_oracle(case):
    S, d, Hq, Hkv, Dh, segs, causal, hpc, accum = case
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs) if segs else None
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, causal, accum)
    layer = up.Layer(desc)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    seg_t = torch.from_numpy(seg).cuda() if seg is not None else None
    Y, lse = layer.forward(Xt, Wt, Wot, seg_t)
    dX, dW, dWo = layer.backward(Xt, Wt, Wot, seg_t, dYt, lse)
    torch.cuda.synchronize()
    assert up.device_status(layer.ws_fwd) == 0 and up.device_status(layer.ws_bwd) == 0
    Y_ref, L_ref = orc.layer_forward(X, W, Wo, seg, Hq, Hkv, Dh, causal)
    dX_ref, dW_ref, dWo_ref = orc.layer_backward(X, W, Wo, seg, dY, Hq, Hkv, Dh, causal)
    y = to_f64(Y)
    assert max_abs_bf16_out(y, Y_ref) <= OUT_MAX_ABS, max_abs_bf16_out(y, Y_ref)
    assert rel_fro(y, Y_ref) <= OUT_REL_FRO, rel_fro(y, Y_ref)
    assert max_abs(to_f64(lse), L_ref) <= 1e-3
    assert rel_fro(to_f64(dX), dX_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dX), dX_ref)
    assert rel_fro(to_f64(dW), dW_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dW), dW_ref)
    assert rel_fro(to_f64(dWo), dWo_ref) <= GRAD_REL_FRO, rel_fro(to_f64(dWo), dWo_ref)


@pytest.mark.parametrize("window,hpc", [(2, 4), (6, 4), (30, 4), (4, 1), (8, 8)])
def test_layer_backward_with_flushed_dkdv_windows(window, hpc):
    # windows of a few work items: every key tile adds its tensor-memory dK / dV accumulators to
    # the fp32 sums many times (up to 32 items per key tile of a whole group here: 4 query heads x
    # 8 query tiles; a window of 30 leaves a ragged last one); the gradients must match the oracle
    # and the unflushed run to rounding
    S, d, Hq, Hkv, Dh = 1000, 256, 8, 2, 128
    segs, causal = [250, 1, 600, 149], True
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    seg_t = torch.from_numpy(seg).cuda()
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, causal)
    plain = up.Layer(desc)
    Y, lse = plain.forward(Xt, Wt, Wot, seg_t)
    ref = [to_f64(t) for t in plain.backward(Xt, Wt, Wot, seg_t, dYt, lse)]
    try:
        up.set_dkdv_window(window)
        flushed = up.Layer(desc)
        if hpc >= Hq // Hkv:                                  # whole groups: now with fp32 sums
            assert flushed.ws_bwd.numel() > plain.ws_bwd.numel()
        got = [to_f64(t) for t in flushed.backward(Xt, Wt, Wot, seg_t, dYt, lse)]
    finally:
        up.set_dkdv_window(0)
    torch.cuda.synchronize()
    assert up.device_status(flushed.ws_bwd) == 0
    dX_ref, dW_ref, dWo_ref = orc.layer_backward(X, W, Wo, seg, dY, Hq, Hkv, Dh, causal)
    for g, r, o in zip(got, ref, (dX_ref, dW_ref, dWo_ref)):
        assert rel_fro(g, o) <= GRAD_REL_FRO, rel_fro(g, o)
        assert rel_fro(g, r) <= 2e-3, rel_fro(g, r)            # the same products, summed in 2 stages
    np.testing.assert_array_equal(got[2], ref[2])               # dWo does not involve dK / dV


def test_layer_output_independent_of_chunking():
    S, d, Hq, Hkv, Dh = 640, 256, 8, 2, 64
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    outs = []
    for hpc in (1, 2, 4, 8):
        layer = up.Layer(up.make_desc(S, d, Hq, Hkv, Dh, hpc, True))
        Y, lse = layer.forward(Xt, Wt, Wot)
        dX, dW, dWo = layer.backward(Xt, Wt, Wot, None, dYt, lse)
        outs.append([to_f64(t) for t in (Y, lse, dX, dW, dWo)])
    for o in outs[1:]:
        assert rel_fro(o[0], outs[0][0]) <= OUT_REL_FRO
        assert max_abs(o[1], outs[0][1]) <= 1e-4
        for i in (2, 3, 4):
            assert rel_fro(o[i], outs[0][i]) <= GRAD_REL_FRO


def test_layer_flags_unsorted_segments():
    S, d, Hq, Hkv, Dh = 256, 128, 2, 1, 64
    X, W, Wo, _ = layer_inputs(S, d, Hq, Hkv, Dh, dy=False)
    seg = np.array([0] * 100 + [2] * 100 + [1] * 56, dtype=np.int32)
    layer = up.Layer(up.make_desc(S, d, Hq, Hkv, Dh, 1, True))
    layer.forward(bf16_tensor(X), bf16_tensor(W), bf16_tensor(Wo), torch.from_numpy(seg).cuda())
    assert up.device_status(layer.ws_fwd) == 5



def test_layer_step_replays_bit_exact_from_a_cuda_graph():
    """The forward and backward calls make no synchronous host call and allocate nothing, so a
    step can be captured once in a CUDA graph; its replays give the eager results bit for bit."""
    S, d, Hq, Hkv, Dh = 640, 256, 8, 2, 64
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    desc = up.make_desc(S, d, Hq, Hkv, Dh, 2, True)
    layer = up.Layer(desc)
    Y = torch.empty_like(Xt); lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    dX = torch.empty_like(Xt); dW = torch.empty(Wt.shape, dtype=torch.float32, device="cuda")
    dWo = torch.empty(Wot.shape, dtype=torch.float32, device="cuda")

    def step(s):
        up.fwd(desc, Xt, Wt, Wot, None, Y, lse, layer.ws_fwd, s)
        up.bwd(desc, Xt, Wt, Wot, None, dYt, lse, dX, dW, dWo, layer.ws_bwd, s)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [t.clone() for t in (Y, lse, dX, dW, dWo)]
    for t in (Y, lse, dX, dW, dWo):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    n0 = up.launch_count()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    assert up.launch_count() > n0
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for got, want in zip((Y, lse, dX, dW, dWo), eager):
        assert torch.equal(got, want)


def test_per_launch_timing_logs_the_schedule():
    """With timing on, every kernel launch of a forward and a backward is logged once with its
    kind and shape, the results are unchanged, and turning it off logs nothing more."""
    S, d, Hq, Hkv, Dh, hpc = 512, 256, 4, 2, 64, 1      # 4 chunks, 2 per KV group (hpc < g)
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    layer = up.Layer(up.make_desc(S, d, Hq, Hkv, Dh, hpc, True))
    Y0, lse0 = layer.forward(Xt, Wt, Wot)
    torch.cuda.synchronize()
    up.timing_records()
    up.timing_enable(True)
    try:
        Y, lse = layer.forward(Xt, Wt, Wot)
        dX, dW, dWo = layer.backward(Xt, Wt, Wot, None, dYt, lse)
        torch.cuda.synchronize()
    finally:
        up.timing_enable(False)
    recs = up.timing_records()
    kinds = [r["kind"] for r in recs]
    n_chunks = Hq // hpc
    assert kinds.count("tile_table") == 2
    assert kinds.count("attn_fwd") == n_chunks and kinds.count("recompute") == n_chunks
    assert kinds.count("bwd_dq") == n_chunks and kinds.count("bwd_dkdv") == n_chunks
    assert kinds.count("qkv_proj") == 2 * n_chunks and kinds.count("o_proj") == n_chunks
    assert kinds.count("dx_proj") == n_chunks and kinds.count("dwqkv") == n_chunks
    assert kinds.count("convert") == 2 + Hkv      # Y and dX sums once each, dK/dV at each group end
    assert kinds.count("zero") == Hkv
    assert all(r["ms"] >= 0 for r in recs)
    epis = [r["epilogue"] for r in recs if r["kind"] == "o_proj"]
    assert epis == [1] + [2] * (n_chunks - 1)     # first chunk stores the fp32 sum, later chunks add
    assert torch.equal(Y, Y0) and torch.equal(lse, lse0)
    layer.forward(Xt, Wt, Wot)
    torch.cuda.synchronize()
    assert up.timing_records() == []


def test_bounded_wait_runs_out_and_the_gpu_stays_usable():
    """The bounded device wait every warp-specialised kernel uses gives up after the limit, raises
    UPIPE_ERR_DEVICE_TIMEOUT in the error word and returns: a probe kernel waits on a barrier that
    nothing completes (and, as a control, on one it completed itself).  A layer call right after
    it, with the default limit restored, still matches the oracle."""
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    try:
        up.set_wait_limit_ns(2_000_000)          # 2 ms
        up.wait_probe(buf, arrive=True)
        assert up.device_status(buf) == 0
        t0 = torch.cuda.Event(enable_timing=True); t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        up.wait_probe(buf, arrive=False)
        t1.record()
        assert up.device_status(buf) == 7        # UPIPE_ERR_DEVICE_TIMEOUT
        assert 2.0 <= t0.elapsed_time(t1) < 1000.0
    finally:
        up.set_wait_limit_ns(0)
    S, d, Hq, Hkv, Dh, segs, causal, hpc, accum = LAYER_CASES[0]
    X, W, Wo, dY = layer_inputs(S, d, Hq, Hkv, Dh)
    seg = ui.segments_from_lengths(segs)
    layer = up.Layer(up.make_desc(S, d, Hq, Hkv, Dh, hpc, causal, accum))
    Xt, Wt, Wot, dYt = (bf16_tensor(x) for x in (X, W, Wo, dY))
    seg_t = torch.from_numpy(seg).cuda()
    Y, lse = layer.forward(Xt, Wt, Wot, seg_t)
    dX, dW, dWo = layer.backward(Xt, Wt, Wot, seg_t, dYt, lse)
    torch.cuda.synchronize()
    assert up.device_status(layer.ws_fwd) == 0 and up.device_status(layer.ws_bwd) == 0
    Y_ref, _ = orc.layer_forward(X, W, Wo, seg, Hq, Hkv, Dh, causal)
    dX_ref, _, _ = orc.layer_backward(X, W, Wo, seg, dY, Hq, Hkv, Dh, causal)
    assert max_abs_bf16_out(to_f64(Y), Y_ref) <= OUT_MAX_ABS and rel_fro(to_f64(Y), Y_ref) <= OUT_REL_FRO
    assert rel_fro(to_f64(dX), dX_ref) <= GRAD_REL_FRO
