"""Pins for the fp64 oracle: each check comes from outside the oracle's own code
(brute force, an independent library routine, finite differences, closed forms, invariants)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
import upipe_inputs as ui


def rand_layer(S, d, Hq, Hkv, Dh, seed=0, std_w=0.3):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((S, d))
    Wqkv = std_w * rng.standard_normal(((Hq + 2 * Hkv) * Dh, d))
    Wo = std_w * rng.standard_normal((d, Hq * Dh))
    dY = rng.standard_normal((S, d))
    return X, Wqkv, Wo, dY


def rand_qkv(S, Hq, Hkv, Dh, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((Hq, S, Dh)), rng.standard_normal((Hkv, S, Dh)),
            rng.standard_normal((Hkv, S, Dh)))


def random_segments(S, rng, max_segs=6):
    k = int(rng.integers(1, max_segs + 1))
    cuts = np.sort(rng.choice(np.arange(1, S), size=min(k - 1, S - 1), replace=False)) if S > 1 else []
    lens = np.diff(np.concatenate([[0], cuts, [S]])).astype(int)
    return ui.segments_from_lengths(lens)


# ------------------------------------------------------------------------------------------
# 1. brute-force per-row softmax (Python floats, one element at a time)
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_attention_matches_bruteforce_rows(causal):
    S, Hq, Hkv, Dh = 23, 4, 2, 5
    Q, K, V = rand_qkv(S, Hq, Hkv, Dh, seed=1)
    seg = ui.segments_from_lengths([9, 1, 13])
    scale = 0.37
    O, LSE = orc.attention_forward(Q, K, V, seg, causal, scale)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        for i in range(S):
            scores = [scale * sum(Q[h, i, e] * K[kv, j, e] for e in range(Dh)) for j in range(S)]
            vis = [seg[i] == seg[j] and (not causal or j <= i) for j in range(S)]
            p, lse = orc.rowsoftmax_bruteforce(scores, vis)
            assert abs(sum(p) - 1.0) < 1e-12
            o = [sum(p[j] * V[kv, j, e] for j in range(S)) for e in range(Dh)]
            np.testing.assert_allclose(O[h, i], o, rtol=0, atol=1e-12)
            assert abs(LSE[h, i] - lse) < 1e-12
            assert LSE[h, i] >= max(s for s, v in zip(scores, vis) if v) - 1e-15


# ------------------------------------------------------------------------------------------
# 2. independent library routine: torch float64 SDPA + autograd
# ------------------------------------------------------------------------------------------

def torch_layer(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal, scale):
    S, d = X.shape
    X = torch.tensor(X, requires_grad=True)
    Wqkv = torch.tensor(Wqkv, requires_grad=True)
    Wo = torch.tensor(Wo, requires_grad=True)
    qkv = torch.nn.functional.linear(X, Wqkv)
    q = qkv[:, : Hq * Dh].reshape(S, Hq, Dh).transpose(0, 1)
    k = qkv[:, Hq * Dh: (Hq + Hkv) * Dh].reshape(S, Hkv, Dh).transpose(0, 1)
    v = qkv[:, (Hq + Hkv) * Dh:].reshape(S, Hkv, Dh).transpose(0, 1)
    g = Hq // Hkv
    k = k.repeat_interleave(g, dim=0)
    v = v.repeat_interleave(g, dim=0)
    i = torch.arange(S)
    mask = torch.ones(S, S, dtype=torch.bool)
    if seg is not None:
        st = torch.tensor(seg)
        mask &= st[:, None] == st[None, :]
    if causal:
        mask &= i[None, :] <= i[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask,
                                                         scale=scale)[0]
    y = torch.nn.functional.linear(o.transpose(0, 1).reshape(S, Hq * Dh), Wo)
    return y, (X, Wqkv, Wo)


@pytest.mark.parametrize("causal,segs,Hq,Hkv", [(True, None, 4, 2), (True, [20, 1, 27], 4, 1),
                                               (False, [30, 18], 3, 3), (False, None, 2, 1)])
def test_layer_matches_torch_autograd(causal, segs, Hq, Hkv):
    S, d, Dh = 48, 16, 8
    X, Wqkv, Wo, dY = rand_layer(S, d, Hq, Hkv, Dh, seed=2)
    seg = None if segs is None else ui.segments_from_lengths(segs)
    scale = orc.default_scale(Dh)
    Y, LSE = orc.layer_forward(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal, scale)
    yt, (Xt, Wt, Wot) = torch_layer(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal, scale)
    np.testing.assert_allclose(Y, yt.detach().numpy(), rtol=1e-11, atol=1e-12)
    yt.backward(torch.tensor(dY))
    dX, dW, dWo = orc.layer_backward(X, Wqkv, Wo, seg, dY, Hq, Hkv, Dh, causal, scale)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dWo, Wot.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_lse_matches_torch_logsumexp():
    S, Hq, Hkv, Dh = 40, 2, 1, 6
    Q, K, V = rand_qkv(S, Hq, Hkv, Dh, seed=3)
    seg = ui.segments_from_lengths([11, 29])
    O, LSE = orc.attention_forward(Q, K, V, seg, True, 0.5)
    for h in range(Hq):
        s = 0.5 * torch.tensor(Q[h]) @ torch.tensor(K[0]).T
        i = torch.arange(S)
        st = torch.tensor(seg)
        mask = (st[:, None] == st[None, :]) & (i[None, :] <= i[:, None])
        ref = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=1).numpy()
        np.testing.assert_allclose(LSE[h], ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------------------------------
# 3. central finite differences of L = sum(dY * Y)
# ------------------------------------------------------------------------------------------

def test_gradients_finite_differences():
    S, d, Hq, Hkv, Dh = 20, 8, 2, 1, 4
    X, Wqkv, Wo, dY = rand_layer(S, d, Hq, Hkv, Dh, seed=4, std_w=0.5)
    seg = ui.segments_from_lengths([7, 13])
    scale = 0.45
    dX, dW, dWo = orc.layer_backward(X, Wqkv, Wo, seg, dY, Hq, Hkv, Dh, True, scale)

    def loss(X_, W_, Wo_):
        Y, _ = orc.layer_forward(X_, W_, Wo_, seg, Hq, Hkv, Dh, True, scale)
        return float((dY * Y).sum())

    rng = np.random.default_rng(5)
    h = 1e-6
    for name, arr, grad in (("X", X, dX), ("W", Wqkv, dW), ("Wo", Wo, dWo)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args_p = dict(X=X, W=Wqkv, Wo=Wo)
            args_m = dict(X=X, W=Wqkv, Wo=Wo)
            args_p[name], args_m[name] = p, m
            fd = (loss(args_p["X"], args_p["W"], args_p["Wo"]) - loss(args_m["X"], args_m["W"], args_m["Wo"])) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])


# ------------------------------------------------------------------------------------------
# 4. closed forms
# ------------------------------------------------------------------------------------------

def test_first_row_and_singleton_segment_copy_v():
    S, Hq, Hkv, Dh = 16, 4, 2, 8
    Q, K, V = rand_qkv(S, Hq, Hkv, Dh, seed=6)
    seg = ui.segments_from_lengths([5, 1, 10])
    O, LSE = orc.attention_forward(Q, K, V, seg, True, 0.3)
    for h in range(Hq):
        kv = h // 2
        np.testing.assert_array_equal(O[h, 0], V[kv, 0])   # causal row 0 sees only itself
        np.testing.assert_array_equal(O[h, 5], V[kv, 5])   # length-1 segment
        assert LSE[h, 5] == pytest.approx(0.3 * Q[h, 5] @ K[kv, 5], abs=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_gives_mean_of_visible_values(causal):
    S, Hq, Hkv, Dh = 30, 2, 1, 4
    Q, K, V = rand_qkv(S, Hq, Hkv, Dh, seed=7)
    Q[:] = 0.0
    seg = ui.segments_from_lengths([12, 18])
    O, LSE = orc.attention_forward(Q, K, V, seg, causal, 1.0)
    for i in range(S):
        vis = [j for j in range(S) if seg[j] == seg[i] and (not causal or j <= i)]
        np.testing.assert_allclose(O[0, i], V[0, vis].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert LSE[0, i] == pytest.approx(math.log(len(vis)), abs=1e-14)


def test_single_token_single_head_is_two_linear_maps():
    d, Dh = 12, 4
    X, Wqkv, Wo, _ = rand_layer(1, d, 1, 1, Dh, seed=8)
    Y, _ = orc.layer_forward(X, Wqkv, Wo, None, 1, 1, Dh, True)
    Wv = Wqkv[2 * Dh: 3 * Dh]
    np.testing.assert_allclose(Y, X @ Wv.T @ Wo.T, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------------------------------
# 5. invariants
# ------------------------------------------------------------------------------------------

def test_causal_future_perturbation_leaves_past_unchanged():
    S, d, Hq, Hkv, Dh = 40, 16, 4, 2, 8
    X, Wqkv, Wo, _ = rand_layer(S, d, Hq, Hkv, Dh, seed=9)
    Y1, L1 = orc.layer_forward(X, Wqkv, Wo, None, Hq, Hkv, Dh, True)
    X2 = X.copy()
    X2[25:] += np.random.default_rng(10).standard_normal(X2[25:].shape)
    Y2, L2 = orc.layer_forward(X2, Wqkv, Wo, None, Hq, Hkv, Dh, True)
    np.testing.assert_array_equal(Y1[:25], Y2[:25])
    np.testing.assert_array_equal(L1[:, :25], L2[:, :25])
    assert np.abs(Y1[25:] - Y2[25:]).max() > 1e-3


@pytest.mark.parametrize("causal", [True, False])
def test_packed_equals_segments_computed_alone(causal):
    S, d, Hq, Hkv, Dh = 50, 16, 4, 2, 8
    lens = [17, 1, 32]
    X, Wqkv, Wo, dY = rand_layer(S, d, Hq, Hkv, Dh, seed=11)
    seg = ui.segments_from_lengths(lens)
    Y, LSE = orc.layer_forward(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal)
    dX, dW, dWo = orc.layer_backward(X, Wqkv, Wo, seg, dY, Hq, Hkv, Dh, causal)
    s0 = 0
    dW_sum, dWo_sum = np.zeros_like(dW), np.zeros_like(dWo)
    for L in lens:
        sl = slice(s0, s0 + L)
        Ys, Ls = orc.layer_forward(X[sl], Wqkv, Wo, None, Hq, Hkv, Dh, causal)
        dXs, dWs, dWos = orc.layer_backward(X[sl], Wqkv, Wo, None, dY[sl], Hq, Hkv, Dh, causal)
        np.testing.assert_allclose(Y[sl], Ys, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(LSE[:, sl], Ls, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dX[sl], dXs, rtol=1e-11, atol=1e-12)
        dW_sum += dWs
        dWo_sum += dWos
        s0 += L
    np.testing.assert_allclose(dW, dW_sum, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dWo, dWo_sum, rtol=1e-11, atol=1e-12)


def test_heads_are_independent_of_grouping():
    """The chunked method runs heads in groups; running the heads of a slice of the layer alone
    (the matching rows of Wqkv and columns of Wo) gives that slice's part of Y."""
    S, d, Hq, Hkv, Dh = 32, 16, 4, 2, 8
    X, Wqkv, Wo, _ = rand_layer(S, d, Hq, Hkv, Dh, seed=12)
    Y, LSE = orc.layer_forward(X, Wqkv, Wo, None, Hq, Hkv, Dh, True)
    Wq, Wk, Wv = orc.split_wqkv(Wqkv, Hq, Hkv, Dh)
    acc = np.zeros_like(Y)
    for kv in range(Hkv):  # one KV group per slice: Q heads 2kv, 2kv+1
        qs = slice(2 * kv * Dh, (2 * kv + 2) * Dh)
        ks = slice(kv * Dh, (kv + 1) * Dh)
        Wsub = np.concatenate([Wq[qs], Wk[ks], Wv[ks]])
        Ysub, Lsub = orc.layer_forward(X, Wsub, Wo[:, qs], None, 2, 1, Dh, True)
        np.testing.assert_allclose(Lsub, LSE[2 * kv: 2 * kv + 2], rtol=1e-13, atol=1e-13)
        acc += Ysub
    np.testing.assert_allclose(acc, Y, rtol=1e-12, atol=1e-12)


def test_rows_helper_matches_full_forward():
    S, d, Hq, Hkv, Dh = 300, 16, 4, 2, 8
    X, Wqkv, Wo, _ = rand_layer(S, d, Hq, Hkv, Dh, seed=13)
    seg = ui.segments_from_lengths([100, 150, 50])
    Y, LSE = orc.layer_forward(X, Wqkv, Wo, seg, Hq, Hkv, Dh, True)
    rows = np.array([0, 99, 100, 101, 255, 299])
    keys = np.arange(0, 300)
    Yr, Lr = orc.layer_forward_rows(X[rows], X[keys], keys, rows, Wqkv, Wo, seg, Hq, Hkv, Dh, True)
    np.testing.assert_allclose(Yr, Y[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Lr, LSE[:, rows], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal,segs,Hq,Hkv", [(True, None, 4, 2), (True, [20, 1, 27], 4, 1),
                                               (False, [30, 18], 2, 2)])
def test_rows_backward_matches_torch_autograd(causal, segs, Hq, Hkv):
    """dY non-zero on a few rows only (a tail window, a segment start, a single row)."""
    S, d, Dh = 48, 16, 8
    X, Wqkv, Wo, dY = rand_layer(S, d, Hq, Hkv, Dh, seed=21)
    seg = None if segs is None else ui.segments_from_lengths(segs)
    scale = orc.default_scale(Dh)
    rows = np.array([0, 20, 21, 33, 40, 41, 42, 43, 44, 45, 46, 47])
    dYz = np.zeros_like(dY)
    dYz[rows] = dY[rows]
    yt, (Xt, Wt, Wot) = torch_layer(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal, scale)
    yt.backward(torch.tensor(dYz))
    dX, dW, dWo = orc.layer_backward_rows(X, Wqkv, Wo, seg, dY[rows], rows, Hq, Hkv, Dh, causal, scale)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dWo, Wot.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_project_kv_blocks_match_one_product():
    S, d, Hq, Hkv, Dh = 300, 16, 4, 2, 8
    X, Wqkv, _, _ = rand_layer(S, d, Hq, Hkv, Dh, seed=5)
    _, Wk, Wv = orc.split_wqkv(Wqkv, Hq, Hkv, Dh)
    K, V = orc.project_kv(X, Wk, Wv, Hkv, Dh, row_block=64)
    np.testing.assert_allclose(K, (X @ Wk.T).reshape(S, Hkv, Dh).transpose(1, 0, 2), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(V, (X @ Wv.T).reshape(S, Hkv, Dh).transpose(1, 0, 2), rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------------------------------
# 5b. ring (P2P) merge of block results
# ------------------------------------------------------------------------------------------

def test_merge_of_disjoint_key_sets_equals_attention_over_their_union():
    S, Dh = 40, 8
    Q, K, V = rand_qkv(S, 2, 1, Dh, seed=31)
    scale = orc.default_scale(Dh)
    O, L = orc.attention_forward(Q, K, V, None, False, scale)
    rng = np.random.default_rng(3)
    sel = rng.permutation(S)
    A, B = np.sort(sel[:13]), np.sort(sel[13:])
    Oa, La = orc.attention_forward(Q, K[:, A], V[:, A], None, False, scale)
    Ob, Lb = orc.attention_forward(Q, K[:, B], V[:, B], None, False, scale)
    Om, Lm = orc.lse_merge(Oa, La, Ob, Lb)
    np.testing.assert_allclose(Om, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Lm, L, rtol=1e-13, atol=1e-13)
    Om2, Lm2 = orc.lse_merge(Ob, Lb, Oa, La)  # order of the blocks does not matter
    np.testing.assert_allclose(Om2, Om, rtol=1e-13, atol=1e-14)


def test_merge_with_an_empty_side():
    rng = np.random.default_rng(4)
    O = rng.standard_normal((3, 5, 4))
    L = rng.standard_normal((3, 5))
    ninf = np.full((3, 5), -np.inf)
    Om, Lm = orc.lse_merge(O, L, np.full_like(O, 7.0), ninf)
    np.testing.assert_array_equal(Lm, L)
    np.testing.assert_allclose(Om, O, rtol=1e-15, atol=0)
    Oz, Lz = orc.lse_merge(np.zeros_like(O), ninf, np.zeros_like(O), ninf)
    assert np.all(np.isneginf(Lz)) and not np.any(Oz)


def test_zigzag_ring_schedule_reproduces_causal_attention():
    """Every device's blocks of the zigzag ring (causal on its own chunks, full on earlier ones,
    skipped on later ones), merged in ring order, give causal attention over the whole sequence;
    and every device computes the same number of blocks (the load balancing)."""
    import long_context_attention_upipe_gb300 as up
    P, C, Dh = 3, 7, 8
    S = 2 * P * C
    Q, K, V = rand_qkv(S, 2, 1, Dh, seed=32)
    scale = orc.default_scale(Dh)
    O, L = orc.attention_forward(Q, K, V, None, True, scale)
    sched = up.ring_block_schedule(P)
    assert len({sum(len(b) for b in steps) for steps in sched}) == 1
    seen = set()
    Oacc = {c: np.zeros((2, C, Dh)) for c in range(2 * P)}
    Lacc = {c: np.full((2, C), -np.inf) for c in range(2 * P)}
    for steps in sched:
        for blocks in steps:
            for qc, kc, kind in blocks:
                assert kc <= qc and (kind == "causal") == (kc == qc)
                seen.add((qc, kc))
                q = Q[:, qc * C:(qc + 1) * C]
                Ob, Lb = orc.attention_forward(q, K[:, kc * C:(kc + 1) * C], V[:, kc * C:(kc + 1) * C], None,
                                               kind == "causal", scale)
                Oacc[qc], Lacc[qc] = orc.lse_merge(Oacc[qc], Lacc[qc], Ob, Lb)
    assert seen == {(a, b) for a in range(2 * P) for b in range(a + 1)}   # each block exactly once
    for c in range(2 * P):
        np.testing.assert_allclose(Oacc[c], O[:, c * C:(c + 1) * C], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(Lacc[c], L[:, c * C:(c + 1) * C], rtol=1e-12, atol=1e-12)


def test_zigzag_ring_blocks_reproduce_the_causal_backward():
    """The blocks of the zigzag ring, each with its query chunk's final log-sum-exp and
    D = dO . O, summed per chunk, give the gradients of causal attention over the whole sequence."""
    import long_context_attention_upipe_gb300 as up
    P, C, Dh = 2, 9, 8
    S = 2 * P * C
    Q, K, V = rand_qkv(S, 4, 2, Dh, seed=33)
    dO = np.random.default_rng(34).standard_normal(Q.shape)
    scale = orc.default_scale(Dh)
    O, L = orc.attention_forward(Q, K, V, None, True, scale)
    dQ, dK, dV = orc.attention_backward(Q, K, V, dO, None, True, scale)
    D = (dO * O).sum(axis=2)
    gq, gk, gv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for steps in up.ring_block_schedule(P):
        for blocks in steps:
            for qc, kc, kind in blocks:
                qs, ks = slice(qc * C, (qc + 1) * C), slice(kc * C, (kc + 1) * C)
                bq, bk, bv = orc.attention_backward_block(Q[:, qs], K[:, ks], V[:, ks], dO[:, qs], L[:, qs], D[:, qs],
                                                          kind == "causal", scale)
                gq[:, qs] += bq
                gk[:, ks] += bk
                gv[:, ks] += bv
    np.testing.assert_allclose(gq, dQ, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(gk, dK, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(gv, dV, rtol=1e-10, atol=1e-11)


def _packed(S, lengths):
    return np.repeat(np.arange(len(lengths)), lengths)[:S] if lengths else None


@pytest.mark.parametrize("P,C,lengths", [(1, 5, None), (2, 5, None), (3, 4, None), (4, 3, None),
                                         (3, 4, [5, 1, 9, 9]), (4, 6, [20, 3, 1, 24])])
def test_ring_steps_partition_the_causal_mask(P, C, lengths):
    """Over its P steps, device r sees every (query, key) pair of the causal + segment mask on its
    rows exactly once (the steps' key shards are disjoint and cover the sequence), and without
    segments every device sees the same number of pairs (the zigzag balance)."""
    S = 2 * P * C
    seg = _packed(S, lengths)
    full = orc.visibility(seg, np.arange(S), np.arange(S), True)
    counts = []
    for r in range(P):
        qpos = orc.zigzag_positions(P, C, r)
        got = np.zeros((2 * C, S), dtype=np.int64)
        for s in range(P):
            kpos = orc.zigzag_positions(P, C, (r - s) % P)
            got[:, kpos] += orc.ring_step_visibility(P, C, r, s, seg)
        np.testing.assert_array_equal(got, full[qpos].astype(np.int64))
        counts.append(int(got.sum()))
    assert sorted(np.concatenate([orc.zigzag_positions(P, C, r) for r in range(P)]).tolist()) == list(range(S))
    if lengths is None:
        assert len(set(counts)) == 1


@pytest.mark.parametrize("P,C,lengths", [(3, 4, None), (4, 6, [20, 3, 1, 24]), (2, 7, [2, 2, 24])])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_step_rows_and_columns_are_intervals(P, C, lengths, causal):
    """In every ring step each query row sees one interval of the visiting shard's rows and each
    key row is seen by one interval of queries, with both ends non-decreasing: the shape the tile
    table and the kernels' per-row masks rely on."""
    seg = _packed(2 * P * C, lengths)
    for r in range(P):
        for s in range(P):
            vis = orc.ring_step_visibility(P, C, r, s, seg, causal)
            for m in (vis, vis.T):
                lo_prev, hi_prev = -1, -1
                for row in m:
                    nz = np.nonzero(row)[0]
                    if nz.size == 0:
                        continue
                    assert nz.size == nz[-1] - nz[0] + 1
                    assert nz[0] >= lo_prev and nz[-1] >= hi_prev
                    lo_prev, hi_prev = nz[0], nz[-1]


@pytest.mark.parametrize("C,lengths", [(64, None), (200, None), (150, [100, 1, 120, 79])])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_step_table_of_a_one_device_ring_is_the_plain_table(C, lengths, causal):
    """A ring of one device is the plain sequence: its step table equals the skip table of
    2C rows computed from the row intervals."""
    seg = _packed(2 * C, lengths)
    q_rows, kv_rows = orc.ring_step_table(1, C, 0, 0, seg, causal)
    want_q, want_kv, _ = orc.tile_table(2 * C, seg, causal)
    np.testing.assert_array_equal(q_rows, want_q)
    np.testing.assert_array_equal(kv_rows, want_kv)


# ------------------------------------------------------------------------------------------
# 6. tile-skip table
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 7, 128, 129, 300, 512, 700])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_counts_match_elementwise_bruteforce(S, causal):
    rng = np.random.default_rng(S + 1000 * causal)
    for trial in range(4):
        seg = None if trial == 0 else random_segments(S, rng)
        brute = orc.tile_classes_bruteforce(S, seg, causal, B=128)
        n = brute.shape[0]
        cls = orc.classes_from_counts(S, orc.tile_counts(S, seg, causal), np.arange(n))
        np.testing.assert_array_equal(cls, brute)
        q_rows, kv_rows, tot = orc.tile_table(S, seg, causal)
        assert tot.tolist() == [int((brute == 1).sum()), int((brute == 2).sum())]
        for i in range(n):  # every class is what the ranges say
            b, fb, fe, e = q_rows[i]
            for j in range(n):
                want = 0 if not (b <= j < e) else (2 if fb <= j < fe else 1)
                assert brute[i, j] == want
            b, fb, fe, e = kv_rows[i]
            for j in range(n):
                want = 0 if not (b <= j < e) else (2 if fb <= j < fe else 1)
                assert brute[j, i] == want
        sel = np.array(sorted({0, n - 1, n // 2}))
        q2, k2, _ = orc.tile_table(S, seg, causal, q_tiles=sel, kv_tiles=sel)
        np.testing.assert_array_equal(q2, q_rows[sel])
        np.testing.assert_array_equal(k2, kv_rows[sel])


def test_tile_table_single_segment_causal_closed_form():
    for S in (128, 1000, 5 * 128 + 64):
        n = -(-S // 128)
        q_rows, kv_rows, tot = orc.tile_table(S, None, True)
        for i in range(n):
            assert q_rows[i].tolist() == ([0, 0, i, i + 1] if i > 0 else [0, 1, 1, 1])
            assert kv_rows[i].tolist() == ([i, i + 1, n, n] if i < n - 1 else [i, i + 1, i + 1, i + 1])
        assert tot.tolist() == [n, n * (n - 1) // 2]
        assert tot.sum() == n * (n + 1) // 2


def test_tile_table_packed_tiny_case():
    """The tiny workload: 300 + 212 tokens in 128-tiles, causal."""
    seg = ui.segments_from_lengths([300, 212])
    q_rows, kv_rows, tot = orc.tile_table(512, seg, True)
    assert q_rows.tolist() == [[0, 1, 1, 1], [0, 0, 1, 2], [0, 3, 3, 3], [2, 4, 4, 4]]
    assert kv_rows.tolist() == [[0, 1, 2, 3], [1, 3, 3, 3], [2, 4, 4, 4], [3, 4, 4, 4]]
    assert tot.tolist() == [7, 1]


def test_visible_pairs_match_tile_counts():
    w = ui.workload("tiny")
    counts = orc.tile_counts(w.S, w.segments(), True)
    assert counts.sum() == w.visible_pairs() == 300 * 301 // 2 + 212 * 213 // 2


def test_noncontiguous_segments_rejected():
    with pytest.raises(ValueError):
        orc.tile_table(10, np.array([0, 0, 1, 1, 0, 2, 2, 2, 2, 2], dtype=np.int32), True)


# ------------------------------------------------------------------------------------------
# 7. the bf16 input path: the oracle widens bf16 exactly
# ------------------------------------------------------------------------------------------

def test_bf16_widening_is_exact():
    vals = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x3C23, 0x7F7F], dtype=np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, 3.140625, 0.0099487304687500, 3.3895313892515355e38]
    np.testing.assert_array_equal(orc.bf16_bits_to_f64(vals), want)
    t = torch.tensor(vals.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(orc.bf16_bits_to_f64(vals), t)


# ------------------------------------------------------------------------------------------
# 8. the sequence-tiled feed-forward step (SwiGLU MLP)
# ------------------------------------------------------------------------------------------

def _mlp_inputs(S=24, d=16, F=40, seed=3):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((S, d))
    Wgu = rng.standard_normal((2 * F, d)) * 0.3
    Wd = rng.standard_normal((d, F)) * 0.3
    dY = rng.standard_normal((S, d))
    return X, Wgu, Wd, dY


def test_silu_special_values():
    assert orc.silu(0.0) == 0.0
    assert orc.silu_grad(0.0) == 0.5
    np.testing.assert_allclose(orc.silu(np.array([30.0, -30.0])), [30.0, -30.0 * math.exp(-30.0)], rtol=1e-12)
    assert orc.silu(-1e4) == 0.0                       # no overflow warning turns into a NaN
    # derivative against a central difference
    x = np.linspace(-6, 6, 97)
    h = 1e-6
    np.testing.assert_allclose(orc.silu_grad(x), (orc.silu(x + h) - orc.silu(x - h)) / (2 * h), atol=1e-8)


def test_mlp_matches_torch_autograd():
    X, Wgu, Wd, dY = _mlp_inputs()
    F = Wgu.shape[0] // 2
    tX, tW, tD = (torch.tensor(a, requires_grad=True) for a in (X, Wgu, Wd))
    Y = (torch.nn.functional.silu(tX @ tW[:F].T) * (tX @ tW[F:].T)) @ tD.T
    Y.backward(torch.tensor(dY))
    np.testing.assert_allclose(orc.mlp_forward(X, Wgu, Wd), Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    dX, dW, dD = orc.mlp_backward(X, Wgu, Wd, dY)
    for got, want in ((dX, tX.grad), (dW, tW.grad), (dD, tD.grad)):
        np.testing.assert_allclose(got, want.numpy(), rtol=1e-11, atol=1e-11)


def test_mlp_gradients_finite_differences():
    X, Wgu, Wd, dY = _mlp_inputs(S=6, d=5, F=7, seed=11)
    dX, dW, dD = orc.mlp_backward(X, Wgu, Wd, dY)
    loss = lambda X_, W_, D_: float((orc.mlp_forward(X_, W_, D_) * dY).sum())
    h = 1e-6
    for arr, grad, which in ((X, dX, 0), (Wgu, dW, 1), (Wd, dD, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            args1, args2 = [X, Wgu, Wd], [X, Wgu, Wd]
            args1[which], args2[which] = a1, a2
            num[idx] = (loss(*args1) - loss(*args2)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7)


def test_mlp_closed_forms_and_row_independence():
    X, Wgu, Wd, dY = _mlp_inputs()
    F = Wgu.shape[0] // 2
    # up projection zero: the output and every gradient but dWu vanish
    W0 = Wgu.copy()
    W0[F:] = 0.0
    assert not np.any(orc.mlp_forward(X, W0, Wd))
    dX, dW, dD = orc.mlp_backward(X, W0, Wd, dY)
    assert not np.any(dX) and not np.any(dW[:F]) and not np.any(dD)
    assert np.any(dW[F:])
    # one row, one hidden unit, by hand
    x, wg, wu, wd = 0.7, -1.3, 0.4, 2.0
    want = (wg * x / (1 + math.exp(-wg * x))) * (wu * x) * wd
    got = orc.mlp_forward(np.array([[x]]), np.array([[wg], [wu]]), np.array([[wd]]))
    assert abs(got[0, 0] - want) < 1e-15
    # rows are independent: perturbing other rows leaves a row's output unchanged (the tiling premise)
    Y = orc.mlp_forward(X, Wgu, Wd)
    X2 = X.copy()
    X2[5:] += 1.0
    np.testing.assert_array_equal(orc.mlp_forward(X2, Wgu, Wd)[:5], Y[:5])
