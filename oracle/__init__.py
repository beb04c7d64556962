"""fp64 CPU oracle for head-chunked causal self-attention with packed segments.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its binding) never calls it and
shares no code with it; the only thing both sides share is the seeded input generator
(``upipe_inputs``), which holds none of the arithmetic below.

What is computed, and where it is stated:

* Attention is computed per head over the whole sequence ("Road to 5 Million Tokens" podcast
  summary, chapter on DeepSpeed Ulysses; neuro-slop.ru transcript, quiz answer on Ulysses:
  each head is computed whole, which is why flash attention applies).  The pages never write
  the formula; this oracle takes the textbook scaled dot product softmax(Q K^T * scale + M) V
  with scale = 1/sqrt(Dh), the plainest reading.
* Compute is quadratic because every element interacts with every other (podcast summary,
  概要 "兩個瓶頸"; transcript quiz, first answer).
* Head chunking changes only which heads run together, not the result (podcast summary,
  章節 "分批算 heads"; transcript, quiz answer on U-Pipe).  So the oracle has no chunks: it
  computes every head at once, which is the result the chunked method must reproduce.
* The mask: causal, and packed sequences attend only inside their own segment; blocks with no
  visible pair are skippable (MaxText long-context article on techmoon.xyz, paragraph on Splash
  attention: fully masked blocks are skipped and packing needs no padding).  GQA is in the
  supported set (same paragraph); query head h reads KV head h // (Hq / Hkv).
* The layer: Q/K/V projections from the hidden states, attention, output projection
  (podcast summary, Q&A chapter: UPipe concerns the layer's query, key and value matrices).

All inputs are bf16 bit patterns widened exactly to float64; nothing is rounded in between.
Matrix products use numpy's float64 matmul as a library step.  Gradients follow the chain rule
of the same definition.

parity: every function here is pinned by tests/test_oracle.py (brute-force per-row softmax,
torch float64 autograd, central finite differences, closed forms, invariants, brute-force
tile classification).  No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf
TILE = 128  # tile edge of the skip table (rows and columns)


# ----------------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------------

def bf16_bits_to_f64(u16) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u16 = np.asarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def default_scale(Dh: int) -> float:
    return 1.0 / np.sqrt(Dh)


def visibility(seg, rows, cols, causal: bool) -> np.ndarray:
    """vis[r, c] = (seg[rows[r]] == seg[cols[c]]) and (not causal or cols[c] <= rows[r]).

    `seg` None means a single segment.  This is the mask definition; everything else uses it.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    if seg is None:
        vis = np.ones((rows.size, cols.size), dtype=bool)
    else:
        seg = np.asarray(seg)
        vis = seg[rows][:, None] == seg[cols][None, :]
    if causal:
        vis &= cols[None, :] <= rows[:, None]
    return vis


def split_wqkv(Wqkv: np.ndarray, Hq: int, Hkv: int, Dh: int):
    """Rows of Wqkv are [Q heads | K heads | V heads], Dh rows per head (nn.Linear layout)."""
    Wq = Wqkv[: Hq * Dh]
    Wk = Wqkv[Hq * Dh: (Hq + Hkv) * Dh]
    Wv = Wqkv[(Hq + Hkv) * Dh: (Hq + 2 * Hkv) * Dh]
    return Wq, Wk, Wv


def heads(M: np.ndarray, H: int, Dh: int) -> np.ndarray:
    """[S, H*Dh] -> [H, S, Dh]."""
    S = M.shape[0]
    return M.reshape(S, H, Dh).transpose(1, 0, 2)


def unheads(M: np.ndarray) -> np.ndarray:
    """[H, S, Dh] -> [S, H*Dh]."""
    H, S, Dh = M.shape
    return M.transpose(1, 0, 2).reshape(S, H * Dh)


# ----------------------------------------------------------------------------------------------
# attention, per head, over the whole sequence
# ----------------------------------------------------------------------------------------------

def attention_forward(Q, K, V, seg, causal: bool, scale: float, rows=None, row_block: int = 1024):
    """O_h[i] = sum_j P_ij V_kv[j],  P_ij = exp(s_ij - m_i) / l_i over visible j,
    s_ij = scale * Q_h[i] . K_kv[j],  m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i),
    LSE_h[i] = m_i + ln l_i  (natural log).  kv = h // (Hq / Hkv).

    Q: [Hq, S, Dh]; K, V: [Hkv, S, Dh] (float64).  `rows` selects query rows (default: all);
    rows are independent, so they are taken `row_block` at a time to bound memory.
    A row that sees no key gets O = 0 and LSE = -inf.
    Returns O [Hq, R, Dh], LSE [Hq, R].
    """
    Hq, S, Dh = Q.shape
    Hkv = K.shape[0]
    g = Hq // Hkv
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(K.shape[1])
    O = np.zeros((Hq, rows.size, Dh))
    LSE = np.full((Hq, rows.size), NEG_INF)
    for r0 in range(0, rows.size, row_block):
        rr = rows[r0: r0 + row_block]
        vis = visibility(seg, rr, cols, causal)
        any_vis = vis.any(axis=1)
        for h in range(Hq):
            kv = h // g
            s = scale * (Q[h, rr] @ K[kv].T)
            s = np.where(vis, s, NEG_INF)
            m = np.where(any_vis, s.max(axis=1), 0.0)
            e = np.where(vis, np.exp(s - m[:, None]), 0.0)
            l = e.sum(axis=1)
            P = np.divide(e, l[:, None], out=np.zeros_like(e), where=l[:, None] > 0)
            O[h, r0: r0 + rr.size] = P @ V[kv]
            with np.errstate(divide="ignore"):
                LSE[h, r0: r0 + rr.size] = np.where(any_vis, m + np.log(l), NEG_INF)
    return O, LSE


def attention_backward(Q, K, V, dO, seg, causal: bool, scale: float, row_block: int = 1024):
    """Gradients of sum(dO * O) for the attention above (chain rule):
    D_i = dO_h[i] . O_h[i];  dP_ij = dO_h[i] . V_kv[j];  dS_ij = P_ij (dP_ij - D_i);
    dQ_h[i] = scale sum_j dS_ij K_kv[j];
    dK_kv[j] = scale sum_{h in group(kv)} sum_i dS_ij Q_h[i];
    dV_kv[j] = sum_{h in group(kv)} sum_i P_ij dO_h[i].
    Returns dQ [Hq,S,Dh], dK, dV [Hkv,S,Dh].
    """
    Hq, S, Dh = Q.shape
    Hkv = K.shape[0]
    g = Hq // Hkv
    cols = np.arange(S)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for r0 in range(0, S, row_block):
        rr = np.arange(r0, min(S, r0 + row_block))
        vis = visibility(seg, rr, cols, causal)
        any_vis = vis.any(axis=1)
        for h in range(Hq):
            kv = h // g
            s = scale * (Q[h, rr] @ K[kv].T)
            s = np.where(vis, s, NEG_INF)
            m = np.where(any_vis, s.max(axis=1), 0.0)
            e = np.where(vis, np.exp(s - m[:, None]), 0.0)
            l = e.sum(axis=1)
            P = np.divide(e, l[:, None], out=np.zeros_like(e), where=l[:, None] > 0)
            O = P @ V[kv]
            D = (dO[h, rr] * O).sum(axis=1)
            dP = dO[h, rr] @ V[kv].T
            dS = P * (dP - D[:, None])
            dQ[h, rr] = scale * (dS @ K[kv])
            dK[kv] += scale * (dS.T @ Q[h, rr])
            dV[kv] += P.T @ dO[h, rr]
    return dQ, dK, dV


# ----------------------------------------------------------------------------------------------
# the layer: projections -> attention -> output projection
# ----------------------------------------------------------------------------------------------

def _widen(a):
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def layer_forward(X, Wqkv, Wo, seg, Hq, Hkv, Dh, causal=True, scale=None, return_all=False):
    """Y = [O_0 ... O_{Hq-1}] Wo^T with Q_h = X Wq_h^T, K_kv = X Wk_kv^T, V_kv = X Wv_kv^T.

    X [S,d], Wqkv [(Hq+2Hkv)Dh, d], Wo [d, Hq Dh]: bf16 bit patterns (uint16) or floats.
    Returns Y [S,d] and LSE [Hq,S] in float64 (and the intermediates if asked).
    """
    X, Wqkv, Wo = _widen(X), _widen(Wqkv), _widen(Wo)
    scale = default_scale(Dh) if scale is None else scale
    Wq, Wk, Wv = split_wqkv(Wqkv, Hq, Hkv, Dh)
    Q = heads(X @ Wq.T, Hq, Dh)
    K = heads(X @ Wk.T, Hkv, Dh)
    V = heads(X @ Wv.T, Hkv, Dh)
    O, LSE = attention_forward(Q, K, V, seg, causal, scale)
    Y = unheads(O) @ Wo.T
    if return_all:
        return Y, LSE, dict(Q=Q, K=K, V=V, O=O)
    return Y, LSE


def project_kv(X_keys, Wk, Wv, Hkv, Dh, row_block: int = 65536):
    """K_kv = X Wk_kv^T and V_kv = X Wv_kv^T for the rows of X_keys ([n, d], bf16 bit patterns or
    floats), widened and multiplied `row_block` rows at a time so that a million-row X never
    exists in float64 at once.  Returns K, V [Hkv, n, Dh]."""
    n = np.asarray(X_keys).shape[0]
    K = np.empty((Hkv, n, Dh))
    V = np.empty((Hkv, n, Dh))
    for a in range(0, n, row_block):
        Xb = _widen(X_keys[a: a + row_block])
        K[:, a: a + Xb.shape[0]] = heads(Xb @ Wk.T, Hkv, Dh)
        V[:, a: a + Xb.shape[0]] = heads(Xb @ Wv.T, Hkv, Dh)
    return K, V


def layer_forward_rows(X_rows, X_keys, key_index, rows, Wqkv, Wo, seg, Hq, Hkv, Dh, causal=True,
                       scale=None):
    """Output rows `rows` of the layer, for long sequences.

    X_rows [R, d] are the hidden states of the query rows; X_keys [n, d] those of the key
    positions `key_index` (sorted), which must include every key any of the rows can see.
    Returns Y [R, d] and LSE [Hq, R].
    """
    Wq, Wk, Wv = split_wqkv(_widen(Wqkv), Hq, Hkv, Dh)
    K, V = project_kv(X_keys, Wk, Wv, Hkv, Dh)
    return layer_forward_rows_kv(X_rows, rows, K, V, key_index, Wqkv, Wo, seg, Hq, Hkv, Dh, causal, scale)


def layer_forward_rows_kv(X_rows, rows, K, V, key_index, Wqkv, Wo, seg, Hq, Hkv, Dh, causal=True, scale=None):
    """As layer_forward_rows, with the keys' K, V [Hkv, n, Dh] (float64, from project_kv) given
    instead of their hidden states, so that a caller can project a multi-million-key sequence
    block by block once and reuse it."""
    X_rows, Wqkv, Wo = _widen(X_rows), _widen(Wqkv), _widen(Wo)
    scale = default_scale(Dh) if scale is None else scale
    rows = np.asarray(rows, dtype=np.int64)
    key_index = np.asarray(key_index, dtype=np.int64)
    Wq, _, _ = split_wqkv(Wqkv, Hq, Hkv, Dh)
    Q = heads(X_rows @ Wq.T, Hq, Dh)
    g = Hq // Hkv
    O = np.zeros((Hq, rows.size, Dh))
    LSE = np.full((Hq, rows.size), NEG_INF)
    vis = visibility(seg, rows, key_index, causal) if seg is not None else (
        (key_index[None, :] <= rows[:, None]) if causal else np.ones((rows.size, key_index.size), bool))
    any_vis = vis.any(axis=1)
    for h in range(Hq):
        kv = h // g
        s = np.where(vis, scale * (Q[h] @ K[kv].T), NEG_INF)
        m = np.where(any_vis, s.max(axis=1), 0.0)
        e = np.where(vis, np.exp(s - m[:, None]), 0.0)
        l = e.sum(axis=1)
        P = np.divide(e, l[:, None], out=np.zeros_like(e), where=l[:, None] > 0)
        O[h] = P @ V[kv]
        with np.errstate(divide="ignore"):
            LSE[h] = np.where(any_vis, m + np.log(l), NEG_INF)
    return unheads(O) @ Wo.T, LSE


def layer_backward(X, Wqkv, Wo, seg, dY, Hq, Hkv, Dh, causal=True, scale=None, return_all=False):
    """Gradients of sum(dY * Y) for the layer above:
    dO = dY Wo (split per head); dWo = dY^T [O_0 ... O_{Hq-1}];
    (dQ, dK, dV) from attention_backward; dQKV = [dQ | dK | dV] (row order of Wqkv);
    dX = dQKV Wqkv; dWqkv = dQKV^T X.
    Returns dX [S,d], dWqkv, dWo (float64).
    """
    X, Wqkv, Wo, dY = _widen(X), _widen(Wqkv), _widen(Wo), _widen(dY)
    scale = default_scale(Dh) if scale is None else scale
    Wq, Wk, Wv = split_wqkv(Wqkv, Hq, Hkv, Dh)
    Q = heads(X @ Wq.T, Hq, Dh)
    K = heads(X @ Wk.T, Hkv, Dh)
    V = heads(X @ Wv.T, Hkv, Dh)
    O, _ = attention_forward(Q, K, V, seg, causal, scale)
    dOcat = dY @ Wo
    dWo = dY.T @ unheads(O)
    dO = heads(dOcat, Hq, Dh)
    dQ, dK, dV = attention_backward(Q, K, V, dO, seg, causal, scale)
    dQKV = np.concatenate([unheads(dQ), unheads(dK), unheads(dV)], axis=1)
    dX = dQKV @ Wqkv
    dWqkv = dQKV.T @ X
    if return_all:
        return dX, dWqkv, dWo, dict(dQ=dQ, dK=dK, dV=dV, dO=dO, O=O)
    return dX, dWqkv, dWo


def layer_backward_rows(X, Wqkv, Wo, seg, dY_rows, rows, Hq, Hkv, Dh, causal=True, scale=None):
    """layer_backward for an upstream gradient dY that is zero on every row except `rows`
    (sorted, distinct), where it equals dY_rows [R, d].  The formulas are those of
    layer_backward; the rows of zero dY contribute exact zeros to every sum (dO, D, dS and P^T dO
    vanish there), so they are left out:
    dO_h[i] = (dY Wo)_h[i] and O_h[i] for i in rows only; dWo = dY_rows^T [O_0 ... O_{Hq-1}](rows);
    for i in rows: D_i = dO_h[i] . O_h[i], dP_ij = dO_h[i] . V_kv[j], dS_ij = P_ij (dP_ij - D_i),
    dQ_h[i] = scale sum_j dS_ij K_kv[j]; dK_kv[j] = scale sum_h sum_{i in rows} dS_ij Q_h[i],
    dV_kv[j] = sum_h sum_{i in rows} P_ij dO_h[i]; dQKV = [dQ | dK | dV] (dQ zero off `rows`);
    dX = dQKV Wqkv; dWqkv = dQKV^T X.  X [S, d] is needed whole (every key and dWqkv).
    Returns dX [S, d], dWqkv, dWo (float64)."""
    X, Wqkv, Wo, dY_rows = _widen(X), _widen(Wqkv), _widen(Wo), _widen(dY_rows)
    scale = default_scale(Dh) if scale is None else scale
    rows = np.asarray(rows, dtype=np.int64)
    S = X.shape[0]
    g = Hq // Hkv
    Wq, Wk, Wv = split_wqkv(Wqkv, Hq, Hkv, Dh)
    Qr = heads(X[rows] @ Wq.T, Hq, Dh)
    K = heads(X @ Wk.T, Hkv, Dh)
    V = heads(X @ Wv.T, Hkv, Dh)
    vis = visibility(seg, rows, np.arange(S), causal)
    any_vis = vis.any(axis=1)
    dOr = heads(dY_rows @ Wo, Hq, Dh)
    Or = np.zeros((Hq, rows.size, Dh))
    dQr = np.zeros((Hq, rows.size, Dh))
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        kv = h // g
        s = np.where(vis, scale * (Qr[h] @ K[kv].T), NEG_INF)
        m = np.where(any_vis, s.max(axis=1), 0.0)
        e = np.where(vis, np.exp(s - m[:, None]), 0.0)
        l = e.sum(axis=1)
        P = np.divide(e, l[:, None], out=np.zeros_like(e), where=l[:, None] > 0)
        Or[h] = P @ V[kv]
        D = (dOr[h] * Or[h]).sum(axis=1)
        dP = dOr[h] @ V[kv].T
        dS = P * (dP - D[:, None])
        dQr[h] = scale * (dS @ K[kv])
        dK[kv] += scale * (dS.T @ Qr[h])
        dV[kv] += P.T @ dOr[h]
    dWo = dY_rows.T @ unheads(Or)
    dQKV = np.zeros((S, (Hq + 2 * Hkv) * Dh))
    dQKV[rows, : Hq * Dh] = unheads(dQr)
    dQKV[:, Hq * Dh: (Hq + Hkv) * Dh] = unheads(dK)
    dQKV[:, (Hq + Hkv) * Dh:] = unheads(dV)
    return dQKV @ Wqkv, dQKV.T @ X, dWo


def lse_merge(O_a, L_a, O_b, L_b):
    """Attention over the union of two disjoint key sets from the per-set results, as ring (P2P)
    context parallelism combines the key/value blocks that visit a device (MaxText long-context
    article on techmoon.xyz, table of the four context-parallel strategies, row "P2P (Ring)").
    With L the natural-log log-sum-exp of a row's scores over a key set and O its softmax-weighted
    values: L = log(e^{L_a} + e^{L_b}), O = (e^{L_a} O_a + e^{L_b} O_b) / e^{L}.  A side with
    L = -inf (no key) contributes nothing; both -inf gives O = 0, L = -inf.
    O_*: [..., Dh], L_*: [...] (float64)."""
    O_a, L_a, O_b, L_b = (np.asarray(x, dtype=np.float64) for x in (O_a, L_a, O_b, L_b))
    L = np.logaddexp(L_a, L_b)
    ok = np.isfinite(L)
    with np.errstate(invalid="ignore", over="ignore"):
        wa = np.where(ok & np.isfinite(L_a), np.exp(L_a - np.where(ok, L, 0.0)), 0.0)
        wb = np.where(ok & np.isfinite(L_b), np.exp(L_b - np.where(ok, L, 0.0)), 0.0)
    return wa[..., None] * O_a + wb[..., None] * O_b, L


def attention_backward_block(Q, K, V, dO, L, D, causal: bool, scale: float):
    """One key/value block's share of the attention backward when each row's softmax runs over more
    keys than the block holds (the ring's backward): with the row's final log-sum-exp L_h[i] and
    D_h[i] = dO_h[i] . O_h[i] of its final output, over the block's visible keys
    P_ij = exp(s_ij - L_i), dP_ij = dO_h[i] . V[j], dS_ij = P_ij (dP_ij - D_i); the block adds
    dQ_h[i] += scale sum_j dS_ij K[j], dK[j] += scale sum_{h,i} dS_ij Q_h[i], dV[j] += sum_{h,i} P_ij dO_h[i].
    Q, dO [Hq, R, Dh]; K, V [Hkv, C, Dh]; L, D [Hq, R]; positions as in attention_forward (row i and
    column j of the block; causal means j <= i).  Returns the block's dQ [Hq, R, Dh], dK, dV [Hkv, C, Dh]."""
    Hq, R, Dh = Q.shape
    Hkv, C = K.shape[0], K.shape[1]
    g = Hq // Hkv
    vis = visibility(None, np.arange(R), np.arange(C), causal)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for h in range(Hq):
        kv = h // g
        s = scale * (Q[h] @ K[kv].T)
        ok = vis & np.isfinite(L[h])[:, None]
        P = np.where(ok, np.exp(np.where(ok, s, 0.0) - np.where(np.isfinite(L[h]), L[h], 0.0)[:, None]), 0.0)
        dP = dO[h] @ V[kv].T
        dS = P * (dP - D[h][:, None])
        dQ[h] = scale * (dS @ K[kv])
        dK[kv] += scale * (dS.T @ Q[h])
        dV[kv] += P.T @ dO[h]
    return dQ, dK, dV


# ----------------------------------------------------------------------------------------------
# the feed-forward step beside the layer, cut into sequence tiles (Arctic sequence tiling)
# ----------------------------------------------------------------------------------------------
# The pages compute the loss and the MLP in pieces along the sequence so that no buffer has a
# multi-million-token axis ("Road to 5 Million Tokens" podcast summary, 概要 and 章節 on sequence
# tiling of the element-wise operations; neuro-slop.ru transcript, Полезные советы: loss and MLP
# can be computed in chunks).  Every row of an MLP is computed independently, so cutting the rows
# into tiles changes nothing: the oracle is the plain, untiled definition.  The pages do not
# write the MLP; for the Llama-3.1-shaped configurations it is the Llama feed-forward block,
# SwiGLU:  Y = (silu(X Wg^T) * (X Wu^T)) Wd^T,  silu(x) = x / (1 + e^-x).

def silu(x):
    """x * sigmoid(x), float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def silu_grad(x):
    """d silu / dx = sigmoid(x) (1 + x (1 - sigmoid(x)))."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        sg = 1.0 / (1.0 + np.exp(-x))
    return sg * (1.0 + x * (1.0 - sg))


def mlp_forward(X, Wgu, Wd, return_all=False):
    """SwiGLU feed-forward of every row of X [S, d]:  G = X Wg^T, U = X Wu^T (Wgu = [Wg; Wu],
    [2F, d], gate rows first, nn.Linear layout), A = silu(G) * U, Y = A Wd^T (Wd [d, F]).
    Inputs are bf16 bit patterns (uint16) or floats, widened exactly to float64."""
    X, Wgu, Wd = _widen(X), _widen(Wgu), _widen(Wd)
    F = Wgu.shape[0] // 2
    G = X @ Wgu[:F].T
    U = X @ Wgu[F:].T
    A = silu(G) * U
    Y = A @ Wd.T
    if return_all:
        return Y, dict(G=G, U=U, A=A)
    return Y


def mlp_backward(X, Wgu, Wd, dY):
    """Gradients of sum(dY * Y) for mlp_forward (chain rule):  dA = dY Wd,  dWd = dY^T A,
    dG = dA * U * silu'(G),  dU = dA * silu(G),  dX = dG Wg + dU Wu,  dWgu = [dG^T X; dU^T X].
    Returns dX [S, d], dWgu [2F, d], dWd [d, F] (float64)."""
    X, Wgu, Wd, dY = _widen(X), _widen(Wgu), _widen(Wd), _widen(dY)
    F = Wgu.shape[0] // 2
    G = X @ Wgu[:F].T
    U = X @ Wgu[F:].T
    A = silu(G) * U
    dA = dY @ Wd
    dWd = dY.T @ A
    dG = dA * U * silu_grad(G)
    dU = dA * silu(G)
    dX = dG @ Wgu[:F] + dU @ Wgu[F:]
    dWgu = np.concatenate([dG.T @ X, dU.T @ X], axis=0)
    return dX, dWgu, dWd


# ----------------------------------------------------------------------------------------------
# tile-skip table (Splash-style block skipping, MaxText article)
# ----------------------------------------------------------------------------------------------

EMPTY, PARTIAL, FULL = 0, 1, 2


def tile_classes_bruteforce(S: int, seg, causal: bool, B: int = TILE) -> np.ndarray:
    """cls[i, j] for B x B tiles by counting visible pairs element by element: EMPTY when no
    pair is visible, FULL when every in-range pair is, PARTIAL otherwise.  Small S only."""
    n = -(-S // B)
    vis = visibility(seg, np.arange(S), np.arange(S), causal)
    cls = np.zeros((n, n), dtype=np.int8)
    for i in range(n):
        for j in range(n):
            blk = vis[i * B: (i + 1) * B, j * B: (j + 1) * B]
            c = int(blk.sum())
            cls[i, j] = EMPTY if c == 0 else (FULL if c == blk.size else PARTIAL)
    return cls


def _row_intervals(S: int, seg, causal: bool):
    """For contiguous (non-decreasing) segment ids, row r sees exactly the columns
    [lo_r, hi_r]: lo_r = first position of r's segment, hi_r = r (causal) or the segment's last
    position.  Returns (lo, hi) as int64 arrays."""
    r = np.arange(S, dtype=np.int64)
    if seg is None:
        start = np.zeros(S, dtype=np.int64)
        end = np.full(S, S - 1, dtype=np.int64)
    else:
        seg = np.asarray(seg)
        if np.any(seg[1:] < seg[:-1]):
            raise ValueError("segment ids are not contiguous (must be non-decreasing)")
        new = np.ones(S, dtype=bool)
        new[1:] = seg[1:] != seg[:-1]
        start = np.maximum.accumulate(np.where(new, r, 0))
        last = np.ones(S, dtype=bool)
        last[:-1] = seg[:-1] != seg[1:]
        end = np.minimum.accumulate(np.where(last, r, S - 1)[::-1])[::-1]
    return start, (r if causal else end)


def tile_counts(S: int, seg, causal: bool, q_tiles=None, B: int = TILE) -> np.ndarray:
    """count[i, j] = number of visible (row, column) pairs in tile (i, j), summed row by row
    from the row intervals above.  `q_tiles` selects the tile rows (default: all)."""
    lo, hi = _row_intervals(S, seg, causal)
    n = -(-S // B)
    q_tiles = np.arange(n) if q_tiles is None else np.asarray(q_tiles, dtype=np.int64)
    c0 = np.arange(n, dtype=np.int64) * B
    c1 = np.minimum(c0 + B, S)  # exclusive
    out = np.zeros((q_tiles.size, n), dtype=np.int64)
    for a, i in enumerate(q_tiles):
        rr = np.arange(i * B, min(S, (i + 1) * B))
        width = np.minimum(hi[rr, None] + 1, c1[None, :]) - np.maximum(lo[rr, None], c0[None, :])
        out[a] = np.maximum(width, 0).sum(axis=0)
    return out


def tile_counts_cols(S: int, seg, causal: bool, kv_tiles, B: int = TILE) -> np.ndarray:
    """count[i, j] for the selected kv tiles j and every q tile i (the transpose view of
    tile_counts), from the same row intervals."""
    lo, hi = _row_intervals(S, seg, causal)
    n = -(-S // B)
    kv_tiles = np.asarray(kv_tiles, dtype=np.int64)
    starts = np.arange(n, dtype=np.int64) * B
    out = np.zeros((kv_tiles.size, n), dtype=np.int64)
    for a, j in enumerate(kv_tiles):
        c0, c1 = j * B, min(S, (j + 1) * B)
        width = np.maximum(np.minimum(hi + 1, c1) - np.maximum(lo, c0), 0)
        out[a] = np.add.reduceat(width, starts)
    return out


def classes_from_counts(S: int, counts: np.ndarray, q_tiles, kv_tiles=None, B: int = TILE) -> np.ndarray:
    """Classes of tiles (q_tiles[a], kv_tiles[b]) from their visible-pair counts[a, b]:
    EMPTY if 0, FULL if every in-range pair is visible, PARTIAL otherwise."""
    n = -(-S // B)
    q_tiles = np.asarray(q_tiles, dtype=np.int64)
    kv_tiles = np.arange(n) if kv_tiles is None else np.asarray(kv_tiles, dtype=np.int64)
    rows_in = np.minimum((q_tiles + 1) * B, S) - q_tiles * B
    cols_in = np.minimum((kv_tiles + 1) * B, S) - kv_tiles * B
    full = counts == rows_in[:, None] * cols_in[None, :]
    return np.where(counts == 0, EMPTY, np.where(full, FULL, PARTIAL)).astype(np.int8)


def ranges_from_classes(cls_rows: np.ndarray) -> np.ndarray:
    """Per tile row: {begin, full_begin, full_end, end} with non-empty tiles [begin, end),
    full tiles [full_begin, full_end) and partial tiles elsewhere in [begin, end); when a row
    has no full tile, full_begin = full_end = end.  Raises if the row is not of that shape."""
    out = np.zeros((cls_rows.shape[0], 4), dtype=np.int32)
    for a, c in enumerate(cls_rows):
        ne = np.nonzero(c != EMPTY)[0]
        fu = np.nonzero(c == FULL)[0]
        b, e = (int(ne[0]), int(ne[-1]) + 1) if ne.size else (0, 0)
        fb, fe = (int(fu[0]), int(fu[-1]) + 1) if fu.size else (e, e)
        if ne.size and (ne.size != e - b or (fu.size and fu.size != fe - fb)):
            raise ValueError("tile row is not a contiguous range")
        out[a] = (b, fb, fe, e)
    return out


def tile_table(S: int, seg, causal: bool, q_tiles=None, kv_tiles=None, B: int = TILE):
    """The skip table: q-major rows {kv_begin, kv_full_begin, kv_full_end, kv_end} for the
    selected q tiles, kv-major rows {q_begin, q_full_begin, q_full_end, q_end} for the selected
    kv tiles, and the totals {partial, full} when all q tiles are selected (else None)."""
    n = -(-S // B)
    all_q = q_tiles is None
    q_tiles = np.arange(n) if q_tiles is None else np.asarray(q_tiles, dtype=np.int64)
    cq = classes_from_counts(S, tile_counts(S, seg, causal, q_tiles, B), q_tiles, None, B)
    q_rows = ranges_from_classes(cq)
    totals = None
    if all_q:
        totals = np.array([(cq == PARTIAL).sum(), (cq == FULL).sum()], dtype=np.int64)
    kv_rows = None
    if all_q and kv_tiles is None:
        kv_rows = ranges_from_classes(cq.T)
    elif kv_tiles is not None:
        kv_tiles = np.asarray(kv_tiles, dtype=np.int64)
        counts = tile_counts_cols(S, seg, causal, kv_tiles, B)
        ck = classes_from_counts(S, counts.T, np.arange(n), kv_tiles, B).T
        kv_rows = ranges_from_classes(ck)
    return q_rows, kv_rows, totals


# ----------------------------------------------------------------------------------------------
# zigzag ring steps (MaxText long-context article: strategy table, row "P2P (Ring)", and the
# paragraph after it: the ring needs causal load balancing, which reorders the sequence)
# ----------------------------------------------------------------------------------------------

def zigzag_positions(P: int, C: int, r: int) -> np.ndarray:
    """Sequence positions of ring device r's rows: the 2P chunks of C rows are dealt so that
    device r holds chunk r and chunk 2P - 1 - r (one early, one late), in that order.  The pages
    name the balancing but not the deal; this pairing is the plainest one that gives every device
    the same causal work."""
    return np.concatenate([np.arange(r * C, (r + 1) * C), np.arange((2 * P - 1 - r) * C, (2 * P - r) * C)])


def ring_step_visibility(P: int, C: int, r: int, s: int, seg, causal: bool = True) -> np.ndarray:
    """vis[i, j]: does device r's row i see row j of the key/value shard that visits it at step s
    (the shard of device (r - s) mod P)?  The mask definition above, on the rows' positions."""
    src = (r - s) % P
    return visibility(seg, zigzag_positions(P, C, r), zigzag_positions(P, C, src), causal)


def ring_step_table(P: int, C: int, r: int, s: int, seg, causal: bool = True, B: int = TILE):
    """The skip-table rows of one ring step, by brute-force tile classification of the step's
    visibility (small C only): q-major rows of device r's query tiles over the visiting shard's
    key tiles, and kv-major rows of the visiting shard's key tiles over device r's query tiles."""
    vis = ring_step_visibility(P, C, r, s, seg, causal)
    S = 2 * C
    n = -(-S // B)
    cls = np.zeros((n, n), dtype=np.int8)
    for i in range(n):
        for j in range(n):
            blk = vis[i * B: (i + 1) * B, j * B: (j + 1) * B]
            c = int(blk.sum())
            cls[i, j] = EMPTY if c == 0 else (FULL if c == blk.size else PARTIAL)
    return ranges_from_classes(cls), ranges_from_classes(cls.T)


# ----------------------------------------------------------------------------------------------
# brute-force row softmax (a pin for the vectorised code above)
# ----------------------------------------------------------------------------------------------

def rowsoftmax_bruteforce(scores_row, visible_row):
    """Softmax of one row over its visible entries, one element at a time, in Python floats."""
    import math
    vals = [float(s) for s, v in zip(scores_row, visible_row) if v]
    if not vals:
        return [0.0] * len(scores_row), float("-inf")
    m = max(vals)
    tot = sum(math.exp(v - m) for v in vals)
    p = [math.exp(float(s) - m) / tot if v else 0.0 for s, v in zip(scores_row, visible_row)]
    return p, m + math.log(tot)
