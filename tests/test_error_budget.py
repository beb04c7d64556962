"""Where the full-size output bar comes from.

The parity bar for a bf16-in / fp32-accumulate output is max-abs 1e-2 beyond the output's own
bf16 rounding.  The layer's output is not one such contraction: at hidden 4096 it passes four
bf16-stored stages (Q/K/V after the projection, P before P V, O before the output projection,
then Y).  This test carries out the plain definition of the layer (the oracle's projections,
mask and softmax) with exactly those roundings and nothing else (round to nearest even, every
sum exact), on rows of the full 32K-token Llama-3.1-8B-shaped layer, and measures how far an
ideal implementation of that arithmetic lands from the float64 oracle:

  * the first 256 rows (keys 0..255) and three late rows that see 16K-32K keys;
  * Y beyond its own bf16 rounding, the relative Frobenius error of Y, and the log-sum-exp.

It pins the full-size bars of tests/test_gpu_fullsize.py to that arithmetic.  Measured here:
Y is 0.0156 beyond its rounding on the first rows (0.0011 on the late ones) and 4.2e-3 / 4.3e-3
relative Frobenius; the log-sum-exp moves by up to 0.011 absolute, 7.1e-3 relative to
max(1, |lse|).  So the ideal implementation already exceeds 1e-2 on Y (no path that stores
those stages in bf16 can meet that bar), stays below the 2e-2 the full-size tests use and below
the 5e-3 relative Frobenius bar; its log-sum-exp misses the small tests' 1e-3 absolute bar at
these score magnitudes but stays within the 1e-2 relative bar the full-size tests apply.
"""
import numpy as np
import pytest

import oracle as orc
import upipe_inputs as ui
from helpers import (FULL_LSE_REL, FULL_MLP_OUT_MAX_ABS, FULL_OUT_MAX_ABS, OUT_MAX_ABS, OUT_REL_FRO, max_abs_bf16_out,
                     rel_fro)


def bf16_round(x):
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to even)."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                     # x = m * 2^e, 0.5 <= |m| < 1
    q = np.ldexp(1.0, e - 8)               # spacing of bf16 values in [2^(e-1), 2^e)
    return np.where(x == 0, 0.0, np.rint(x / q) * q)


def test_bf16_round_is_round_to_nearest_even():
    assert bf16_round(1.0) == 1.0
    assert bf16_round(1.0 + 2 ** -8) == 1.0                  # tie -> even (1.0)
    assert bf16_round(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6    # tie -> even (odd neighbour is 1 + 2^-7)
    assert bf16_round(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    # against the generator's own bf16 rounding of the same values (an independent routine)
    rng = np.random.default_rng(0)
    v = rng.standard_normal(10000) * 10.0
    want = np.array([ui._host_lib().ug_bf16_rne_host(float(t)) for t in v], dtype=np.uint16)
    np.testing.assert_array_equal(bf16_round(v), ui.bf16_to_f64(want))


def rounded_layer_rows(rows, X, Wqkv, Wo, Hq, Hkv, Dh):
    """Y rows and LSE of the causal layer (one segment) with the GPU path's bf16 stage roundings:
    Q, K, V stored in bf16; P = exp(s - m) rounded to bf16 before P V while the row sum l takes
    the unrounded values; O = (sum_j bf16(P_ij) V_j) / l stored in bf16; Y = bf16(O_cat Wo^T)."""
    rows = np.asarray(rows)
    n_keys = int(rows.max()) + 1
    Wq, Wk, Wv = orc.split_wqkv(orc.bf16_bits_to_f64(Wqkv), Hq, Hkv, Dh)
    Wo = orc.bf16_bits_to_f64(Wo)
    scale = orc.default_scale(Dh)
    K, V = orc.project_kv(X[:n_keys], Wk, Wv, Hkv, Dh)
    K, V = bf16_round(K), bf16_round(V)
    Q = bf16_round(orc.heads(orc.bf16_bits_to_f64(X[rows]) @ Wq.T, Hq, Dh))
    g = Hq // Hkv
    vis = orc.visibility(None, rows, np.arange(n_keys), True)
    O = np.zeros((Hq, rows.size, Dh))
    L = np.zeros((Hq, rows.size))
    for h in range(Hq):
        s = np.where(vis, scale * (Q[h] @ K[h // g].T), -np.inf)
        m = s.max(axis=1)
        p = np.where(vis, np.exp(s - m[:, None]), 0.0)
        l = p.sum(axis=1)
        O[h] = bf16_round((bf16_round(p) @ V[h // g]) / l[:, None])
        L[h] = m + np.log(l)
    return bf16_round(orc.unheads(O) @ Wo.T), L


@pytest.fixture(scope="module")
def budget():
    w = ui.workload("llama8b_32k")
    S, d, Hq, Hkv, Dh = w.S, w.d, w.Hq, w.Hkv, w.Dh
    X = ui.normal_bf16(S * d, ui.TID_X).reshape(S, d)
    W = ui.normal_bf16((Hq + 2 * Hkv) * Dh * d, ui.TID_WQKV, ui.W_STD).reshape(-1, d)
    Wo = ui.normal_bf16(d * Hq * Dh, ui.TID_WO, ui.W_STD).reshape(d, -1)
    out = []
    for rows in (np.arange(256), np.array([16383, S - 2, S - 1])):
        Y_sim, L_sim = rounded_layer_rows(rows, X, W, Wo, Hq, Hkv, Dh)
        n_keys = int(rows.max()) + 1
        Y_ref, L_ref = orc.layer_forward_rows(X[rows], X[:n_keys], np.arange(n_keys), rows, W, Wo, None,
                                              Hq, Hkv, Dh, True)
        out.append((Y_sim, L_sim, Y_ref, L_ref))
    return out


def test_full_size_output_bar_follows_from_the_bf16_stages(budget):
    errs = [max_abs_bf16_out(Y_sim, Y_ref) for Y_sim, _, Y_ref, _ in budget]
    fro = [rel_fro(Y_sim, Y_ref) for Y_sim, _, Y_ref, _ in budget]
    worst = max(errs)
    # an exact implementation of the stated roundings already misses the single-contraction bar ...
    assert worst > OUT_MAX_ABS, errs
    # ... by about 0.0156 on the first rows (fewest keys, so the least averaging of P's rounding);
    # the full-size bar is that figure rounded up to 2e-2, leaving a fifth of it for the GPU's own
    # summation order
    assert worst <= 0.8 * FULL_OUT_MAX_ABS, errs
    assert max(fro) <= 0.9 * OUT_REL_FRO, fro


def test_full_size_lse_bar_follows_from_the_bf16_stages(budget):
    abs_err = max(float(np.abs(L_sim - L_ref).max()) for _, L_sim, _, L_ref in budget)
    rel_err = max(float((np.abs(L_sim - L_ref) / np.maximum(1.0, np.abs(L_ref))).max())
                  for _, L_sim, _, L_ref in budget)
    assert rel_err <= 0.75 * FULL_LSE_REL, rel_err
    assert abs_err > 1e-3, abs_err          # why the small tests' 1e-3 absolute bar is not used here


def test_full_size_mlp_bar_follows_from_the_bf16_stages():
    """The sequence-tiled SwiGLU MLP at the Llama-3.1-8B shape (hidden 4096, ffn 14336) stores the
    gate/up projection H and A = silu(G) U in bf16, then Y.  Exactly those roundings (nothing else)
    on the rows tests/test_gpu_mlp.py checks land 0.029 beyond Y's rounding from the fp64 oracle,
    with a relative Frobenius error of 3.5e-3: above the 2e-2 of the attention layer, within 0.8 of
    the 4e-2 the MLP test uses, and below the 5e-3 relative bar."""
    S, d, F, T = 32768, 4096, 14336, 4096
    rows = np.array([0, 1, T - 1, T, 2 * T + 5, S // 2, S - T - 1, S - T, S - 2, S - 1])
    X = ui.normal_bf16_rows(rows, d, ui.TID_X)
    Wgu = ui.normal_bf16(2 * F * d, 6, ui.W_STD).reshape(2 * F, d)
    Wd = ui.normal_bf16(d * F, 7, ui.W_STD).reshape(d, F)
    H = bf16_round(orc.bf16_bits_to_f64(X) @ orc.bf16_bits_to_f64(Wgu).T)
    A = bf16_round(orc.silu(H[:, :F]) * H[:, F:])
    Y_sim = bf16_round(A @ orc.bf16_bits_to_f64(Wd).T)
    Y_ref = orc.mlp_forward(X, Wgu, Wd)
    err = max_abs_bf16_out(Y_sim, Y_ref)
    assert FULL_OUT_MAX_ABS < err <= 0.8 * FULL_MLP_OUT_MAX_ABS, err
    assert rel_fro(Y_sim, Y_ref) <= 0.8 * OUT_REL_FRO, rel_fro(Y_sim, Y_ref)
