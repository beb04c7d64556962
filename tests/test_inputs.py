"""The seeded input generator (shared by the oracle and the CUDA path)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import upipe_inputs as ui


def test_splitmix64_published_stream():
    # SplitMix64 seeded with 0 (Vigna's reference generator): first three outputs
    lib = ui._host_lib()
    g = 0x9E3779B97F4A7C15
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [lib.ug_mix64_host(((n + 1) * g) & (2**64 - 1)) for n in range(3)]
    assert got == want


def _bf16_rne_exact(x: float) -> int:
    """Round-to-nearest-even to bf16 with exact rational arithmetic."""
    if x == 0:
        return 0x8000 if math.copysign(1, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    f = Fraction(abs(x))
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > f:
        e -= 1
    while Fraction(2) ** (e + 1) <= f:
        e += 1
    q = f / Fraction(2) ** (e - 7)  # in [128, 256)
    n = math.floor(q)
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    if n == 256:
        n, e = 128, e + 1
    return sign | ((e + 127) << 7) | (n - 128)


def test_bf16_rounding_exact():
    lib = ui._host_lib()
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000))
    # ties and near-ties
    vals += [1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-40, -(1.0 + 2**-8 - 2**-40), 0.0099487304687500]
    for v in vals:
        assert lib.ug_bf16_rne_host(float(v)) == _bf16_rne_exact(float(v)), v


def test_log_within_one_ulp():
    lib = ui._host_lib()
    rng = np.random.default_rng(1)
    for v in list(rng.random(2000)) + [1.0, 0.5, 1e-300, 0.7071067811865476, 0.7071067811865475]:
        a, b = lib.ug_log_host(float(v)), math.log(float(v))
        assert abs(a - b) <= 2 * math.ulp(b) + 1e-300, (v, a, b)


def test_normal_statistics_and_determinism():
    scipy_stats = pytest.importorskip("scipy.stats")
    x = ui.bf16_to_f64(ui.normal_bf16(200000, ui.TID_X))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert scipy_stats.kstest(x, "norm").pvalue > 1e-4 or abs(x.std() - 1) < 0.01
    w = ui.bf16_to_f64(ui.normal_bf16(100000, ui.TID_WQKV, std=ui.W_STD))
    assert abs(w.std() - 0.02) < 0.0005
    a = ui.normal_bf16(1000, 3, first=5000)
    b = ui.normal_bf16(6000, 3)[5000:]
    np.testing.assert_array_equal(a, b)
    rows = ui.normal_bf16_rows([3, 0, 7], 11, 3)
    full = ui.normal_bf16(8 * 11, 3).reshape(8, 11)
    np.testing.assert_array_equal(rows, full[[3, 0, 7]])
    assert not np.array_equal(ui.normal_bf16(100, 0), ui.normal_bf16(100, 1))


def test_segment_recipe():
    L = ui.loguniform_lengths(131072)
    assert sum(L) == 131072
    assert all(1024 <= x < 32768 for x in L[:-1])
    assert L == ui.loguniform_lengths(131072)
    seg = ui.segments_from_lengths(L)
    assert seg.dtype == np.int32 and np.all(np.diff(seg) >= 0) and seg[-1] == len(L) - 1


def test_metric_flops_of_the_workloads():
    """The metric counts algorithmic FLOPs: attention 4 Dh per visible (query, key) pair and head
    forward, 3.5x that forward+backward, and the projections 2 M N K forward, 3x forward+backward.
    The visible pairs of the packed 131K workload are recounted here from the oracle's per-tile
    counts (a row-by-row count of the mask, independent of the closed form used by the metric)."""
    import oracle as orc
    w = ui.workload("packed_131k")
    pairs = int(orc.tile_counts(w.S, w.segments(), True).sum())
    assert pairs == w.visible_pairs()
    assert abs(pairs / (w.S * (w.S + 1) / 2) - 0.1095) < 5e-4       # 10.95% of dense causal pairs
    w2 = ui.workload("llama8b_32k")
    attn_fwd = 4 * 128 * (32768 * 32769 // 2) * 32
    proj_fwd = 2 * 32768 * 4096 * (32 + 16) * 128 + 2 * 32768 * 32 * 128 * 4096
    assert w2.flops_fwd_bwd() == 3.5 * attn_fwd + 3 * proj_fwd
    assert abs(w2.flops_fwd_bwd() / 1e12 - 39.03) < 0.01
    assert abs(ui.workload("ulysses_1m").flops_fwd_bwd() / 1e15 - 3.974) < 0.001
    assert abs(ui.workload("share32b_5m").flops_fwd_bwd() / 1e15 - 179.554) < 0.001
