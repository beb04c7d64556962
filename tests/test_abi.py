"""C-ABI library: loads, exports every declared symbol, and rejects bad arguments on the host
before any launch (these calls touch no GPU)."""
import ctypes
import os
import re

import pytest
import torch

import long_context_attention_upipe_gb300 as up

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "upipe_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(upipe_(?:attn|mlp)_\w+)\s*\(", src)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 10
    L = ctypes.CDLL(up.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(up.EXPORTS)


def test_status_strings():
    for code in range(8):
        assert up.lib().upipe_attn_status_string(code)


def test_workspace_grows_with_chunk_not_heads():
    sizes = [up.workspace_bytes(up.make_desc(32768, 4096, 32, 8, 128, h), 1) for h in (4, 8, 32)]
    assert sizes[0] < sizes[1] < sizes[2]
    # doubling the head count at a fixed chunk size leaves the workspace unchanged
    a = up.workspace_bytes(up.make_desc(32768, 4096, 32, 8, 128, 8), 0)
    b = up.workspace_bytes(up.make_desc(32768, 4096, 64, 16, 128, 8), 0)
    assert a == b


@pytest.mark.parametrize("bad", [
    dict(S=0), dict(Hq=6, Hkv=4), dict(hpc=3), dict(Dh=96), dict(d=100), dict(causal=2), dict(accum=3),
    dict(Hq=32, Hkv=8, hpc=6), dict(scale=-1.0)])
def test_bad_descriptors_rejected(bad):
    kw = dict(S=512, d=256, Hq=4, Hkv=2, Dh=64, hpc=2, causal=1, accum=0, scale=0.0)
    kw.update(bad)
    d = up.make_desc(kw["S"], kw["d"], kw["Hq"], kw["Hkv"], kw["Dh"], kw["hpc"], True, kw["accum"], kw["scale"])
    d.causal = kw["causal"]
    n = ctypes.c_size_t(0)
    rc = up.lib().upipe_attn_workspace_size(ctypes.byref(d), 0, ctypes.byref(n))
    assert rc in (1, 2)


def test_fwd_host_checks_run_before_any_launch():
    d = up.make_desc(512, 256, 4, 2, 64, 2)
    L = up.lib()
    launches = up.launch_count()
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x10008)
    args = [fake] * 6
    assert L.upipe_attn_fwd(ctypes.byref(d), None, *args[1:], fake, 1 << 40, None) == 1       # NULL X
    assert L.upipe_attn_fwd(ctypes.byref(d), odd, fake, fake, None, fake, fake, fake, 1 << 40, None) == 3
    assert L.upipe_attn_fwd(ctypes.byref(d), fake, fake, fake, None, fake, fake, fake, 16, None) == 4
    assert L.upipe_attn_bwd(ctypes.byref(d), fake, fake, fake, None, fake, fake, fake, fake, fake, fake, 16, None) == 4
    bad = up.make_desc(512, 256, 4, 2, 96, 2)
    assert L.upipe_attn_fwd(ctypes.byref(bad), fake, fake, fake, None, fake, fake, fake, 1 << 40, None) == 2
    t = up.make_desc(512, 256, 4, 2, 64, 2)
    assert L.upipe_attn_build_tile_table(ctypes.byref(t), None, fake, 16, None, None) == 4
    assert L.upipe_attn_build_tile_table(ctypes.byref(t), odd, fake, 1 << 20, None, None) == 3
    assert L.upipe_attn_last_device_error(None, None, ctypes.byref(ctypes.c_int32())) == 1   # NULL workspace
    assert L.upipe_attn_no_alloc_device_status(None, None) == 1                            # NULL code
    core = [fake] * 6 + [None, fake]                                  # q k v dO lse D, no segments, table
    assert L.upipe_attn_core_bwd_dkdv_acc(ctypes.byref(d), *core, None, fake, None, None, None) == 1   # NULL dk_acc
    assert L.upipe_attn_core_bwd_dkdv_acc(ctypes.byref(d), *core, fake, fake, fake, None, None) == 1   # dk without dv
    assert L.upipe_attn_core_bwd_dkdv_acc(ctypes.byref(d), *core, odd, fake, None, None, None) == 3
    assert L.upipe_attn_core_bwd_dkdv_acc(ctypes.byref(d), *core, fake, fake, fake, odd, None) == 3
    assert up.launch_count() == launches  # rejected calls launch nothing


def test_offload_entry_points_check_arguments_before_any_launch():
    d = up.make_desc(512, 256, 4, 2, 64, 2)
    L = up.lib()
    launches = up.launch_count()
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: the checks fail first
    n = ctypes.c_size_t(0)
    assert L.upipe_attn_workspace_size_offload(ctypes.byref(d), 0, 100, ctypes.byref(n)) == 1   # not a multiple of 128
    assert L.upipe_attn_workspace_size_offload(ctypes.byref(d), 1, -128, ctypes.byref(n)) == 1
    assert L.upipe_attn_fwd_offload(ctypes.byref(d), fake, fake, fake, None, fake, fake, fake, 1 << 40, 96, None) == 1
    assert L.upipe_attn_fwd_offload(ctypes.byref(d), fake, fake, fake, None, fake, fake, fake, 16, 0, None) == 4
    assert L.upipe_attn_bwd_offload(ctypes.byref(d), fake, fake, fake, None, None, fake, fake, fake, fake, fake, 1 << 40,
                                    0, None) == 1                                               # NULL dY
    assert up.launch_count() == launches


def test_wait_limit_and_probe_check_arguments():
    L = up.lib()
    assert L.upipe_attn_set_wait_limit_ns(61 * 10 ** 9) == 1      # above the 60 s cap
    assert L.upipe_attn_set_wait_limit_ns(0) == 0                  # the default
    for bad in (-2, 1, 3, 4097, (1 << 24) + 2):
        assert L.upipe_attn_set_dkdv_window(bad) == 1               # odd, negative or too long
    assert L.upipe_attn_set_dkdv_window(2) == 0
    assert L.upipe_attn_set_dkdv_window(0) == 0                     # the default
    fake = ctypes.c_void_p(0x10000)
    assert L.upipe_attn_wait_probe(None, 64, 0, None) == 1
    assert L.upipe_attn_wait_probe(fake, 16, 0, None) == 1         # smaller than a table header
    assert L.upipe_attn_wait_probe(ctypes.c_void_p(0x10008), 64, 0, None) == 3


def test_mlp_host_checks_and_workspace_grow_with_the_tile():
    L = up.lib()
    fake = ctypes.c_void_p(0x10000)
    n = ctypes.c_size_t(0)
    for bad in (up.make_mlp_desc(0, 256, 512), up.make_mlp_desc(512, 256, 512, 100), up.make_mlp_desc(512, 256, 512, -128)):
        assert L.upipe_mlp_workspace_size(ctypes.byref(bad), 0, ctypes.byref(n)) == 1
    assert L.upipe_mlp_workspace_size(ctypes.byref(up.make_mlp_desc(512, 100, 512)), 0, ctypes.byref(n)) == 2
    d = up.make_mlp_desc(1 << 20, 4096, 14336, 8192)
    launches = up.launch_count()
    assert L.upipe_mlp_fwd(ctypes.byref(d), fake, fake, fake, fake, fake, 16, None) == 4
    assert L.upipe_mlp_bwd(ctypes.byref(d), fake, fake, fake, None, fake, fake, fake, fake, 1 << 40, None) == 1
    assert up.launch_count() == launches
    # the workspace holds one tile: it grows with tile_rows, not with S
    F, T = 14336, 8192
    assert up.mlp_workspace_bytes(d, 0) >= T * 3 * F * 2
    assert up.mlp_workspace_bytes(d, 0) < T * 3 * F * 2 + 4096
    assert up.mlp_workspace_bytes(up.make_mlp_desc(1 << 21, 4096, F, T), 1) == up.mlp_workspace_bytes(d, 1)
    untiled = up.mlp_workspace_bytes(up.make_mlp_desc(1 << 20, 4096, F, 0), 1)
    assert untiled > 100 * up.mlp_workspace_bytes(d, 1) // 2


def test_offload_workspace_adds_the_staging_buffers():
    d = up.make_desc(1 << 20, 4096, 4, 1, 128, 4)
    for pass_, tensors in ((0, 2), (1, 4)):           # X twice; X and dY twice each
        base = up.workspace_bytes(d, pass_)
        off = up.workspace_bytes_offload(d, pass_, 65536)
        assert off - base >= tensors * 65536 * 4096 * 2
        assert off - base < tensors * 65536 * 4096 * 2 + (64 << 20)   # plus block split-K partials, alignment
    assert up.workspace_bytes_offload(d, 1, 0) == up.workspace_bytes_offload(d, 1, 65536)   # the default


def test_backward_workspace_holds_fp32_kv_sums_past_the_window():
    # 1M tokens, one KV group of 4 query heads per chunk: 4 x 8192 items per key tile > 4096, so the
    # default window already plans the fp32 dK / dV sums; a 32K sequence (4 x 256 items) does not
    S, Dh = 1 << 20, 128
    sums = 2 * S * Dh * 4
    long_ = up.make_desc(S, 4096, 4, 1, Dh, 4)
    short = up.make_desc(32768, 4096, 4, 1, Dh, 4)
    base_long, base_short = up.workspace_bytes(long_, 1), up.workspace_bytes(short, 1)
    fwd = up.workspace_bytes(long_, 0)
    try:
        up.set_dkdv_window((1 << 24))                   # longer than any key tile's items: no sums
        assert base_long - up.workspace_bytes(long_, 1) >= sums
        up.set_dkdv_window(512)                         # 32K now exceeds it too
        assert up.workspace_bytes(short, 1) - base_short >= 2 * 32768 * Dh * 4
        assert up.workspace_bytes(long_, 0) == fwd       # the forward keeps no dK / dV
    finally:
        up.set_dkdv_window(0)
    assert up.workspace_bytes(long_, 1) == base_long


def test_ring_entry_points_check_arguments_before_any_launch():
    L = up.lib()
    launches = up.launch_count()
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x10008)
    assert L.upipe_attn_lse_merge(8, 128, None, fake, fake, fake, None, None) == 1          # NULL O_b
    assert L.upipe_attn_lse_merge(-1, 128, fake, fake, fake, fake, None, None) == 1         # negative rows
    assert L.upipe_attn_lse_merge(8, 96, fake, fake, fake, fake, None, None) == 2           # head_dim
    assert L.upipe_attn_lse_merge(8, 128, fake, fake, odd, fake, None, None) == 3           # alignment
    assert L.upipe_attn_lse_merge(8, 128, fake, fake, fake, fake, odd, None) == 3           # O_out alignment
    assert L.upipe_attn_ring_bwd_prep(0, 128, 128, fake, fake, fake, fake, None) == 1       # no heads
    assert L.upipe_attn_ring_bwd_prep(2, 0, 128, fake, fake, fake, fake, None) == 1         # empty chunk
    assert L.upipe_attn_ring_bwd_prep(2, 128, 80, fake, fake, fake, fake, None) == 2        # head_dim
    assert L.upipe_attn_ring_bwd_prep(2, 128, 64, fake, odd, fake, fake, None) == 3         # alignment
    assert L.upipe_attn_accumulate(16, None, fake, None, None) == 1                         # NULL source
    assert L.upipe_attn_accumulate(16, fake, odd, None, None) == 3                          # alignment
    assert up.launch_count() == launches  # rejected calls launch nothing
    # zero rows / elements are valid and launch nothing
    assert L.upipe_attn_lse_merge(0, 64, fake, fake, fake, fake, None, None) == 0
    assert L.upipe_attn_accumulate(0, fake, fake, None, None) == 0
    assert up.launch_count() == launches


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8])
def test_zigzag_ring_schedule_is_balanced_and_complete(P):
    """Each device computes 2P + 1 blocks (the zigzag balance); over all devices every block with
    key chunk <= query chunk is computed exactly once, causal exactly on the diagonal; a contiguous
    split (device r holding chunks 2r and 2r + 1) would not be balanced."""
    sched = up.ring_block_schedule(P)
    assert [sum(len(b) for b in steps) for steps in sched] == [2 * P + 1] * P
    blocks = [blk for steps in sched for b in steps for blk in b]
    assert sorted((q, k) for q, k, _ in blocks) == sorted((q, k) for q in range(2 * P) for k in range(q + 1))
    assert all((kind == "causal") == (q == k) for q, k, kind in blocks)
    if P > 1:
        contiguous = [sum(1 for q in (2 * r, 2 * r + 1) for k in range(q + 1)) for r in range(P)]
        assert len(set(contiguous)) > 1


def test_ring_step_calls_check_their_arguments_before_any_launch():
    L = up.lib()
    launches = up.launch_count()
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x10008)
    n = ctypes.c_size_t()
    ok = up.make_ring_desc(4, 256, 8, 2, 128)
    assert L.upipe_attn_ring_tables_size(ctypes.byref(ok), ctypes.byref(n)) == 0 and n.value > 0
    bad = [
        (up.make_ring_desc(0, 256, 8, 2, 128), 1),                           # no devices
        (up.make_ring_desc(4, 0, 8, 2, 128), 1),                             # empty chunk
        (up.make_ring_desc(4, 1 << 30, 8, 2, 128), 1),                       # 2C above 2^31 - 1
        (up.make_ring_desc(4, 256, 6, 4, 128), 1),                           # Hq not a multiple of Hkv
        (up.make_ring_desc(4, 256, 8, 2, 96), 2),                            # head_dim
        (up.make_ring_desc(4, 256, 8, 2, 128, dev_first=3, dev_count=2), 1),  # devices past the ring
        (up.make_ring_desc(4, 256, 8, 2, 128, dev_count=2, kv_count=3), 1),  # shard count neither P nor dev_count
    ]
    for d, code in bad:
        assert L.upipe_attn_ring_tables_size(ctypes.byref(d), ctypes.byref(n)) == code
        assert L.upipe_attn_ring_build_tables(ctypes.byref(d), None, fake, 1 << 20, None) == code
        assert L.upipe_attn_ring_fwd_step(ctypes.byref(d), 0, fake, fake, fake, None, fake, fake, fake, None, None) == code
    assert L.upipe_attn_ring_build_tables(ctypes.byref(ok), None, fake, n.value - 16, None) == 4   # too small
    assert L.upipe_attn_ring_build_tables(ctypes.byref(ok), odd, fake, n.value, None) == 3         # seg alignment
    f = L.upipe_attn_ring_fwd_step
    assert f(ctypes.byref(ok), 4, fake, fake, fake, None, fake, fake, fake, None, None) == 1       # step past P - 1
    assert f(ctypes.byref(ok), -1, fake, fake, fake, None, fake, fake, fake, None, None) == 1
    assert f(ctypes.byref(ok), 0, fake, fake, fake, None, fake, None, fake, None, None) == 1       # no accumulator
    assert f(ctypes.byref(ok), 0, fake, fake, fake, None, fake, fake, fake, odd, None) == 3        # o alignment
    b = L.upipe_attn_ring_bwd_step
    assert b(ctypes.byref(ok), 0, fake, fake, fake, fake, None, None, fake, fake, fake, fake, None, None, None,
             None) == 1                                                                         # no D
    assert b(ctypes.byref(ok), 0, fake, fake, fake, fake, fake, None, fake, fake, odd, fake, None, None, None,
             None) == 3                                                                         # dk_acc alignment
    r = L.upipe_attn_ring_fwd
    assert r(ctypes.byref(bad[0][0]), fake, fake, fake, None, fake, fake, fake, None, None) == 1
    assert r(ctypes.byref(ok), fake, None, fake, None, fake, fake, fake, None, None) == 1            # no k
    assert r(ctypes.byref(ok), fake, fake, fake, odd, fake, fake, fake, None, None) == 3             # seg alignment
    rb = L.upipe_attn_ring_bwd
    assert rb(ctypes.byref(ok), fake, fake, fake, None, fake, fake, None, fake, fake, fake, fake, fake, None, None,
              None, None) == 1                                                                    # no o
    assert rb(ctypes.byref(ok), fake, fake, fake, fake, fake, odd, None, fake, fake, fake, fake, fake, None, None,
              None, None) == 3                                                                    # lse alignment
    assert up.launch_count() == launches  # rejected calls launch nothing


def test_ring_tables_size_grows_with_the_batch():
    one = up.ring_tables_bytes(up.make_ring_desc(4, 4096, 8, 2, 128, dev_first=1, dev_count=1, kv_count=1))
    all_ = up.ring_tables_bytes(up.make_ring_desc(4, 4096, 8, 2, 128))
    nt = 8192 // 128
    assert one == 4 * (((32 + 2 * nt * 16 + 4 * (nt // 2 + nt)) + 15) // 16 * 16)
    assert all_ > 3 * one


def test_zigzag_reordering_round_trips_and_balances():
    P, C = 3, 5
    x = torch.arange(2 * P * C, dtype=torch.float32).reshape(1, -1, 1).repeat(2, 1, 3)
    xs = up.to_zigzag(x, P)
    assert tuple(xs.shape) == (P, 2, 2 * C, 3)
    for r in range(P):
        pos = up.zigzag_positions(P, C, r)
        assert torch.equal(xs[r, 0, :, 0], pos.float())
        assert bool((pos[1:] > pos[:-1]).all())           # local rows in sequence order
    assert torch.equal(up.from_zigzag(xs, P), x)
