"""The forward entry point that allocates nothing (upipe_attn_fwd_no_alloc).

It serves callers that are not allowed to allocate device memory themselves, such as code being
recorded into a CUDA graph that someone else captures, or a plugin that is handed only input and
output pointers.  Its workspace is a fixed device array inside the library.  Here it is called
through the C-ABI and must reproduce the regular upipe_attn_fwd (which uses a caller-allocated
workspace) on the same inputs, on two calls in a row (the second call finds the array holding
the first call's leftovers).  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import long_context_attention_upipe_gb300 as up
import upipe_inputs as ui
from helpers import OUT_MAX_ABS, OUT_REL_FRO, bf16_tensor, layer_inputs, max_abs, rel_fro, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from long_context_attention_upipe_gb300 import _build
    _build.build()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_no_alloc_forward_matches_regular_forward_twice():
    S, d, Hq, Hkv, Dh, hpc = 512, 256, 4, 2, 64, 2
    X, W, Wo, _ = layer_inputs(S, d, Hq, Hkv, Dh, dy=False)
    seg = torch.from_numpy(ui.segments_from_lengths([300, 212])).cuda()
    Xt, Wt, Wot = bf16_tensor(X), bf16_tensor(W), bf16_tensor(Wo)
    desc = up.make_desc(S, d, Hq, Hkv, Dh, hpc, True)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    # reference: the regular entry point with a workspace allocated by the caller
    ws = torch.empty(up.workspace_bytes(desc, 0), dtype=torch.uint8, device="cuda")
    Y_ref = torch.empty_like(Xt)
    lse_ref = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    rc = up.lib().upipe_attn_fwd(ctypes.byref(desc), _ptr(Xt), _ptr(Wt), _ptr(Wot), _ptr(seg), _ptr(Y_ref),
                                 _ptr(lse_ref), _ptr(ws), ws.numel(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    want_y, want_lse = to_f64(Y_ref), to_f64(lse_ref)

    for _ in range(2):
        Y = torch.full_like(Xt, float("nan"))
        lse = torch.full((Hq, S), float("nan"), dtype=torch.float32, device="cuda")
        rc = up.lib().upipe_attn_fwd_no_alloc(ctypes.byref(desc), _ptr(Xt), _ptr(Wt), _ptr(Wot), _ptr(seg), _ptr(Y),
                                              _ptr(lse), stream)
        assert rc == 0, up.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        got_y, got_lse = to_f64(Y), to_f64(lse)
        assert np.isfinite(got_y).all() and np.isfinite(got_lse).all()
        assert max_abs(got_y, want_y) <= OUT_MAX_ABS
        assert rel_fro(got_y, want_y) <= OUT_REL_FRO
        assert max_abs(got_lse, want_lse) <= 1e-3


def test_no_alloc_forward_reports_device_errors():
    # segment ids that decrease are only visible on the device; the error word of the library's
    # own array must report them, and the next good call must clear it again
    S, d, Hq, Hkv, Dh = 256, 128, 2, 1, 64
    X, W, Wo, _ = layer_inputs(S, d, Hq, Hkv, Dh, dy=False)
    Xt, Wt, Wot = bf16_tensor(X), bf16_tensor(W), bf16_tensor(Wo)
    desc = up.make_desc(S, d, Hq, Hkv, Dh, 1, True)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    Y = torch.empty_like(Xt)
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    for ids, want in (([0] * 100 + [2] * 100 + [1] * 56, 5), ([0] * 100 + [1] * 156, 0)):
        seg = torch.tensor(ids, dtype=torch.int32, device="cuda")
        rc = up.lib().upipe_attn_fwd_no_alloc(ctypes.byref(desc), _ptr(Xt), _ptr(Wt), _ptr(Wot), _ptr(seg), _ptr(Y),
                                              _ptr(lse), stream)
        assert rc == 0
        assert up.no_alloc_device_status() == want


def test_no_alloc_forward_rejects_too_large_descriptor():
    # the 32k-token, 8-head chunk needs a forward workspace far above the 32 MiB array
    desc = up.make_desc(32768, 4096, 32, 8, 128, 8, True)
    assert up.workspace_bytes(desc, 0) > (32 << 20)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    rc = up.lib().upipe_attn_fwd_no_alloc(ctypes.byref(desc), fake, fake, fake, None, fake, fake, None)
    assert rc == 4  # UPIPE_ERR_WORKSPACE_TOO_SMALL
