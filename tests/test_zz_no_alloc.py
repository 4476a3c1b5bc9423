"""moe_layer_forward_noalloc: the layer with the library's static scratch array
instead of a caller workspace, for callers that cannot allocate device memory
where they run the layer. Checked through the C ABI against moe_layer_forward
on the same inputs, two calls in a row, for the one-launch single-token path
and the multi-token path. Both entry points run the same deterministic kernels,
so the outputs must agree bit for bit. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workload as wl
from harness import gpu_layer, tol_ok

pytestmark = pytest.mark.gpu


def _noalloc(nv, layer, x):
    d = layer.desc()
    T = x.shape[0]
    y = torch.empty(T, layer.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(T, layer.k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, layer.k, dtype=torch.float32, device="cuda")
    st = nv.lib.moe_layer_forward_noalloc(ctypes.byref(d), ctypes.c_void_p(x.data_ptr()), T,
                                          ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                          ctypes.c_void_p(w.data_ptr()), nv._stream())
    assert st == nv.NVFP4_OK, st
    return y, ids, w


@pytest.mark.parametrize("shape,T", [(wl.TINY, 1), (wl.SMALL256, 1), (wl.TINY, 5), (wl.QWEN36_35B_A3B, 1),
                                     (wl.QWEN36_35B_A3B, 64)])
def test_noalloc_matches_workspace_entry_point(nv, shape, T):
    L = wl.LayerInputs(shape, seed=7)
    layer = gpu_layer(L)
    x = wl.activations(7, T, shape.H).cuda()
    y_ref, ids_ref, w_ref = nv.moe_layer_forward(layer, x, want_route=True)
    for _ in range(2):   # two calls in a row share the static scratch
        y, ids, w = _noalloc(nv, layer, x)
        torch.cuda.synchronize()
        ok, err, bound = tol_ok(y.float().cpu().numpy().astype(np.float64),
                                y_ref.float().cpu().numpy().astype(np.float64))
        assert ok, (err, bound)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        assert torch.equal(ids, ids_ref)
        assert torch.equal(w, w_ref)


def test_noalloc_large_then_small_then_large(nv):
    """A smaller call after a larger one, then a larger one with other inputs: what the
    previous call left in the shared scratch must not leak into the next result."""
    shape = wl.QWEN36_35B_A3B
    L = wl.LayerInputs(shape, seed=8)
    layer = gpu_layer(L)
    for T, seed in ((64, 8), (1, 9), (64, 10), (8, 11), (1, 12)):
        x = wl.activations(seed, T, shape.H).cuda()
        y_ref, ids_ref, w_ref = nv.moe_layer_forward(layer, x, want_route=True)
        y, ids, w = _noalloc(nv, layer, x)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), T
        assert torch.equal(ids, ids_ref) and torch.equal(w, w_ref), T


def test_noalloc_status_reports_a_timeout(nv):
    """The static scratch's status word is readable: OK after a normal call; with the wait
    limit at 1 ns the single-token grid form's exchange polls run out (it always polls
    before its peers publish), the timeout is recorded and read back, clearing works, and
    the next call (which clears the scratch) is exact again."""
    from harness import single_token_form
    L = wl.LayerInputs(wl.SMALL256, seed=13)
    layer = gpu_layer(L)
    x = wl.activations(13, 1, wl.SMALL256.H).cuda()
    y_ref = nv.moe_layer_forward(layer, x)
    with single_token_form(nv, 1):
        _noalloc(nv, layer, x)
        assert nv.noalloc_status() == nv.NVFP4_OK
        try:
            nv.set_device_wait_limit(1)
            _noalloc(nv, layer, x)
            assert nv.noalloc_status(clear=True) == nv.NVFP4_ERR_DEVICE_TIMEOUT
            assert nv.noalloc_status() == nv.NVFP4_OK
        finally:
            nv.set_device_wait_limit(0)
        y, _, _ = _noalloc(nv, layer, x)
        assert nv.noalloc_status() == nv.NVFP4_OK
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_rejects_oversized_scratch(nv):
    L = wl.LayerInputs(wl.QWEN36_35B_A3B, seed=0)
    layer = gpu_layer(L)
    x = torch.zeros(64, 2048, dtype=torch.bfloat16, device="cuda")
    d = layer.desc()
    d.E, d.k, d.I, d.Is = 256, 8, 8192, 8192    # 64 tokens x 8 x 8192 intermediates: far above 8 MiB
    y = torch.empty(64, 2048, dtype=torch.bfloat16, device="cuda")
    st = nv.lib.moe_layer_forward_noalloc(ctypes.byref(d), ctypes.c_void_p(x.data_ptr()), 64,
                                          ctypes.c_void_p(y.data_ptr()), None, None, nv._stream())
    assert st == nv.NVFP4_ERR_WORKSPACE_TOO_SMALL
