"""Bounded device waits: with the wait limit lowered to 1 ns, the one-launch
decode kernel's exchange polls run out, the blocks record
NVFP4_ERR_DEVICE_TIMEOUT in the workspace and return (no hang, no trap); after
the limit is restored and the workspace re-initialised the same call is
correct again."""
import numpy as np
import pytest
import torch

import workload as wl
from harness import check_layer_parity, gpu_layer, single_token_form

pytestmark = pytest.mark.gpu


def _tag_period(sms):
    # every single-token launch adds this to the workspace's launch counter (the lcm of the
    # grid sizes either form can launch: the SM count and cs * k, cs in {8, 12, 16}, k <= 8)
    from math import gcd
    l = sms
    for cs in (8, 12, 16):
        for k in range(1, 9):
            l = l // gcd(l, cs * k) * (cs * k)
    return l


@pytest.mark.parametrize("form", [2, 1], ids=["cluster", "grid"])
def test_split_launch_tags_time_out(nv, form):
    """The host drops the counter one short of a launch boundary, so the first CTA of the
    next launch takes one tag and the others the next: their exchange words never match,
    every bounded poll runs out (a flag that nothing sets), the timeout is recorded and the
    CTAs return; after re-initialising the workspace the same call is correct."""
    L = wl.LayerInputs(wl.SMALL256, seed=2)
    layer = gpu_layer(L)
    x = wl.activations(2, 1, 256).cuda()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 1))
    with single_token_form(nv, form):
        assert nv.single_token_form_used(layer, 1) in ((2, 1) if form == 2 else (1,))
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        start = torch.tensor([_tag_period(sms) - 1], dtype=torch.int64, device="cuda")
        ws.buf[8:16].copy_(start.view(torch.uint8))      # the header's launch counter
        try:
            nv.set_device_wait_limit(1_000_000)           # 1 ms
            nv.moe_layer_forward(layer, x, ws=ws)
            torch.cuda.synchronize()
            assert ws.status(clear=True) == nv.NVFP4_ERR_DEVICE_TIMEOUT
        finally:
            nv.set_device_wait_limit(0)
        nv.lib.nvfp4_workspace_init(ws.ptr(), ws.nbytes, nv._stream())
        y, ids, w = nv.moe_layer_forward(layer, x, ws=ws, want_route=True)
        torch.cuda.synchronize()
        assert ws.status() == nv.NVFP4_OK
        check_layer_parity(L, x, y, ids, w)


@pytest.mark.parametrize("form", [2, 1], ids=["cluster", "grid"])
def test_grid_barrier_timeout_is_reported(nv, form):
    L = wl.LayerInputs(wl.SMALL256, seed=0)
    layer = gpu_layer(L)
    x = wl.activations(0, 1, 256).cuda()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 1))
    with single_token_form(nv, form):
        try:
            nv.set_device_wait_limit(1)
            nv.moe_layer_forward(layer, x, ws=ws)
            torch.cuda.synchronize()
            st = ws.status(clear=True)
            # the grid form always polls before its peers publish; the cluster form's few
            # global polls can find their words already there (then the call is complete)
            assert st == nv.NVFP4_ERR_DEVICE_TIMEOUT or (form == 2 and st == nv.NVFP4_OK)
        finally:
            nv.set_device_wait_limit(0)
        # the context is still usable; a fresh workspace state gives the right answer
        nv.lib.nvfp4_workspace_init(ws.ptr(), ws.nbytes, nv._stream())
        y, ids, w = nv.moe_layer_forward(layer, x, ws=ws, want_route=True)
        torch.cuda.synchronize()
    assert ws.status() == nv.NVFP4_OK
    check_layer_parity(L, x, y, ids, w)


def test_gemv_wait_timeout_is_reported(nv):
    """The dense GEMV's chunk waits with the limit at 1 ns: the rows whose chunk had not
    landed become quiet NaN, the workspace records the timeout, the CTAs drain their copies
    and return; afterwards the same call is exact again."""
    import oracle
    from harness import tol_ok
    w = wl.dense_weight_f32(5, 8192, 2048)
    x = wl.activations(5, 1, 2048)
    W = nv.nvfp4_pack(w.cuda(), 1)
    ws = nv.Workspace(256)
    y = torch.empty(1, 8192, dtype=torch.bfloat16, device="cuda")
    wc = W.c()
    try:
        nv.set_device_wait_limit(1)
        st = nv.lib.nvfp4_gemv_w4a16(nv.ctypes.byref(wc), nv._ptr(x.cuda()), 1, nv._ptr(y), ws.ptr(), ws.nbytes,
                                     nv._stream())
        assert st == nv.NVFP4_OK
        torch.cuda.synchronize()
        code = ws.status(clear=True)
        nan_rows = int(torch.isnan(y.float()).sum())
        # the status and the NaN rows go together: either no wait ran out or both show it
        assert (code == nv.NVFP4_ERR_DEVICE_TIMEOUT) == (nan_rows > 0)
        assert code in (nv.NVFP4_OK, nv.NVFP4_ERR_DEVICE_TIMEOUT)
    finally:
        nv.set_device_wait_limit(0)
    y2 = nv.nvfp4_gemv_w4a16(W, x.cuda())
    torch.cuda.synchronize()
    ref = oracle.gemv(oracle.pack(w, 1), x)
    ok, err, bound = tol_ok(y2.float().cpu().numpy().astype(np.float64), ref)
    assert ok, (err, bound)


def test_multi_token_path_has_no_waits(nv):
    """The multi-token decode kernels hand work on with completion counters and never wait
    on another CTA: a call with the wait limit at 1 ns is still exact and reports OK."""
    L = wl.LayerInputs(wl.SMALL256, seed=6)
    layer = gpu_layer(L)
    x = wl.activations(6, 12, wl.SMALL256.H).cuda()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 12))
    try:
        nv.set_device_wait_limit(1)
        y, ids, w = nv.moe_layer_forward(layer, x, ws=ws, want_route=True)
        torch.cuda.synchronize()
    finally:
        nv.set_device_wait_limit(0)
    assert ws.status() == nv.NVFP4_OK
    check_layer_parity(L, x, y, ids, w)
