"""Bounded device waits: with the wait limit lowered to 1 ns, the one-launch
decode kernel's exchange polls run out, the blocks record
NVFP4_ERR_DEVICE_TIMEOUT in the workspace and return (no hang, no trap); after
the limit is restored and the workspace re-initialised the same call is
correct again."""
import numpy as np
import pytest
import torch

import workload as wl
from harness import check_layer_parity, gpu_layer

pytestmark = pytest.mark.gpu


def test_grid_barrier_timeout_is_reported(nv):
    L = wl.LayerInputs(wl.SMALL256, seed=0)
    layer = gpu_layer(L)
    x = wl.activations(0, 1, 256).cuda()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 1))
    try:
        nv.set_device_wait_limit(1)
        nv.moe_layer_forward(layer, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status(clear=True) == nv.NVFP4_ERR_DEVICE_TIMEOUT
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
