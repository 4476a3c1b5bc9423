"""Bounded device waits: with the wait limit lowered to 1 ns, the one-launch
decode kernel's grid barrier runs out, the blocks record
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
    L = wl.LayerInputs(wl.TINY, seed=0)
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
