"""moe_layer_forward on the prefill path (T > 64 tokens) against the oracle.

The layer is the same as on the decode path (lynn-engine tutorials index, row
06; lynn-engine README, P28/P29 notes) computed as grouped tensor-core GEMMs
(lynn-engine README, P2/P3-A notes). Bar as for decode: max|gpu - oracle| <=
1e-2 * max|oracle| + 1e-3 per output tensor; expert ids exact as sets and
weights within 1e-5 for every token whose k-th/(k+1)-th logit gap exceeds 1e-3.
At full size every token is checked: the oracle's routed experts are evaluated in
spawned worker processes (harness.ParityCheck), and routing is also checked on
every token against the oracle's fp64 router.
"""
import json
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import ParityCheck, check_layer_parity, gpu_layer

pytestmark = pytest.mark.gpu

QW = wl.QWEN36_35B_A3B
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "prefill_zipf.json")


def _forward(nv, layer, x):
    y, ids, w = nv.moe_layer_forward(layer, x.cuda(), want_route=True)
    torch.cuda.synchronize()
    return y, ids, w


def _check_routing_all(L, x, ids_gpu, w_gpu, gap_min=1e-3):
    """Routing of every token against the oracle's fp64 router."""
    logits = oracle.router_logits(x, L.router_w("cpu"))
    ids_o, w_o, _ = oracle.route(logits, L.shape.k)
    gap = oracle.logit_gap(logits, L.shape.k)
    ids_g = ids_gpu.cpu().numpy()
    w_g = w_gpu.cpu().numpy()
    clear = gap > gap_min
    assert np.array_equal(np.sort(ids_g[clear], 1), np.sort(ids_o[clear], 1))
    for t in np.flatnonzero(clear):
        wo = dict(zip(ids_o[t].tolist(), w_o[t].tolist()))
        for e, wv in zip(ids_g[t].tolist(), w_g[t].tolist()):
            assert abs(wv - wo[e]) <= 1e-5, (t, e, wv, wo[e])
    return ids_o


SM = wl.SMALL256


@pytest.mark.parametrize("T", [65, 200, 777])
def test_small_prefill(nv, T):
    """Every token of a small layer on the grouped tensor-core path: several token
    tiles per expert and ragged tails."""
    L = wl.LayerInputs(SM, seed=100 + T)
    layer = gpu_layer(L)
    x = wl.activations(100 + T, T, SM.H)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w)


def test_small_prefill_no_shared_expert(nv):
    L = wl.LayerInputs(SM, seed=7)
    layer = gpu_layer(L, with_shared=False)
    x = wl.activations(7, 300, SM.H)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w, with_shared=False)


def test_small_prefill_skewed_routing(nv):
    """Strongly skewed router: some experts get no tokens, others several 256-row tiles."""
    shape = replace(SM, router_kappa=1.5)
    L = wl.LayerInputs(shape, seed=11)
    layer = gpu_layer(L)
    x = wl.activations(11, 1600, shape.H)
    y, ids, w = _forward(nv, layer, x)
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=shape.E)
    assert counts.max() > 512
    check_layer_parity(L, x, y, ids, w)


def test_tiny_prefill_chunked(nv):
    """I = 128 is outside the grouped path's shapes: 64-token chunks of the decode path."""
    L = wl.LayerInputs(wl.TINY, seed=13)
    layer = gpu_layer(L)
    x = wl.activations(13, 150, wl.TINY.H)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w)


def test_tiny_prefill_fp16_scales(nv):
    """FP16-scaled layers above 64 tokens run as 64-token chunks of the decode path."""
    L = wl.LayerInputs(wl.TINY, seed=5)
    layer = gpu_layer(L, kind=1)
    x = wl.activations(5, 150, wl.TINY.H)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w, kind=1)


def test_prefill_deterministic(nv):
    L = wl.LayerInputs(SM, seed=3)
    layer = gpu_layer(L)
    x = wl.activations(3, 500, SM.H).cuda()
    y1 = nv.moe_layer_forward(layer, x)
    y2 = nv.moe_layer_forward(layer, x)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_qwen_prefill_300_every_token(nv):
    L = wl.LayerInputs(QW, seed=4)
    layer = gpu_layer(L)
    T = 300
    x = wl.activations(4, T, QW.H)
    y, ids, w = _forward(nv, layer, x)
    _check_routing_all(L, x, ids, w)
    ParityCheck(L, x, y, ids, w).check()


def test_qwen_prefill_4096_zipf(nv):
    """The 4096-token prefill workload with the skewed router (kappa from the
    golden calibration): per-expert counts must match the calibration exactly
    on every token with a clear routing margin; output parity on every token."""
    with open(GOLDEN) as f:
        gold = json.load(f)
    shape = replace(QW, router_kappa=gold["kappa"])
    L = wl.LayerInputs(shape, seed=gold["seed"])
    layer = gpu_layer(L)
    T = gold["T"]
    x = wl.activations(gold["seed"], T, shape.H)
    y, ids, w = _forward(nv, layer, x)
    ids_o = _check_routing_all(L, x, ids, w)
    assert np.array_equal(np.bincount(ids_o.ravel(), minlength=shape.E), np.array(gold["counts"]))
    g = np.bincount(ids.cpu().numpy().ravel(), minlength=shape.E)
    assert abs(int(g.max()) - gold["max_count"]) <= 8
    ParityCheck(L, x, y, ids, w).check()


def test_prefill_wait_timeout_is_reported(nv):
    """The grouped tensor-core kernels' bounded waits with the limit at 1 ns: the first wait
    that is not already satisfied runs out, the CTA raises its abort flag, stops issuing copies
    and MMAs, waits (with the library's fixed limit) for the ones in flight, frees its tensor
    memory and returns; the workspace records the timeout. Afterwards the same call is correct."""
    L = wl.LayerInputs(wl.SMALL256, seed=31)
    layer = gpu_layer(L)
    x = wl.activations(31, 300, 256)
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 300))
    try:
        nv.set_device_wait_limit(1)
        nv.moe_layer_forward(layer, x.cuda(), ws=ws)
        torch.cuda.synchronize()
        assert ws.status(clear=True) == nv.NVFP4_ERR_DEVICE_TIMEOUT
    finally:
        nv.set_device_wait_limit(0)
    nv.lib.nvfp4_workspace_init(ws.ptr(), ws.nbytes, nv._stream())
    y, ids, w = nv.moe_layer_forward(layer, x.cuda(), ws=ws, want_route=True)
    torch.cuda.synchronize()
    assert ws.status() == nv.NVFP4_OK
    check_layer_parity(L, x, y, ids, w)
