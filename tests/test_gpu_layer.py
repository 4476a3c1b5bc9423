"""moe_layer_forward on the GPU against the oracle.

Bar (per output tensor): max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3; expert
ids as sets, exact, for every token whose k-th/(k+1)-th router logit gap
exceeds 1e-3 (other tokens are checked against the oracle evaluated on the
GPU's expert set); renormalised weights within 1e-5 per expert id.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import (ParityCheck, check_layer_parity, gpu_layer, margin_tokens, oracle_layer, single_token_form,
                     tol_ok)

pytestmark = pytest.mark.gpu

QW = wl.QWEN36_35B_A3B


def _forward(nv, layer, x):
    y, ids, w = nv.moe_layer_forward(layer, x.cuda(), want_route=True)
    torch.cuda.synchronize()
    return y, ids, w


def test_tiny_layer_one_token(nv):
    L = wl.LayerInputs(wl.TINY, seed=0)
    layer = gpu_layer(L)
    x = wl.activations(0, 1, 256)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w)


@pytest.mark.parametrize("T", [2, 5, 8, 64])
def test_tiny_layer_tokens(nv, T):
    L = wl.LayerInputs(wl.TINY, seed=T)
    layer = gpu_layer(L)
    x = wl.activations(T, T, 256)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w)


@pytest.mark.parametrize("form", [2, 1], ids=["cluster", "grid"])
def test_decode_one_token_seeds_0_31(nv, form):
    """Single-token decode through a Qwen3.6-35B-A3B-shaped layer, seeds 0..31,
    router margins above 1e-3 (tokens redrawn from their seed stream until so), on the
    cluster form and on the persistent-grid form."""
    errs = []
    for seed in range(32):
        L = wl.LayerInputs(QW, seed=seed)
        layer = gpu_layer(L)
        x, _ = margin_tokens(L, seed, 1)
        with single_token_form(nv, form):
            y, ids, w = _forward(nv, layer, x)
        err, bound, near = check_layer_parity(L, x, y, ids, w)
        assert near == 0
        errs.append(err / bound)
        del layer
        torch.cuda.empty_cache()
    assert max(errs) < 1.0


@pytest.mark.parametrize("T,seed", [(8, 0), (8, 5), (64, 1), (33, 2)])
def test_decode_batched_every_token(nv, T, seed):
    """8, 33 and 64 concurrent tokens in one call; every token against the oracle."""
    L = wl.LayerInputs(QW, seed=seed)
    layer = gpu_layer(L)
    x = wl.activations(seed, T, QW.H)
    y, ids, w = _forward(nv, layer, x)
    ParityCheck(L, x, y, ids, w).check()


def test_fp16_scale_layer(nv):
    shape = wl.MoEShape(H=512, E=32, k=4, I=256, Is=128)
    L = wl.LayerInputs(shape, seed=3)
    layer = gpu_layer(L, kind=1)
    x = wl.activations(3, 4, 512)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w, kind=1)


@pytest.mark.parametrize("shape", [
    wl.MoEShape(H=32, E=1, k=1, I=32, Is=32),
    wl.MoEShape(H=64, E=4, k=4, I=32, Is=64),
    wl.MoEShape(H=96, E=7, k=3, I=96, Is=0),
    wl.MoEShape(H=2048, E=256, k=1, I=64, Is=32),
])
def test_edge_shapes(nv, shape):
    L = wl.LayerInputs(shape, seed=11)
    layer = gpu_layer(L, with_shared=shape.Is > 0)
    x = wl.activations(11, 3, shape.H)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w, with_shared=shape.Is > 0)


def test_zero_tokens_is_noop(nv):
    L = wl.LayerInputs(wl.TINY, seed=0)
    layer = gpu_layer(L)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    y = nv.moe_layer_forward(layer, x)
    assert y.shape == (0, 256)


def test_deterministic_bits(nv):
    L = wl.LayerInputs(QW, seed=4)
    layer = gpu_layer(L)
    x = wl.activations(4, 8, QW.H).cuda()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, 8))
    y0 = nv.moe_layer_forward(layer, x, ws=ws)
    for _ in range(10):
        assert torch.equal(nv.moe_layer_forward(layer, x, ws=ws), y0)


def test_workspace_too_small(nv):
    L = wl.LayerInputs(wl.TINY, seed=0)
    layer = gpu_layer(L)
    ws = nv.Workspace(256)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.moe_layer_forward(layer, wl.activations(0, 1, 256).cuda(), ws=ws)
    assert ei.value.status == nv.NVFP4_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("kind", [2, 3])
@pytest.mark.parametrize("T", [1, 6])
def test_layer_other_scale_contracts(nv, kind, T):
    """A layer stored with FP32 per-16 or E8M0 per-32 scales runs on the fp32 multi-token
    kernels (the fast paths take E4M3 / FP16 only and refuse nothing silently)."""
    shape = wl.MoEShape(H=512, E=32, k=4, I=256, Is=256)
    L = wl.LayerInputs(shape, seed=60 + kind)
    layer = gpu_layer(L, kind=kind)
    x = wl.activations(60 + kind, T, 512)
    y, ids, w = _forward(nv, layer, x)
    check_layer_parity(L, x, y, ids, w, kind=kind)
    assert nv.launches_per_layer_call(T, 512, kind=kind, E=32, I=256, Is=256, k=4) == 5
