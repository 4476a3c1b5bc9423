"""moe_layer_forward_residual on the GPU against the oracle: the layer inside the residual
stream with the pre-MoE RMSNorm fused in (lynn-engine tutorials index, row 01: RMSNorm =
(1.0 + weight) x x_norm; Lynn Engine write-up, "Fused Kernels").

Bar, element by element: |gpu - oracle| <= 2^-8 |oracle| + 1e-2 max|layer part| + 1e-3,
where the oracle is h + layer(bf16(norm(h))) in fp64: the first term is the one bf16 rounding
of the output, the others the layer's stated bar on its own contribution. The GPU computes
the norm in fp32 (the oracle in fp64), so a normalised element can land one bf16 step away;
routing is compared as for the layer (ids exact where the oracle's k-th/(k+1)-th logit gap
exceeds 1e-3, other tokens re-evaluated on the GPU's expert set). Every path is covered: the
single-token kernel (norm in its staging, residual in its epilogue), the multi-token
tensor-core and fp32 paths, the grouped prefill path, and the output written in place.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import gpu_layer

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _inputs(shape, seed, T, scale=3.0):
    h = (wl.normal(wl.stream_key(seed, 91), T * shape.H, scale).view(T, shape.H)).to(torch.bfloat16)
    w = (wl.normal(wl.stream_key(seed, 92), shape.H, 0.1)).to(torch.bfloat16)
    return h, w


def _oracle(L, h, w, kind, force_ids=None, with_shared=True):
    shape = L.shape
    xb, _ = oracle.rmsnorm(h, w, EPS)
    lg = oracle.router_logits(xb, L.router_w("cpu"))
    ids, _, _ = oracle.route(lg, shape.k)
    need = ids if force_ids is None else np.asarray(force_ids)
    experts = {}
    for e in sorted(set(need.ravel().tolist())):
        experts[e] = tuple(oracle.pack(m, kind) for m in L.expert_f32(e))
    shared = tuple(oracle.pack(m, kind) for m in L.shared_f32()) if with_shared else None
    res = oracle.moe_layer_residual(h, w, EPS, L.router_w("cpu"), L.shared_sigmoid_w("cpu"), experts, shared,
                                    shape.k, force_ids=force_ids, batched=h.shape[0] > 8)
    return res, lg


def _check(L, h, w, out, ids, kind=0, with_shared=True):
    res, lg = _oracle(L, h, w, kind, with_shared=with_shared)
    gap = oracle.logit_gap(lg, L.shape.k)
    ids_g = ids.cpu().numpy()
    near = gap <= 1e-3
    clear = ~near
    assert np.array_equal(np.sort(ids_g[clear], 1), np.sort(res.ids[clear], 1))
    ref = res.y
    if near.any():
        forced = res.ids.copy()
        forced[near] = ids_g[near]
        ref = _oracle(L, h, w, kind, force_ids=forced, with_shared=with_shared)[0].y
    got = out.float().cpu().numpy().astype(np.float64)
    layer_part = ref - h.double().numpy()
    bound = 2.0 ** -8 * np.abs(ref) + 1e-2 * np.abs(layer_part).max() + 1e-3
    err = np.abs(got - ref)
    assert np.all(err <= bound), (float((err - bound).max()), int((err > bound).sum()))
    # the layer's contribution is really there (not just the residual passed through)
    assert np.abs(layer_part).max() > 0


@pytest.mark.parametrize("shape,T", [(wl.QWEN36_35B_A3B, 1), (wl.SMALL256, 1), (wl.QWEN36_35B_A3B, 8),
                                     (wl.QWEN36_35B_A3B, 64), (wl.TINY, 5), (wl.SMALL256, 300)])
def test_residual_layer(nv, shape, T):
    L = wl.LayerInputs(shape, seed=20 + T)
    layer = gpu_layer(L)
    h, w = _inputs(shape, 20 + T, T)
    out, ids, _ = nv.moe_layer_forward_residual(layer, h.cuda(), w.cuda(), EPS, want_route=True)
    torch.cuda.synchronize()
    _check(L, h, w, out, ids)


def test_residual_layer_grid_form(nv):
    """The fused single-token norm + residual on the persistent-grid form as well."""
    from harness import single_token_form
    shape = wl.QWEN36_35B_A3B
    L = wl.LayerInputs(shape, seed=21)
    layer = gpu_layer(L)
    h, w = _inputs(shape, 21, 1)
    with single_token_form(nv, 1):
        out, ids, _ = nv.moe_layer_forward_residual(layer, h.cuda(), w.cuda(), EPS, want_route=True)
        torch.cuda.synchronize()
    _check(L, h, w, out, ids)


def test_residual_layer_fp16_scales(nv):
    shape = wl.MoEShape(H=512, E=32, k=4, I=256, Is=128)
    L = wl.LayerInputs(shape, seed=23)
    layer = gpu_layer(L, kind=1)
    h, w = _inputs(shape, 23, 3)
    out, ids, _ = nv.moe_layer_forward_residual(layer, h.cuda(), w.cuda(), EPS, want_route=True)
    torch.cuda.synchronize()
    _check(L, h, w, out, ids, kind=1)


@pytest.mark.parametrize("T", [1, 8])
def test_residual_in_place(nv, T):
    """h_out may be h itself: every CTA reads its inputs before any output is written."""
    shape = wl.QWEN36_35B_A3B
    L = wl.LayerInputs(shape, seed=30 + T)
    layer = gpu_layer(L)
    h, w = _inputs(shape, 30 + T, T)
    ref_out = nv.moe_layer_forward_residual(layer, h.cuda(), w.cuda(), EPS)
    hb = h.cuda().clone()
    out = nv.moe_layer_forward_residual(layer, hb, w.cuda(), EPS, h_out=hb)
    torch.cuda.synchronize()
    assert out.data_ptr() == hb.data_ptr()
    assert torch.equal(hb.view(torch.int16), ref_out.view(torch.int16))


def test_residual_equals_norm_then_layer_then_add_on_the_gpu(nv):
    """The fused single-token call routes like the plain layer on the normalised row."""
    shape = wl.QWEN36_35B_A3B
    L = wl.LayerInputs(shape, seed=40)
    layer = gpu_layer(L)
    h, w = _inputs(shape, 40, 1)
    out, ids, wts = nv.moe_layer_forward_residual(layer, h.cuda(), w.cuda(), EPS, want_route=True)
    xb, _ = oracle.rmsnorm(h, w, EPS)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    y2, ids2, w2 = nv.moe_layer_forward(layer, x, want_route=True)
    torch.cuda.synchronize()
    gap = oracle.logit_gap(oracle.router_logits(xb, L.router_w("cpu")), shape.k)
    if gap[0] > 1e-3:
        assert torch.equal(torch.sort(ids, 1).values, torch.sort(ids2, 1).values)
