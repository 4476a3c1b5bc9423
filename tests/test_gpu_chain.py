"""Forty Qwen3.6-35B-A3B-shaped MoE layers, all resident (~18 GB of NVFP4
weights), chained for one decode step at 1, 8 and 64 tokens.

The layer has no residual or norm around it, and SwiGLU is quadratic in its
input for small inputs (silu(g) ~ g/2), so a raw chain y_l -> x_{l+1} collapses
super-exponentially: within a few layers the activations fall below fp32's
range and every later layer computes zeros. Two chains are therefore run:

* renormalised: x_{l+1} = y_l * 2^-e_t per token, with e_t = floor(log2 max|y_l[t]|)
  (an exact power-of-two rescale standing in for the norm that sits between MoE
  layers outside this layer); every layer sees unit-scale inputs;
* raw: x_{l+1} = y_l exactly; layers are checked while the oracle output stays
  above 1e-20 (fp32 intermediates of the SwiGLU product still far from underflow),
  later ones for finiteness and the absolute part of the bar.

Parity is per layer, teacher-forced: the oracle gets the GPU's bf16 input of that
layer. Every layer and every token is checked (the oracle's experts run in
spawned worker processes, all layers in flight at once). Besides the usual bar
(max|gpu - oracle| <= 1e-2 max|oracle| + 1e-3) each checked layer meets the
scale-free bound max|gpu - oracle| <= 2e-2 max|oracle|.
"""
import pytest
import torch

import workload as wl
from harness import ParityCheck, check_layer_parity, gpu_layer, oracle_layer

pytestmark = pytest.mark.gpu

QW = wl.QWEN36_35B_A3B
N_LAYERS = 40
SEED = 0


@pytest.fixture(scope="module")
def chain(nv):
    layers = [gpu_layer(wl.LayerInputs(QW, seed=SEED, layer=l)) for l in range(N_LAYERS)]
    yield layers
    del layers
    torch.cuda.empty_cache()


def _pow2_renorm(y: torch.Tensor) -> torch.Tensor:
    """y * 2^-floor(log2 max|y[t]|) per token (exact in bf16); zero rows stay zero."""
    yf = y.float()
    m = yf.abs().amax(dim=1, keepdim=True)
    e = torch.where(m > 0, torch.floor(torch.log2(m)), torch.zeros_like(m))
    return (yf * torch.exp2(-e)).to(torch.bfloat16)


def _run_chain(nv, layers, x0, renorm):
    xs, outs = [x0], []
    x = x0.cuda()
    for layer in layers:
        y, ids, w = nv.moe_layer_forward(layer, x, want_route=True)
        outs.append((y, ids, w))
        x = _pow2_renorm(y) if renorm else y
        xs.append(x.cpu())
    torch.cuda.synchronize()
    return xs, outs


def _check(l, x, y, ids, w):
    check_layer_parity(wl.LayerInputs(QW, seed=SEED, layer=l), x, y, ids, w, rel_only=2e-2)


def _check_all_layers(xs, outs):
    checks = [ParityCheck(wl.LayerInputs(QW, seed=SEED, layer=l), xs[l], *outs[l], rel_only=2e-2)
              for l in range(N_LAYERS)]
    for c in checks:
        c.check()


def test_chain_40_layers_one_token(nv, chain):
    x0 = wl.activations(SEED, 1, QW.H)
    xs, outs = _run_chain(nv, chain, x0, renorm=True)
    _check_all_layers(xs, outs)


def test_chain_40_layers_8_tokens(nv, chain):
    x0 = wl.activations(SEED + 1, 8, QW.H)
    xs, outs = _run_chain(nv, chain, x0, renorm=True)
    assert all(torch.isfinite(o[0].float()).all() for o in outs)
    _check_all_layers(xs, outs)


def test_chain_40_layers_64_tokens(nv, chain):
    x0 = wl.activations(SEED + 2, 64, QW.H)
    xs, outs = _run_chain(nv, chain, x0, renorm=True)
    assert all(torch.isfinite(o[0].float()).all() for o in outs)
    _check_all_layers(xs, outs)


def test_chain_40_layers_raw(nv, chain):
    """x_{l+1} = y_l exactly: checked while outputs stay well inside fp32's range."""
    x0 = wl.activations(SEED + 3, 8, QW.H)
    xs, outs = _run_chain(nv, chain, x0, renorm=False)
    checked = 0
    for l in range(N_LAYERS):
        y, ids, w = outs[l]
        assert torch.isfinite(y.float()).all()
        assert float(y.float().abs().max()) <= 1.0
        if checked < N_LAYERS:
            res, _ = oracle_layer(wl.LayerInputs(QW, seed=SEED, layer=l), xs[l], force_ids=ids.cpu().numpy())
            if float(abs(res.y).max()) < 1e-20:
                break
            _check(l, xs[l], y, ids, w)
            checked += 1
    assert checked >= 2
