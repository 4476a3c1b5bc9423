"""Pins for the oracle's pre-MoE RMSNorm and the residual form of the layer.

lynn-engine tutorials index, row 01 and the Qwen 3.6 config block: RMSNorm is
(1.0 + weight) x x_norm, x_norm = h / sqrt(mean(h^2) + eps) (not Llama's
weight x x_norm). The normalised activations are rounded once to bf16, the type
the layer consumes; the residual output is h + layer(x).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import oracle_experts, oracle_shared


def _bf16_value(bits: int) -> Fraction:
    b = np.array([bits << 16], np.uint32).view(np.float32)[0]
    return Fraction(float(b))


def _nearest_bf16_brute(v: float) -> int:
    """Nearest bf16 by exact comparison over the neighbours of v's fp32 truncation."""
    f32 = np.array([v], np.float64).astype(np.float32)
    base = int(f32.view(np.uint32)[0] >> 16)
    best, bd = None, None
    tv = Fraction(v)
    for c in range(max(0, (base & 0x7FFF) - 2), (base & 0x7FFF) + 3):
        if (c & 0x7F80) == 0x7F80:
            continue
        bits = (base & 0x8000) | c
        dist = abs(_bf16_value(bits) - tv)
        if best is None or dist < bd or (dist == bd and (bits & 1) == 0):
            best, bd = bits, dist
    return best


def test_bf16_rounding_matches_brute_force(orc):
    rng = np.random.default_rng(0)
    vals = list(rng.normal(size=300) * np.exp2(rng.integers(-60, 60, size=300)))
    # exact midpoints between neighbouring bf16 values (ties go to the even mantissa)
    for m in (1.0, 3.5, -0.15625, 2.0 ** -126, 1.5 * 2.0 ** -130):
        b = oracle.bf16_from_double(m)
        lo, hi = float(_bf16_value(b)), float(_bf16_value(b + 1))
        vals += [(lo + hi) / 2, -(lo + hi) / 2, lo, np.nextafter((lo + hi) / 2, hi)]
    for v in vals:
        assert oracle.bf16_from_double(float(v)) == _nearest_bf16_brute(float(v)), v


def _rows(seed, T, H, scale=1.0):
    return (wl.normal(wl.stream_key(seed, 77), T * H, scale).view(T, H)).to(torch.bfloat16)


def test_unit_weight_gives_unit_rms(orc):
    h = _rows(1, 5, 256)
    _, f = oracle.rmsnorm(h, torch.zeros(256, dtype=torch.bfloat16), 0.0)
    assert np.allclose(np.sqrt((f ** 2).mean(axis=1)), 1.0, rtol=1e-12)


def test_one_plus_weight_convention(orc):
    """(1 + w) multiplies the normalised row: w = -1 gives zeros, and the output is linear in
    (1 + w) element by element (not Llama's w x x_norm)."""
    h = _rows(2, 3, 128)
    w0 = torch.zeros(128, dtype=torch.bfloat16)
    _, f0 = oracle.rmsnorm(h, w0, 1e-6)
    wm = torch.full((128,), -1.0, dtype=torch.bfloat16)
    bm, fm = oracle.rmsnorm(h, wm, 1e-6)
    assert np.all(fm == 0.0) and np.all((bm & 0x7FFF) == 0)
    w = (wl.normal(wl.stream_key(3), 128, 0.5)).to(torch.bfloat16)
    _, fw = oracle.rmsnorm(h, w, 1e-6)
    onep = 1.0 + w.double().numpy()
    assert np.allclose(fw, f0 * onep[None, :], rtol=1e-15, atol=0)
    # Llama's convention would give w * x_norm: different
    assert not np.allclose(fw, f0 * w.double().numpy()[None, :])


def test_power_of_two_scale_invariance(orc):
    """With eps = 0, scaling a row by a power of two leaves every output bit unchanged."""
    h = _rows(4, 4, 512)
    w = (wl.normal(wl.stream_key(5), 512, 0.1)).to(torch.bfloat16)
    b0, _ = oracle.rmsnorm(h, w, 0.0)
    for k in (-20, -3, 7, 40):
        bk, _ = oracle.rmsnorm((h.float() * 2.0 ** k).to(torch.bfloat16), w, 0.0)
        assert np.array_equal(bk, b0), k


def test_constant_row_closed_form(orc):
    for c, eps in ((0.5, 1e-6), (-3.0, 1e-2), (1e-3, 1e-6)):
        cb = torch.full((1, 64), c, dtype=torch.bfloat16)
        _, f = oracle.rmsnorm(cb, torch.zeros(64, dtype=torch.bfloat16), eps)
        cv = float(cb[0, 0])
        assert np.allclose(f, cv / np.sqrt(cv * cv + eps), rtol=1e-14)


def test_rounding_is_direct_from_fp64(orc):
    """Every output is the bf16 nearest to its fp64 value."""
    h = _rows(6, 2, 256)
    w = (wl.normal(wl.stream_key(7), 256, 0.3)).to(torch.bfloat16)
    b, f = oracle.rmsnorm(h, w, 1e-6)
    for t in range(2):
        for i in range(0, 256, 17):
            assert b[t, i] == _nearest_bf16_brute(float(f[t, i]))


@pytest.mark.parametrize("batched", [False, True])
def test_residual_layer_with_zero_experts_is_identity(orc, batched):
    """All expert matrices zero: the layer adds nothing, y = h exactly."""
    shape = wl.TINY
    L = wl.LayerInputs(shape, seed=9)
    h = _rows(8, 3, shape.H, 2.0)
    w = (wl.normal(wl.stream_key(9), shape.H, 0.1)).to(torch.bfloat16)
    zero = lambda m: oracle.pack(m * 0)
    experts = {e: tuple(zero(m) for m in L.expert_f32(e)) for e in range(shape.E)}
    shared = tuple(zero(m) for m in L.shared_f32())
    res = oracle.moe_layer_residual(h, w, 1e-6, L.router_w("cpu"), L.shared_sigmoid_w("cpu"), experts, shared,
                                    shape.k, batched=batched)
    assert np.array_equal(res.y, h.double().numpy())


def test_residual_layer_composes_norm_and_layer(orc):
    """The residual form routes on, and feeds the experts with, the normalised bf16 rows."""
    shape = wl.TINY
    L = wl.LayerInputs(shape, seed=10)
    h = _rows(10, 4, shape.H, 3.0)
    w = (wl.normal(wl.stream_key(10), shape.H, 0.1)).to(torch.bfloat16)
    xb, _ = oracle.rmsnorm(h, w, 1e-6)
    ids, _, _ = oracle.route(oracle.router_logits(xb, L.router_w("cpu")), shape.k)
    experts = oracle_experts(L, ids)
    shared = oracle_shared(L)
    res = oracle.moe_layer_residual(h, w, 1e-6, L.router_w("cpu"), L.shared_sigmoid_w("cpu"), experts, shared,
                                    shape.k)
    plain = oracle.moe_layer(xb, L.router_w("cpu"), L.shared_sigmoid_w("cpu"), experts, shared, shape.k)
    assert np.array_equal(res.ids, plain.ids)
    assert np.array_equal(res.y, plain.y + h.double().numpy())
