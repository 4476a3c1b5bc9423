"""Pins for the oracle's many-token form of the layer (oracle.moe_layer_batched).

It is the same definition as oracle.moe_layer (lynn-engine tutorials index, row
06: softmax over all experts, top-k, renormalise, sigmoid-gated shared expert;
README P28/P29 notes: SwiGLU experts and the weighted sum), evaluated expert by
expert with numpy's fp64 matmul as the library step. Its pieces are pinned here
against the per-token C oracle (itself pinned to textbook routines, closed forms
and brute force in test_oracle_*.py): the table dequantiser bit for bit, the
layer within fp64 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import oracle_experts, oracle_shared


def _rand_packed(kind, N, K, key, scale_exp=0):
    w = wl.normal(wl.stream_key(key), N * K, 0.02 * 2.0 ** scale_exp).view(N, K)
    return oracle.pack(w, kind)


@pytest.mark.parametrize("kind", [0, 1, 2, 3])
@pytest.mark.parametrize("scale_exp", [-30, 0, 20])
def test_table_dequant_is_bit_exact(orc, kind, scale_exp):
    p = _rand_packed(kind, 33, 96, 7 + kind, scale_exp)
    assert np.array_equal(oracle.dequant_table(p), oracle.dequant(p))


@pytest.mark.parametrize("kind", [0, 1])
def test_table_dequant_every_code_and_scale(orc, kind):
    """Every E2M1 code against every E4M3 scale byte (or a spread of FP16 codes)."""
    scodes = np.arange(256) if kind == 0 else np.arange(0, 65536, 257)
    scodes = scodes[[oracle.e4m3_decode(int(b)) == oracle.e4m3_decode(int(b)) for b in scodes]] if kind == 0 \
        else scodes[[np.isfinite(oracle.fp16_decode(int(b))) for b in scodes]]
    N, K = len(scodes), 16
    packed = np.tile(np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], np.uint8), (N, 1))
    scales = scodes.astype(np.uint8 if kind == 0 else np.uint16).reshape(N, 1)
    p = oracle.Packed(packed, scales, 0.75, kind, N, K)
    assert np.array_equal(oracle.dequant_table(p), oracle.dequant(p))


def test_swiglu_rows_equals_c_swiglu(orc):
    H, I = 128, 64
    g, u, d = (_rand_packed(0, I, H, 11), _rand_packed(0, I, H, 12), _rand_packed(0, H, I, 13))
    x = wl.activations(3, 5, H)
    got = oracle.swiglu_rows(g, u, d, oracle.bf16_rows(x))
    want = oracle.swiglu(g, u, d, x)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def _layer_pair(shape, seed, T, force=False, with_shared=True, kind=0):
    L = wl.LayerInputs(shape, seed=seed)
    x = wl.activations(seed, T, shape.H)
    wg = L.router_w("cpu")
    sgv = L.shared_sigmoid_w("cpu")
    lg = oracle.router_logits(x, wg)
    ids, _, _ = oracle.route(lg, shape.k)
    force_ids = None
    if force:
        # a different valid expert set per token: the ranks k-1 and k swapped
        order = np.argsort(-lg, axis=1, kind="stable")
        force_ids = order[:, :shape.k].copy()
        force_ids[:, -1] = order[:, shape.k]
        ids = force_ids
    experts = oracle_experts(L, ids, kind)
    shared = oracle_shared(L, kind) if with_shared else None
    a = oracle.moe_layer(x, wg, sgv, experts, shared, shape.k, kind, force_ids=force_ids)
    b = oracle.moe_layer_batched(x, wg, sgv, experts, shared, shape.k, force_ids=force_ids)
    return a, b


@pytest.mark.parametrize("shape,T,force,with_shared,kind", [
    (wl.TINY, 9, False, True, 0), (wl.TINY, 6, True, True, 1), (wl.SMALL256, 5, False, False, 0),
    (wl.QWEN36_35B_A3B, 2, False, True, 0), (wl.QWEN36_35B_A3B, 1, True, True, 0)])
def test_batched_layer_equals_per_token_layer(orc, shape, T, force, with_shared, kind):
    a, b = _layer_pair(shape, 17 + T, T, force, with_shared, kind)
    assert np.array_equal(a.ids, b.ids)
    assert np.allclose(a.w, b.w, rtol=1e-14, atol=0)
    assert np.allclose(a.sigmoid, b.sigmoid, rtol=1e-13, atol=0)
    assert np.max(np.abs(a.y - b.y)) <= 1e-12 * np.max(np.abs(a.y))


def test_batched_layer_with_external_expert_rows(orc):
    """The hook the tests use to evaluate experts in worker processes gives the same result."""
    shape = wl.TINY
    L = wl.LayerInputs(shape, seed=4)
    x = wl.activations(4, 12, shape.H)
    wg, sgv = L.router_w("cpu"), L.shared_sigmoid_w("cpu")
    ids, _, _ = oracle.route(oracle.router_logits(x, wg), shape.k)
    experts = oracle_experts(L, ids)
    shared = oracle_shared(L)
    xr = oracle.bf16_rows(x)
    calls = []

    def rows(e, tt):
        calls.append(e)
        return oracle.swiglu_rows(*experts[e], xr[tt])

    a = oracle.moe_layer_batched(x, wg, sgv, experts, shared, shape.k)
    b = oracle.moe_layer_batched(x, wg, sgv, {}, shared, shape.k, expert_rows=rows)
    assert np.array_equal(a.y, b.y)
    assert sorted(calls) == sorted(set(int(e) for e in ids.ravel()))


def test_parity_check_in_worker_pool(orc):
    """The full-size parity checker (experts evaluated in spawned worker processes) accepts
    the oracle's own bf16-rounded output and rejects it with one element moved past the bar
    (2 % of the output's largest magnitude plus 2e-3)."""
    from harness import ParityCheck, oracle_layer
    shape = wl.TINY
    L = wl.LayerInputs(shape, seed=21)
    T = 40
    x = wl.activations(21, T, shape.H)
    res, _ = oracle_layer(L, x)
    y = torch.tensor(res.y, dtype=torch.float32).to(torch.bfloat16)
    ids = torch.tensor(res.ids)
    w = torch.tensor(res.w, dtype=torch.float32)
    err, bound, near = ParityCheck(L, x, y, ids, w).check()
    assert err <= bound
    bad = y.float().clone()
    bad[T // 2, 7] += 0.02 * float(np.abs(res.y).max()) + 2e-3
    with pytest.raises(AssertionError):
        ParityCheck(L, x, bad.to(torch.bfloat16), ids, w).check()
