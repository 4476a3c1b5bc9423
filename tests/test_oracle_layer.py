"""Pins for the oracle's GEMV and MoE layer.

Reductions to textbook routines (numpy matmul on the dequantised matrices),
exact dyadic results, and invariants of the layer (identical experts make the
routing irrelevant because renormalised weights sum to one; relabelling the
experts; per-token independence; top-k order independence, as in the
lynn-engine README, P20 note: unsorted top-k gives the same expert set, the same
paired weights and the same output).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import oracle_layer


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _dense_swiglu(orc, g, u, d, x):
    G, U, D = orc.dequant(g), orc.dequant(u), orc.dequant(d)
    xv = x.double().numpy()
    return (_silu(xv @ G.T) * (xv @ U.T)) @ D.T


@pytest.mark.parametrize("kind", [0, 1])
def test_gemv_equals_numpy_matmul(orc, kind):
    w = wl.normal(wl.stream_key(21), 40 * 96, 0.02).view(40, 96)
    x = wl.activations(21, 3, 96)
    p = orc.pack(w, kind)
    got = orc.gemv(p, x)
    want = x.double().numpy() @ orc.dequant(p).T
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def test_gemv_dyadic_exact(orc):
    """On-grid weights with power-of-two scales and integer activations give an exact result."""
    rng = np.random.default_rng(22)
    N, K = 9, 64
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, ::16] = 7
    sexp = rng.integers(-3, 4, size=(N, K // 16))
    mags = np.array([oracle.e2m1_decode(int(c)) for c in codes.ravel()]).reshape(N, K)
    W = (mags * np.repeat(2.0 ** sexp, 16, axis=1)).astype(np.float32)
    p = orc.pack(W, 1)        # FP16 scales: tensor scale 1, block scales exact powers of two
    xi = rng.integers(-8, 9, size=(2, K))
    x = torch.tensor(xi, dtype=torch.bfloat16)
    got = orc.gemv(p, x)
    for t in range(2):
        for n in range(N):
            exact = sum(Fraction(float(W[n, k])) * int(xi[t, k]) for k in range(K))
            assert Fraction(got[t, n]) == exact


def _packs(orc, shape, key, kind=0, zero=False):
    H, I = shape
    g = wl.normal(wl.stream_key(key, 1), I * H, 0.02).view(I, H)
    u = wl.normal(wl.stream_key(key, 2), I * H, 0.02).view(I, H)
    d = wl.normal(wl.stream_key(key, 3), H * I, 0.02).view(H, I)
    if zero:
        g, u, d = g * 0, u * 0, d * 0
    return orc.pack(g, kind), orc.pack(u, kind), orc.pack(d, kind)


def test_single_expert_reduces_to_dense_swiglu(orc):
    H, I = 64, 32
    x = wl.activations(5, 3, H)
    wg = torch.zeros(1, H, dtype=torch.bfloat16)
    e0 = _packs(orc, (H, I), 30)
    zero_sh = _packs(orc, (H, I), 31, zero=True)
    sgv = wl.normal(wl.stream_key(32), H, 0.02).to(torch.bfloat16)
    res = orc.moe_layer(x, wg, sgv, {0: e0}, zero_sh, k=1)
    want = _dense_swiglu(orc, *e0, x)
    assert np.allclose(res.y, want, rtol=1e-12, atol=1e-14)
    assert np.all(res.w == 1.0) and np.all(res.ids == 0)
    # and without any shared expert at all
    res2 = orc.moe_layer(x, wg, sgv, {0: e0}, None, k=1)
    assert np.allclose(res2.y, want, rtol=1e-12, atol=1e-14)


def test_identical_experts_make_routing_irrelevant(orc):
    H, I, E, k = 64, 32, 6, 3
    x = wl.activations(6, 4, H)
    wg = wl.normal(wl.stream_key(33), E * H, 0.5).view(E, H).to(torch.bfloat16)
    same = _packs(orc, (H, I), 34)
    sh = _packs(orc, (H, 48), 35)
    sgv = wl.normal(wl.stream_key(36), H, 0.3).to(torch.bfloat16)
    res = orc.moe_layer(x, wg, sgv, {e: same for e in range(E)}, sh, k=k)
    sig = 1.0 / (1.0 + np.exp(-(x.double().numpy() @ sgv.double().numpy())))
    want = _dense_swiglu(orc, *same, x) + sig[:, None] * _dense_swiglu(orc, *sh, x)
    assert np.allclose(res.y, want, rtol=1e-11, atol=1e-14)
    assert np.allclose(res.sigmoid, sig, rtol=1e-14)


def test_shared_only_when_routed_down_is_zero(orc):
    H, I, E = 64, 32, 4
    x = wl.activations(7, 2, H)
    wg = wl.normal(wl.stream_key(37), E * H, 0.5).view(E, H).to(torch.bfloat16)
    experts = {}
    for e in range(E):
        g, u, _ = _packs(orc, (H, I), 40 + e)
        experts[e] = (g, u, _packs(orc, (H, I), 0, zero=True)[2])
    sh = _packs(orc, (H, I), 39)
    sgv = wl.normal(wl.stream_key(38), H, 0.3).to(torch.bfloat16)
    res = orc.moe_layer(x, wg, sgv, experts, sh, k=2)
    sig = 1.0 / (1.0 + np.exp(-(x.double().numpy() @ sgv.double().numpy())))
    assert np.allclose(res.y, sig[:, None] * _dense_swiglu(orc, *sh, x), rtol=1e-12, atol=1e-15)


def test_relabelling_experts_is_invariant(orc):
    H, I, E, k = 64, 32, 8, 2
    x = wl.activations(8, 5, H)
    wg = wl.normal(wl.stream_key(50), E * H, 0.3).view(E, H).to(torch.bfloat16)
    experts = {e: _packs(orc, (H, I), 60 + e) for e in range(E)}
    sh = _packs(orc, (H, I), 59)
    sgv = wl.normal(wl.stream_key(51), H, 0.3).to(torch.bfloat16)
    base = orc.moe_layer(x, wg, sgv, experts, sh, k=k)
    perm = [5, 2, 7, 0, 3, 6, 1, 4]            # new id of old expert e is perm[e]
    wg2 = torch.zeros_like(wg)
    ex2 = {}
    for e in range(E):
        wg2[perm[e]] = wg[e]
        ex2[perm[e]] = experts[e]
    res = orc.moe_layer(x, wg2, sgv, ex2, sh, k=k)
    assert np.allclose(res.y, base.y, rtol=1e-13, atol=1e-16)
    inv = {perm[e]: e for e in range(E)}
    for t in range(5):
        assert sorted(inv[i] for i in res.ids[t]) == sorted(base.ids[t].tolist())


def test_tokens_are_independent_and_topk_order_free(orc):
    L = wl.LayerInputs(wl.TINY, seed=0)
    x = wl.activations(0, 5, 256)
    res, _ = oracle_layer(L, x)
    for t in range(5):
        r1, _ = oracle_layer(L, x[t:t + 1])
        assert np.allclose(r1.y[0], res.y[t], rtol=1e-13, atol=1e-16)
    # P20: same expert set in another order gives the same output
    rev = res.ids[:, ::-1].copy()
    r2, _ = oracle_layer(L, x, force_ids=rev)
    assert np.allclose(r2.y, res.y, rtol=1e-12, atol=1e-16)


def test_tiny_layer_scale(orc):
    """Config-0 layer output is finite, O(0.1), and depends on both routed and shared parts."""
    L = wl.LayerInputs(wl.TINY, seed=0)
    x = wl.activations(0, 1, 256)
    res, logits = oracle_layer(L, x)
    assert np.all(np.isfinite(res.y))
    assert 1e-3 < np.abs(res.y).max() < 10
    no_sh, _ = oracle_layer(L, x, with_shared=False)
    assert not np.allclose(no_sh.y, res.y)


def test_forced_expert_set_renormalises_over_it(orc):
    """The tests re-evaluate near-tie tokens on the GPU's expert set: with forced
    ids the layer must be sum_j w'_j SwiGLU_j(x) + sigmoid(gs.x) SwiGLU_s(x), w' the
    softmax of the forced experts' logits (the renormalised probabilities)."""
    H, I, E, k = 64, 32, 6, 2
    x = wl.activations(9, 3, H)
    wg = wl.normal(wl.stream_key(70), E * H, 0.4).view(E, H).to(torch.bfloat16)
    experts = {e: _packs(orc, (H, I), 80 + e) for e in range(E)}
    sh = _packs(orc, (H, I), 79)
    sgv = wl.normal(wl.stream_key(71), H, 0.3).to(torch.bfloat16)
    base = orc.moe_layer(x, wg, sgv, experts, sh, k=k)
    forced = np.array([[e for e in range(E) if e not in base.ids[t]][:k] for t in range(3)], np.int32)
    res = orc.moe_layer(x, wg, sgv, experts, sh, k=k, force_ids=forced)
    logits = x.double().numpy() @ wg.double().numpy().T
    sig = 1.0 / (1.0 + np.exp(-(x.double().numpy() @ sgv.double().numpy())))
    shared = _dense_swiglu(orc, *sh, x)
    for t in range(3):
        l = logits[t, forced[t]]
        wt = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
        want = sum(wt[j] * _dense_swiglu(orc, *experts[int(forced[t, j])], x[t:t + 1])[0] for j in range(k))
        want = want + sig[t] * shared[t]
        assert np.allclose(res.y[t], want, rtol=1e-11, atol=1e-15)
        assert sorted(res.ids[t].tolist()) == sorted(forced[t].tolist())


@pytest.mark.parametrize("kind", [0, 1])
def test_orc_swiglu_equals_dense_swiglu(orc, kind):
    """The oracle's single-expert entry point (bf16 tokens in, fp64 out) is the textbook
    SwiGLU on the dequantised matrices, token by token."""
    H, I = 96, 64
    g, u, d = _packs(orc, (H, I), 40 + kind, kind)
    x = wl.activations(40 + kind, 4, H)
    got = orc.swiglu(g, u, d, x)
    want = _dense_swiglu(orc, g, u, d, x)
    assert got.shape == (4, H)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)
    # one token at a time gives the same rows
    for t in range(4):
        assert np.array_equal(orc.swiglu(g, u, d, x[t:t + 1])[0], got[t])
