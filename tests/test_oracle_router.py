"""Pins for the oracle's router: logits, softmax-all -> top-k -> renormalise.

The router is the one in the lynn-engine tutorials (row 06, MoE router):
softmax over all experts, keep the top k, renormalise. The tutorial states it
is mathematically the same as taking the top-k logits and applying softmax to
them; that identity, the sum-to-one property and a brute-force subset search
pin the oracle independently of its own code.
"""
import itertools

import numpy as np
import pytest
import torch

import workload as wl


def _softmax(v):
    v = np.asarray(v, np.float64)
    e = np.exp(v - v.max())
    return e / e.sum()


def test_router_logits_match_numpy(orc):
    x = wl.activations(3, 4, 64)
    wg = wl.normal(wl.stream_key(11), 10 * 64, 0.02).view(10, 64).to(torch.bfloat16)
    got = orc.router_logits(x, wg)
    want = x.double().numpy() @ wg.double().numpy().T
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("E,k", [(16, 2), (256, 8), (7, 7), (5, 1)])
def test_topk_then_softmax_identity(orc, E, k):
    rng = np.random.default_rng(E * 31 + k)
    logits = rng.normal(0, 0.5, size=(64, E))
    ids, w, p = orc.route(logits, k)
    for t in range(64):
        # top-k of the logits (same order as top-k of p: softmax is monotone)
        order = np.argsort(-logits[t], kind="stable")[:k]
        assert set(order.tolist()) == set(ids[t].tolist())
        sm = _softmax(logits[t, ids[t]])
        assert np.max(np.abs(sm - w[t])) <= 1e-12
        assert abs(w[t].sum() - 1.0) <= 1e-12
        assert np.all(np.diff(w[t]) <= 0)          # sorted, largest first
        assert np.allclose(p[t], _softmax(logits[t]), rtol=1e-12)


def test_topk_brute_force_subsets(orc):
    rng = np.random.default_rng(12)
    for E in range(2, 11):
        for k in range(1, min(3, E) + 1):
            logits = rng.normal(0, 1, size=(5, E))
            ids, w, p = orc.route(logits, k)
            for t in range(5):
                best = max(itertools.combinations(range(E), k), key=lambda s: sum(p[t, list(s)]))
                assert set(best) == set(ids[t].tolist())


def test_ties_lower_index_first(orc):
    logits = np.array([[0.0, 1.0, 1.0, 0.5, 1.0, 0.5]])
    ids, w, _ = orc.route(logits, 4)
    assert ids[0].tolist() == [1, 2, 4, 3]
    assert np.allclose(w[0, :3], w[0, 0])


def test_underflowed_probabilities_rank_by_logits(orc):
    """Logits 1000 apart: every p but the first underflows to 0 in fp64. softmax is
    monotone, so the top-k of p is still the top-k of the logits."""
    logits = np.array([[0.0, -1000.0, -2000.0, -1500.0, -3000.0]])
    ids, w, p = orc.route(logits, 4)
    assert np.all(p[0, 1:] == 0.0)
    assert ids[0].tolist() == [0, 1, 3, 2]
    assert w[0].tolist() == [1.0, 0.0, 0.0, 0.0]


def test_route_rejects_bad_k(orc):
    with pytest.raises(ValueError):
        orc.route(np.zeros((1, 4)), 5)
    with pytest.raises(ValueError):
        orc.route(np.zeros((1, 4)), 0)


def test_logit_gap_is_kth_minus_next(orc):
    """logit_gap (which tokens count as near ties in the parity tests): the k-th largest logit
    minus the (k+1)-th, whatever the order of the experts; infinite when every expert is
    selected."""
    lg = np.array([[0.5, 3.0, -1.0, 2.0, 2.75],      # sorted: 3, 2.75, 2, 0.5, -1
                   [1.0, 1.0, 1.0, 0.0, -2.0]])     # an exact tie at the boundary
    assert np.allclose(orc.logit_gap(lg, 1), [0.25, 0.0])
    assert np.allclose(orc.logit_gap(lg, 2), [0.75, 0.0])
    assert np.allclose(orc.logit_gap(lg, 3), [1.5, 1.0])
    assert np.all(np.isinf(orc.logit_gap(lg, 5)))
    rng = np.random.default_rng(3)
    r = rng.standard_normal((50, 16))
    for k in (1, 4, 8):
        s = -np.sort(-r, axis=1)
        assert np.array_equal(orc.logit_gap(r, k), s[:, k - 1] - s[:, k])
        assert np.array_equal(orc.logit_gap(r[:, rng.permutation(16)], k), orc.logit_gap(r, k))
