"""moe_route_topk on the GPU against the oracle's router tail.

Both sides see the same fp32 logits, so the expert order (descending
probability, lower id on exact ties) is compared exactly; renormalised weights
within 1e-6; the per-expert offsets and token lists are integer work and must be
bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workload as wl

pytestmark = pytest.mark.gpu


def _expected_lists(ids, E):
    T, k = ids.shape
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")      # entries grouped by expert, ascending entry
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, order.astype(np.int32)


def _check(nv, logits, k):
    T, E = logits.shape
    ids, w, off, tl = nv.moe_route_topk(logits.cuda(), k)
    torch.cuda.synchronize()
    rid, rw, _ = oracle.route(logits.double().numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(w.cpu().numpy() - rw).max() <= 1e-6
    assert np.allclose(w.cpu().double().numpy().sum(1), 1.0, atol=1e-6)
    eo, etl = _expected_lists(rid, E)
    assert np.array_equal(off.cpu().numpy(), eo)
    assert np.array_equal(tl.cpu().numpy(), etl)


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (64, 256, 8), (5, 16, 2), (3, 8, 8), (1, 1, 1),
                                   (37, 100, 3), (4096, 256, 8), (2000, 64, 6)])
def test_route_random(nv, T, E, k):
    logits = wl.normal(wl.stream_key(200, T, E, k), T * E, 1.0).view(T, E)
    _check(nv, logits, k)


def test_route_exact_ties(nv):
    # logits on a coarse grid: many exact ties, resolved towards the lower id
    z = wl.normal(wl.stream_key(201), 64 * 256, 1.0).view(64, 256)
    logits = torch.round(z * 2) / 2
    _check(nv, logits, 8)
    _check(nv, torch.zeros(4, 32), 5)


def test_route_large_magnitudes(nv):
    z = wl.normal(wl.stream_key(202), 16 * 256, 1.0).view(16, 256) * 80.0
    _check(nv, z, 8)
