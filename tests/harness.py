"""Test-side helpers: build oracle inputs from the seeded generator.

Only the tests use this module. Oracle results come from ``oracle`` only; the
CUDA library's outputs are compared against them, never fed back.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workload as wl


def oracle_experts(L: wl.LayerInputs, ids, kind=oracle.SCALE_E4M3, cache=None):
    """Oracle-packed (gate, up, down) for every expert id in ``ids``."""
    out = {} if cache is None else cache
    for e in sorted(set(int(i) for i in np.asarray(ids).ravel())):
        if e in out:
            continue
        g, u, d = L.expert_f32(e, device="cpu")
        out[e] = (oracle.pack(g, kind), oracle.pack(u, kind), oracle.pack(d, kind))
    return out


def oracle_shared(L: wl.LayerInputs, kind=oracle.SCALE_E4M3):
    g, u, d = L.shared_f32(device="cpu")
    return (oracle.pack(g, kind), oracle.pack(u, kind), oracle.pack(d, kind))


def oracle_layer(L: wl.LayerInputs, x, kind=oracle.SCALE_E4M3, force_ids=None, cache=None,
                 with_shared=True):
    """Full oracle layer for tokens x (bf16 [T,H]) on layer L (packs only the experts it needs)."""
    wg = L.router_w("cpu")
    logits = oracle.router_logits(x, wg)
    ids, _, _ = oracle.route(logits, L.shape.k)
    need = ids if force_ids is None else np.asarray(force_ids)
    experts = oracle_experts(L, need, kind, cache)
    shared = oracle_shared(L, kind) if with_shared else None
    res = oracle.moe_layer(x, wg, L.shared_sigmoid_w("cpu"), experts, shared, L.shape.k, kind,
                           force_ids=force_ids)
    return res, logits


def margin_tokens(L: wl.LayerInputs, seed: int, T: int, gap: float = 1e-3, max_attempts: int = 64,
                  layer: int = 0):
    """x [T,H] bf16 where every token's k-th/(k+1)-th router logit gap exceeds ``gap``
    (a token is redrawn from its seed stream until it does); returns (x, attempts)."""
    wg = L.router_w("cpu")
    attempts = [0] * T
    x = wl.activations(seed, T, L.shape.H, layer=layer, attempts=attempts)
    for _ in range(max_attempts):
        g = oracle.logit_gap(oracle.router_logits(x, wg), L.shape.k)
        bad = [t for t in range(T) if not g[t] > gap]
        if not bad:
            return x, attempts
        for t in bad:
            attempts[t] += 1
        x = wl.activations(seed, T, L.shape.H, layer=layer, attempts=attempts)
    raise RuntimeError("could not draw margin tokens")


def tol_ok(gpu: np.ndarray, ref: np.ndarray, rel=1e-2, abs_=1e-3):
    """max|gpu - ref| <= rel * max|ref| + abs (per output tensor)."""
    err = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    bound = rel * (float(np.max(np.abs(ref))) if ref.size else 0.0) + abs_
    return err <= bound, err, bound


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_layer(L: wl.LayerInputs, kind=0, device="cuda", with_shared=True):
    """Device layer in the library's layout, every expert packed on the GPU by nvfp4_pack."""
    import nvfp4_w4a16_moe_gb300 as nv
    s = L.shape
    Is = s.Is if with_shared else 0
    layer = nv.MoELayer.allocate(s.H, s.E, s.k, s.I, Is, kind, device)
    layer.router_w.copy_(L.router_w(device))
    for e in range(s.E):
        layer.pack_expert(e, *L.expert_f32(e, device=device))
    if with_shared:
        layer.pack_shared(*L.shared_f32(device=device), L.shared_sigmoid_w(device))
    return layer


def check_layer_parity(L: wl.LayerInputs, x_gpu, y_gpu, ids_gpu, w_gpu, kind=0, with_shared=True,
                       cache=None, gap_min=1e-3, rel_only=None):
    """Compare one GPU layer call with the oracle. Tokens whose k-th/(k+1)-th logit gap
    is <= gap_min are re-evaluated by the oracle on the GPU's expert set (several
    routings are correct there). With ``rel_only`` the error must also stay within
    rel_only * max|oracle| (no absolute term). Returns (err, bound, n_near_ties)."""
    x = x_gpu.cpu()
    ids_g = ids_gpu.cpu().numpy()
    w_g = w_gpu.cpu().numpy()
    res, logits = oracle_layer(L, x, kind, cache=cache, with_shared=with_shared)
    gap = oracle.logit_gap(logits, L.shape.k)
    near = gap <= gap_min
    for t in np.flatnonzero(~near):
        assert sorted(ids_g[t].tolist()) == sorted(res.ids[t].tolist()), (t, ids_g[t], res.ids[t])
        # weights compared by expert id
        wo = dict(zip(res.ids[t].tolist(), res.w[t].tolist()))
        for e, wv in zip(ids_g[t].tolist(), w_g[t].tolist()):
            assert abs(wv - wo[e]) <= 1e-5, (t, e, wv, wo[e])
    ref = res.y
    if near.any():
        forced = res.ids.copy()
        forced[near] = ids_g[near]
        ref2, _ = oracle_layer(L, x, kind, force_ids=forced, cache=cache, with_shared=with_shared)
        ref = ref2.y
    got = y_gpu.float().cpu().numpy().astype(np.float64)
    ok, err, bound = tol_ok(got, ref)
    assert ok, "max|gpu-oracle| %.4g > %.4g" % (err, bound)
    if rel_only is not None:
        ok2, err2, bound2 = tol_ok(got, ref, rel=rel_only, abs_=0.0)
        assert ok2, "max|gpu-oracle| %.4g > %.4g (scale-free)" % (err2, bound2)
    return err, bound, int(near.sum())
