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
