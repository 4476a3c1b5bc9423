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


# ------------------------------------------------------------------------------------
# The oracle at full size: every token of a call, with the routed experts evaluated in
# worker processes (oracle.moe_layer_batched with its expert_rows hook). Workers are
# started with "spawn" (never forked from a process that holds a CUDA context), one
# BLAS / OpenMP thread each.

_POOL = None
_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")


def _worker_init():
    torch.set_num_threads(1)


def oracle_pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        import os
        for k in _THREAD_ENV:
            os.environ[k] = "1"     # read by the workers' numpy / torch at import
        n = max(1, min(48, os.cpu_count() or 1))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"),
                                       initializer=_worker_init)
    return _POOL


def _expert_rows_task(shape, seed, layer, kind, e, xbits):
    """SwiGLU rows of routed expert e (redrawn from its seed, packed by the oracle) for the
    given bf16 token rows."""
    L = wl.LayerInputs(shape, seed=seed, layer=layer)
    packs = [oracle.pack(m, kind) for m in L.expert_f32(e, device="cpu")]
    return oracle.swiglu_rows(*packs, oracle.bf16_rows(xbits))


class OracleJob:
    """One oracle layer evaluation of x (bf16 [T, H]) on layer L, its experts submitted to
    the worker pool at construction; result() assembles the layer."""

    def __init__(self, L: wl.LayerInputs, x, kind=oracle.SCALE_E4M3, force_ids=None, with_shared=True,
                 logits=None):
        self.L, self.kind, self.with_shared = L, kind, with_shared
        self.x = x
        self.wg = L.router_w("cpu")
        if logits is None:
            logits = oracle.router_logits(x, self.wg)
        self.logits = logits
        ids, w, p = oracle.route(logits, L.shape.k)
        if force_ids is not None:
            ids = np.asarray(force_ids, np.int32).copy()
            w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
            w = w / w.sum(axis=1, keepdims=True)
        self.ids, self.w = ids, w
        xb = oracle._np(x, np.uint16)
        pool = oracle_pool()
        self.fut = {}
        for e in np.unique(ids):
            tt, _ = np.nonzero(ids == e)
            self.fut[int(e)] = pool.submit(_expert_rows_task, L.shape, L.seed, L.layer, kind, int(e), xb[tt])

    def result(self) -> oracle.LayerResult:
        shared = oracle_shared(self.L, self.kind) if self.with_shared else None

        def rows(e, tt):
            r = self.fut[e].result()
            assert r.shape[0] == len(tt)
            return r
        return oracle.moe_layer_batched(self.x, self.wg, self.L.shared_sigmoid_w("cpu"), {}, shared,
                                        self.L.shape.k, expert_rows=rows, routing=(self.ids, self.w))


class ParityCheck:
    """check_layer_parity for every token of a large call, with the oracle in the worker pool.
    Construction submits the work (so that many layers can be in flight at once); check()
    asserts the same bar as check_layer_parity and returns (err, bound, n_near_ties)."""

    def __init__(self, L: wl.LayerInputs, x_gpu, y_gpu, ids_gpu, w_gpu, kind=0, with_shared=True,
                 gap_min=1e-3, rel_only=None):
        self.x = x_gpu.cpu()
        self.y = y_gpu.float().cpu().numpy().astype(np.float64)
        self.ids_g = ids_gpu.cpu().numpy()
        self.w_g = w_gpu.cpu().numpy()
        self.rel_only = rel_only
        self.job = OracleJob(L, self.x, kind, with_shared=with_shared)
        gap = oracle.logit_gap(self.job.logits, L.shape.k)
        self.near = np.flatnonzero(gap <= gap_min)
        self.job_near = None
        if self.near.size:
            idx = torch.tensor(self.near, dtype=torch.long)
            self.job_near = OracleJob(L, self.x[idx], kind, force_ids=self.ids_g[self.near],
                                      with_shared=with_shared, logits=self.job.logits[self.near])

    def check(self):
        res = self.job.result()
        clear = np.ones(len(self.ids_g), bool)
        clear[self.near] = False
        ids_o = res.ids
        assert np.array_equal(np.sort(self.ids_g[clear], 1), np.sort(ids_o[clear], 1)), "expert ids differ"
        # weights by expert id: sort both sides by id
        og = np.argsort(self.ids_g, 1, kind="stable")
        oo = np.argsort(ids_o, 1, kind="stable")
        wg = np.take_along_axis(self.w_g, og, 1)[clear]
        wo = np.take_along_axis(res.w, oo, 1)[clear]
        if wg.size:
            assert float(np.abs(wg - wo).max()) <= 1e-5, float(np.abs(wg - wo).max())
        ref = res.y.copy()
        if self.job_near is not None:
            ref[self.near] = self.job_near.result().y
        ok, err, bound = tol_ok(self.y, ref)
        assert ok, "max|gpu-oracle| %.4g > %.4g" % (err, bound)
        if self.rel_only is not None:
            ok2, err2, bound2 = tol_ok(self.y, ref, rel=self.rel_only, abs_=0.0)
            assert ok2, "max|gpu-oracle| %.4g > %.4g (scale-free)" % (err2, bound2)
        return err, bound, int(self.near.size)


class single_token_form:
    """Run the enclosed calls with the given single-token kernel form (1 the persistent-grid
    form, 2 the cluster form where supported), then restore automatic (the grid form)."""

    def __init__(self, nv, form: int):
        self.nv, self.form = nv, form

    def __enter__(self):
        self.nv.set_single_token_form(self.form)
        return self

    def __exit__(self, *exc):
        self.nv.set_single_token_form(0)
        return False
