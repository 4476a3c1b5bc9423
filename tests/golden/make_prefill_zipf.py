"""Writes prefill_zipf.json: the router skew exponent kappa of the 4096-token
prefill workload (Qwen3.6-35B-A3B-shaped layer, seed 2) and the per-expert
token counts it gives.

The workload asks for a Zipf(1.1)-skewed expert popularity with per-expert
counts from about 0 to about 1000 for 4096 tokens and top-8 routing. A router
with no bias can only skew popularity through the scale of its rows, so router
row e is scaled by rank_e^-kappa (rank = a seeded permutation of 1..E), and
kappa is found by bisection so that the busiest expert receives about 1000 of
the 4096*8 entries. Counts come from the oracle's fp64 router and top-k only.
The file also records how far the realised popularity is from Zipf(1.1): the
least-squares slope of log(count) against log(rank) over all experts and over
the 32 busiest (a Zipf(alpha) popularity has slope alpha).

Run from the repository root:  python tests/golden/make_prefill_zipf.py
"""
import json
import os
import sys
from dataclasses import replace

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workload as wl  # noqa: E402

T, SEED, TARGET_MAX = 4096, 2, 1000


def counts_for(kappa: float, x) -> np.ndarray:
    shape = replace(wl.QWEN36_35B_A3B, router_kappa=kappa)
    L = wl.LayerInputs(shape, seed=SEED)
    logits = oracle.router_logits(x, L.router_w("cpu"))
    ids, _, _ = oracle.route(logits, shape.k)
    return np.bincount(ids.ravel(), minlength=shape.E)


def rank_count_slope(c: np.ndarray, top: int = 0) -> float:
    """Least-squares slope s of log(count) = a - s log(rank) over the experts with entries,
    ranked by count (rank 1 = busiest); top > 0 fits the `top` busiest only. A Zipf(alpha)
    popularity gives s = alpha."""
    v = np.sort(np.asarray(c, np.float64))[::-1]
    v = v[v > 0]
    if top:
        v = v[:top]
    r = np.arange(1, len(v) + 1, dtype=np.float64)
    A = np.stack([np.ones_like(r), -np.log(r)], axis=1)
    coef, *_ = np.linalg.lstsq(A, np.log(v), rcond=None)
    return float(coef[1])


def main():
    oracle.build()
    x = wl.activations(SEED, T, wl.QWEN36_35B_A3B.H)
    lo, hi = 0.0, 2.0
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        if counts_for(mid, x).max() < TARGET_MAX:
            lo = mid
        else:
            hi = mid
    kappa = round(hi, 4)
    c = counts_for(kappa, x)
    out = {
        "what": "router skew exponent of the 4096-token prefill workload (seed 2) and its per-expert counts",
        "T": T, "seed": SEED, "k": wl.QWEN36_35B_A3B.k, "E": wl.QWEN36_35B_A3B.E,
        "kappa": kappa,
        "max_count": int(c.max()), "min_count": int(c.min()),
        "empty_experts": int((c == 0).sum()),
        "zipf_target": 1.1,
        "rank_count_slope_all": round(rank_count_slope(c), 4),
        "rank_count_slope_top32": round(rank_count_slope(c, 32), 4),
        "counts": [int(v) for v in c],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "prefill_zipf.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("kappa", kappa, "max", c.max(), "min", c.min(), "empty", (c == 0).sum(),
          "slope", out["rank_count_slope_all"], out["rank_count_slope_top32"])


if __name__ == "__main__":
    main()
