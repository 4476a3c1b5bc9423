"""The stored skew record of the 4096-token prefill workload (tests/golden/prefill_zipf.json) is
self-consistent, and its rank-count slope is what the fit gives on the stored counts; the fit
itself is pinned on exact Zipf counts, where the slope is the exponent."""
import importlib.util
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _writer():
    spec = importlib.util.spec_from_file_location("make_prefill_zipf",
                                                  os.path.join(HERE, "golden", "make_prefill_zipf.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_slope_of_exact_zipf_counts_is_the_exponent():
    fit = _writer().rank_count_slope
    r = np.arange(1, 257, dtype=np.float64)
    for alpha in (0.5, 1.1, 2.0):
        c = 1000.0 * r ** -alpha
        assert abs(fit(c) - alpha) < 1e-12
        assert abs(fit(c, 32) - alpha) < 1e-12
    # the order of the experts does not matter; empty experts are left out of the fit
    c = 1000.0 * r ** -1.1
    rng = np.random.default_rng(0)
    assert abs(fit(rng.permutation(np.append(c, [0.0, 0.0]))) - 1.1) < 1e-12


def test_stored_skew_record_is_consistent():
    g = json.load(open(os.path.join(HERE, "golden", "prefill_zipf.json")))
    c = np.asarray(g["counts"])
    assert c.size == g["E"] and int(c.sum()) == g["T"] * g["k"]
    assert int(c.max()) == g["max_count"] and int(c.min()) == g["min_count"]
    assert int((c == 0).sum()) == g["empty_experts"]
    fit = _writer().rank_count_slope
    assert abs(fit(c) - g["rank_count_slope_all"]) < 1e-4
    assert abs(fit(c, 32) - g["rank_count_slope_top32"]) < 1e-4
    # the realised popularity is skewed but flatter than the Zipf(1.1) the workload names
    assert 0.0 < g["rank_count_slope_top32"] < g["rank_count_slope_all"] < g["zipf_target"]
