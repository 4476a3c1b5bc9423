"""Benchmark: single-token decode through a Qwen3.6-35B-A3B-shaped NVFP4 MoE layer.

One step = one token through one MoE layer (router GEMV, softmax-all -> top-8 ->
renormalise, 8 routed SwiGLU experts + sigmoid-gated shared expert, combine),
hidden 2048, 256 experts, intermediate 512, E4M3 block scales. Steps rotate over
32 independently seeded layer instances (seeds 0..31, ~14.5 GB of packed
weights), so consecutive steps never hit the same weights in L2 (129 MB).

Prints one JSON line. ``--impl reference`` times the CPU oracle instead (the
reference arm for this build), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 MoE-layer decode: µs/token and achieved HBM GB/s as % of GB300 peak"
UNIT = "us/token"
N_SEEDS = 32
WORKLOAD = ("qwen3.6-35b-a3b-shaped MoE layer decode, T=1 token/step, H=2048 E=256 top-8 I=512 "
            "shared Is=512 sigmoid gate, NVFP4 E4M3 per-16 scales, seeds 0..31")


CHAIN_LAYERS = 40   # layers of the batched decode step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--seeds", type=int, default=N_SEEDS, help="layer instances to rotate over")
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "batched", "gemv", "lm_head"],
                    help="decode: the single-token layer (default, the headline); prefill: one "
                         "4096-token layer call with the skewed router; batched: one --tokens-token "
                         "decode call per step; gemv: the dense W4A16 GEMV, 1 token, K=2048 -> N=8192 "
                         "(and the lm_head); lm_head: the 248320 x 2048 lm_head GEMV alone")
    ap.add_argument("--tokens", type=int, default=64, help="tokens per call of --workload batched (1..64)")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload: time only the single-token steps (skip the batched, 40-layer, "
                         "GEMV and prefill figures)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replicas_timing(ms_local: float, steps: int, world: int, device=None):
    """Whole-job timing of N independent replicas: the timed region's maximum over
    ranks (the job ends when the slowest replica does), then microseconds per token
    over the tokens all ranks processed (each rank runs `steps` single-token steps).
    Every rank returns the same (ms, us_per_token)."""
    ms = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, 1e3 * ms / (steps * world)


def ncu_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu capture, or
    None when the kernel source changed since that capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "moe_decode_t1_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    sp = os.path.join(ROOT, d["source"])
    if not os.path.exists(sp):
        return None
    src = open(sp, "rb").read()
    if hashlib.sha256(src).hexdigest()[:16] != d["source_sha256_prefix"]:
        return None
    return d["dram_bytes_read"] + d["dram_bytes_write"]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (median SM clock, throttle reasons)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------ oracle arm

def _oracle_token_inputs(seed):
    """Everything the oracle needs for one single-token step of layer instance ``seed``
    (the experts its router picks, packed beforehand as the GPU's weights are)."""
    import oracle
    import workload as wl
    shape = wl.QWEN36_35B_A3B
    L = wl.LayerInputs(shape, seed=seed % N_SEEDS)
    x = wl.activations(seed % N_SEEDS, 1, shape.H)
    wg = L.router_w("cpu")
    ids, _, _ = oracle.route(oracle.router_logits(x, wg), shape.k)
    experts = {e: tuple(oracle.pack(m) for m in L.expert_f32(e)) for e in ids.ravel().tolist()}
    shared = tuple(oracle.pack(m) for m in L.shared_f32())
    return x, wg, L.shared_sigmoid_w("cpu"), experts, shared, shape.k


def cpu_oracle_sample(budget_s: float, threads: int = 1, max_tokens: int = 64):
    """Time the CPU oracle on single-token steps of the same workload, one token per layer
    instance (seeds 0..31 in turn). threads = 1: tokens one after another, ~budget_s of
    oracle time. threads > 1: 2 * threads tokens run concurrently on that many host threads
    (each a plain oracle call; ctypes releases the GIL), timed by the wall clock.
    Returns (us_per_token, tokens, seconds)."""
    import concurrent.futures as cf
    import oracle
    if threads <= 1:
        times, t_start, seed = [], time.time(), 0
        while len(times) < max_tokens and (time.time() - t_start) < budget_s:
            inp = _oracle_token_inputs(seed)
            t0 = time.perf_counter()
            oracle.moe_layer(*inp)
            times.append(time.perf_counter() - t0)
            seed += 1
        return 1e6 * sum(times) / len(times), len(times), sum(times)
    n = 2 * threads
    with cf.ThreadPoolExecutor(threads) as ex:
        inputs = list(ex.map(_oracle_token_inputs, range(n)))
        t0 = time.perf_counter()
        list(ex.map(lambda a: oracle.moe_layer(*a), inputs))
        wall = time.perf_counter() - t0
    return 1e6 * wall / n, n, wall


def cpu_baseline_block(budget_s: float):
    """The oracle timed on the host: all cores (the reported value) and one thread."""
    cores = os.cpu_count() or 1
    us1, n1, t1 = cpu_oracle_sample(budget_s, 1)
    usn, nn, tn = cpu_oracle_sample(budget_s, cores)
    return {"value": usn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d single-token layer calls (one per layer instance, seeds 0..%d) on %d host threads, "
                      "%.1f s wall" % (nn, min(nn, N_SEEDS) - 1, cores, tn),
            "single_thread": {"value": us1, "unit": UNIT, "cores": 1,
                              "sample": "%d single-token layer calls one after another, %.1f s" % (n1, t1)}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    cpu = cpu_baseline_block(max(5.0, args.cpu_seconds))
    us = cpu["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": int(cpu["sample"].split()[0]), "warmup": 0, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": cpu["sample"]},
        "cpu_baseline": cpu,
        "tokens_per_s": 1e6 / us,
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ GPU arm

def build_layers(nv, wl, device, n):
    shape = wl.QWEN36_35B_A3B
    layers, xs = [], []
    for seed in range(n):
        L = wl.LayerInputs(shape, seed=seed)
        layer = nv.MoELayer.allocate(shape.H, shape.E, shape.k, shape.I, shape.Is, nv.SCALE_E4M3, device)
        layer.router_w.copy_(L.router_w(device))
        for e in range(shape.E):
            layer.pack_expert(e, *L.expert_f32(e, device=device))
        layer.pack_shared(*L.shared_f32(device=device), L.shared_sigmoid_w(device))
        layers.append(layer)
        xs.append(wl.activations(seed, 1, shape.H, device=device))
    torch.cuda.synchronize()
    return layers, xs


def step_bytes(layer, ids_row, T=1):
    """Algorithmic bytes of one layer call: distinct active experts' packed weights,
    scales and tensor scales, the shared expert, the router, x and y, routing outputs."""
    H, I, Is = layer.H, layer.I, layer.Is
    per_expert = layer.weight_bytes_per_expert()
    distinct = len(set(int(v) for v in ids_row))
    shared = 2 * Is * H // 2 + 2 * Is * H // 16 + H * Is // 2 + H * Is // 16 + 12 + 2 * H
    router = layer.E * H * 2
    acts = 2 * H * T * 2
    return distinct * per_expert + shared + router + acts


PREFILL_GOLDEN = os.path.join(ROOT, "tests", "golden", "prefill_zipf.json")


def prefill_flops(shape, T, has_shared=True):
    """Algorithmic FLOPs of one layer call: router GEMM, routed and shared SwiGLU experts."""
    f = 2 * T * shape.E * shape.H + 2 * T * shape.k * 3 * shape.I * shape.H
    if has_shared:
        f += 2 * T * 3 * shape.Is * shape.H + 2 * T * shape.H
    return f


def measure_prefill(nv, wl, device, steps, warmup):
    """One 4096-token call of the Qwen3.6-35B-A3B-shaped layer per step, router rows
    scaled by rank^-kappa (kappa from the committed calibration) so that per-expert
    token counts range from about 20 to 1000. Returns the measured figures."""
    import dataclasses
    gold = json.load(open(PREFILL_GOLDEN))
    shape = dataclasses.replace(wl.QWEN36_35B_A3B, router_kappa=gold["kappa"])
    T, seed = gold["T"], gold["seed"]
    L = wl.LayerInputs(shape, seed=seed)
    layer = nv.MoELayer.allocate(shape.H, shape.E, shape.k, shape.I, shape.Is, nv.SCALE_E4M3, device)
    layer.router_w.copy_(L.router_w(device))
    for e in range(shape.E):
        layer.pack_expert(e, *L.expert_f32(e, device=device))
    layer.pack_shared(*L.shared_f32(device=device), L.shared_sigmoid_w(device))
    x = wl.activations(seed, T, shape.H, device=device)
    d = layer.desc()
    ws = nv.Workspace(nv.moe_layer_workspace_size(layer, T), device=device)
    y = torch.empty(T, shape.H, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        nv.moe_layer_forward(layer, x, ws=ws, y=y, desc=d)
    torch.cuda.synchronize()
    K = max(1, steps)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index or 0) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(K):
            nv.moe_layer_forward(layer, x, ws=ws, y=y, desc=d)
        ev1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.2)
    ms = ev0.elapsed_time(ev1) / K
    # end to end: pinned host x in, y out, every step
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(y, device="cpu").pin_memory()
    xd = torch.empty_like(x)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    Ke = min(K, 20)
    e0.record(stream)
    for _ in range(Ke):
        xd.copy_(xh, non_blocking=True)
        nv.moe_layer_forward(layer, xd, ws=ws, y=y, desc=d)
        yh.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    flops = prefill_flops(shape, T)
    tflops = flops / (ms * 1e-3) / 1e12
    mp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak, kind = (json.load(open(mp)).get("bf16_tflops_sustained"), "measured (sustained)") if os.path.exists(mp) \
        else (1700.0, "fallback (sustained)")
    res = {"us_per_call": 1e3 * ms, "tokens_per_s": T / (ms * 1e-3), "tflops": tflops, "peak_tflops": peak,
           "peak_kind": kind, "frac_of_bf16_peak": tflops / peak if peak else None, "flops_per_call": flops,
           "e2e_us_per_call": 1e3 * e2e_ms, "calls": K, "tokens": T, "kappa": gold["kappa"],
           "entries_per_expert": [gold["min_count"], gold["max_count"]], "clocks": clk.summary(),
           "launches_per_call": nv.launches_per_layer_call(T, shape.H)}
    del layer, ws, x, y
    torch.cuda.empty_cache()
    return res


def run_prefill(args, nv, wl, device):
    r = measure_prefill(nv, wl, device, args.steps, args.warmup)
    T = r["tokens"]
    line = {
        "metric": "NVFP4 MoE-layer prefill: us per 4096-token layer call", "value": r["us_per_call"],
        "unit": "us/call", "n_gpus": 1, "steps": r["calls"], "warmup": max(3, args.warmup),
        "ms_per_step": r["us_per_call"] * 1e-3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-act/nvfp4-weight, bf16 MMA, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16, router rows scaled by "
                "rank^-%g)" % r["kappa"],
        "config": {"workload": "qwen3.6-35b-a3b-shaped MoE layer prefill, T=%d tokens, H=2048 E=256 top-8 I=512 "
                               "Is=512, skewed router (per-expert entries %d..%d), seed 2"
                               % (T, r["entries_per_expert"][0], r["entries_per_expert"][1]),
                   "tokens_per_step": T, "l2": "inputs larger than L2 (453 MB of NVFP4 weights per call)"},
        "tokens_per_s": r["tokens_per_s"],
        "roofline": {"bound": "tensor", "achieved": r["tflops"], "peak": r["peak_tflops"], "unit": "TFLOP/s",
                     "frac": r["frac_of_bf16_peak"], "peak_kind": r["peak_kind"], "traffic": None,
                     "flops_per_launch": r["flops_per_call"],
                     "kernel": "whole step (router GEMM, top-k, expert lists, grouped tcgen05 gate/up and down "
                               "GEMMs, combine): algorithmic FLOPs / step time"},
        "e2e": {"value": r["e2e_us_per_call"], "unit": "us/call", "h2d_bytes_per_step": 2 * T * 2048,
                "d2h_bytes_per_step": 2 * T * 2048},
        "gpu_launches": r["launches_per_call"] * r["calls"],
        "clocks": r["clocks"],
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def graph_of(calls, cap_stream):
    """Capture the given zero-argument launches once as one CUDA graph (after one eager
    pass, which also warms the library's per-device state)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap_stream):
        for c in calls:
            c()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap_stream):
            for c in calls:
                c()
    torch.cuda.synchronize()
    return g


def time_graph(g, reps, stream, device=None, clocks=False):
    """Device time (ms) of `reps` back-to-back replays, CUDA events on the launching stream."""
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(device.index or 0) if clocks else None
    if clk:
        clk.__enter__()
        time.sleep(0.3)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(reps):
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if clk:
        time.sleep(0.2)
        clk.__exit__()
    return ev0.elapsed_time(ev1), (clk.summary() if clk else None)


def measure_batched(nv, wl, device, layers, descs, Tb, rotate, stream, reps=None):
    """Decode calls of Tb tokens. rotate=True: one call per step over the layer instances
    (graph passes), the per-call figure; rotate=False: one decode step through all the
    stacked layers (each with its own seeded input), the per-step figure."""
    n_inst = len(layers)
    H = layers[0].H
    xb = [wl.activations(100 + i, Tb, H, device=device) for i in range(n_inst)]
    yb = [torch.empty(Tb, H, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
    ws = nv.Workspace(nv.moe_layer_workspace_size(layers[0], Tb), device=device)
    ids = []
    for i in range(n_inst):
        _, ids_i, _ = nv.moe_layer_forward(layers[i], xb[i], ws=ws, want_route=True, desc=descs[i])
        ids.append(ids_i.cpu().numpy().ravel())
    bytes_call = sum(step_bytes(layers[i], ids[i], T=Tb) for i in range(n_inst)) / n_inst
    cap = torch.cuda.Stream(device=device)
    calls = [(lambda i=i: nv.moe_layer_forward(layers[i], xb[i], ws=ws, y=yb[i], desc=descs[i]))
             for i in range(n_inst)]
    g = graph_of(calls, cap)
    for _ in range(3):
        g.replay()
    reps = reps or max(1, 256 // n_inst)
    ms, _ = time_graph(g, reps, stream)
    us_call = 1e3 * ms / (reps * n_inst)
    peak, _ = measured_peaks()
    gbs = bytes_call / (us_call * 1e-6) / 1e9
    out = {"tokens": Tb, "us_per_call": us_call, "us_per_token": us_call / Tb, "tokens_per_s": 1e6 * Tb / us_call,
           "bytes_per_call": bytes_call, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak if peak else None,
           "launches_per_call": nv.launches_per_layer_call(Tb, H)}
    if not rotate:
        out = {"tokens": Tb, "layers": n_inst, "ms_per_decode_step": us_call * n_inst / 1e3,
               "us_per_layer_call": us_call, "tokens_per_s": 1e6 * Tb / (us_call * n_inst),
               "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak if peak else None,
               "bytes_per_layer_call": bytes_call}
    del ws, xb, yb, g
    return out


def run_batched(args, nv, wl, device):
    """One decode step of --tokens tokens through 40 stacked layers with independent
    weights (18.1 GB resident): the 40 layer calls in sequence on one stream, graph
    replayed; bytes per call are the distinct active experts' weights plus the shared
    expert, the router and the activations."""
    Tb = args.tokens
    n_inst = CHAIN_LAYERS if args.seeds == N_SEEDS else max(1, args.seeds)
    layers, _ = build_layers(nv, wl, device, n_inst)
    descs = [l.desc() for l in layers]
    stream = torch.cuda.current_stream()
    reps = max(1, -(-max(1, args.steps) // n_inst))
    r = measure_batched(nv, wl, device, layers, descs, Tb, False, stream, reps=reps)
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "NVFP4 MoE-layer decode, %d tokens per call: us/token and achieved HBM GB/s" % Tb,
        "value": r["us_per_layer_call"] / Tb, "unit": "us/token", "n_gpus": 1, "steps": reps * n_inst,
        "warmup": 3, "ms_per_step": r["us_per_layer_call"] * 1e-3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-act/nvfp4-weight, f16 MMA, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": "qwen3.6-35b-a3b-shaped MoE layer decode, T=%d tokens per call, H=2048 E=256 "
                               "top-8 I=512 shared Is=512, NVFP4 E4M3 per-16 scales, %d stacked layers with "
                               "independent weights (%.1f GB resident)" % (Tb, n_inst, n_inst * 0.4531),
                   "tokens_per_step": Tb,
                   "l2": "inputs larger than L2: every layer's weights are read once per decode step"},
        "decode_step": r,
        "roofline": {"bound": "hbm", "achieved": r["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": r["frac_of_hbm_peak"], "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": r["bytes_per_layer_call"],
                     "kernel": "whole call (router, route, gate/up, down, combine): algorithmic bytes / call time"},
        "gpu_launches": nv.launches_per_layer_call(Tb, layers[0].H) * reps * n_inst,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def measure_gemv(nv, wl, device, reps=10):
    """Dense NVFP4 W4A16 GEMV like a GatedDeltaNet in_proj_qkv: 1 token, K=2048 -> N=8192,
    FP16 block scales and E4M3 block scales. 16 packed weight instances (168 MB) rotate
    so that every call reads cold weights; one CUDA graph replays a pass over them. Bytes
    per call: codes, scales, tensor scale, x, y."""
    N, K, T = 8192, 2048, 1
    n_inst = 16
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    res = {}
    for kind, name in ((nv.SCALE_FP16, "fp16"), (nv.SCALE_E4M3, "e4m3")):
        Ws = [nv.nvfp4_pack(wl.dense_weight_f32(1 + i, N, K, device=device), kind) for i in range(n_inst)]
        xs = [wl.activations(1 + i, T, K, device=device) for i in range(n_inst)]
        ys = [torch.empty(T, N, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
        sb = 2 if kind == nv.SCALE_FP16 else 1
        bytes_call = N * K // 2 + N * (K // 16) * sb + 4 + 2 * K * T + 2 * N * T
        cap = torch.cuda.Stream(device=device)
        g = graph_of([(lambda i=i: nv.nvfp4_gemv_w4a16(Ws[i], xs[i], y=ys[i])) for i in range(n_inst)], cap)
        for _ in range(3):
            g.replay()
        ms, clk = time_graph(g, reps, stream, device, clocks=(kind == nv.SCALE_FP16))
        us = 1e3 * ms / (reps * n_inst)
        gbs = bytes_call / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": us, "bytes_per_call": bytes_call, "achieved_gbs": gbs,
                     "frac_of_hbm_peak": gbs / peak if peak else None, "calls": reps * n_inst}
        if clk:
            res["clocks"] = clk
        del Ws, xs, ys, g
    res.update(measure_lm_head(nv, wl, device, reps))
    res["peak_kind"] = peak_kind
    return res


def measure_lm_head(nv, wl, device, reps=10):
    """The lm_head of the same model as one dense GEMV: vocab 248320 x hidden 2048 (318 / 287
    MB per call with FP16 / E4M3 block scales), two instances rotating, each larger than L2."""
    N, K, T, n_inst = 248320, 2048, 1, 2
    stream = torch.cuda.current_stream()
    res = {}
    for kind, name in ((nv.SCALE_FP16, "lm_head_fp16"), (nv.SCALE_E4M3, "lm_head_e4m3")):
        Ws = []
        for i in range(n_inst):
            w = wl.dense_weight_f32(40 + i, N, K, device=device)
            Ws.append(nv.nvfp4_pack(w, kind))
            del w
        xs = [wl.activations(40 + i, T, K, device=device) for i in range(n_inst)]
        ys = [torch.empty(T, N, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
        sb = 2 if kind == nv.SCALE_FP16 else 1
        bytes_call = N * K // 2 + N * (K // 16) * sb + 4 + 2 * K * T + 2 * N * T
        cap = torch.cuda.Stream(device=device)
        g = graph_of([(lambda i=i: nv.nvfp4_gemv_w4a16(Ws[i], xs[i], y=ys[i])) for i in range(n_inst)], cap)
        for _ in range(3):
            g.replay()
        r2 = max(4, reps)
        ms, _ = time_graph(g, r2, stream, device)
        us = 1e3 * ms / (r2 * n_inst)
        gbs = bytes_call / (us * 1e-6) / 1e9
        peak, _ = measured_peaks()
        res[name] = {"us_per_call": us, "bytes_per_call": bytes_call, "achieved_gbs": gbs,
                     "frac_of_hbm_peak": gbs / peak if peak else None, "calls": r2 * n_inst,
                     "shape": "T=1, K=2048 -> N=248320"}
        del Ws, xs, ys, g
        torch.cuda.empty_cache()
    return res


def run_gemv(args, nv, wl, device):
    reps = max(1, -(-max(1, args.steps) // 16))
    res = measure_gemv(nv, wl, device, reps)
    f = res["fp16"]
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "NVFP4 dense W4A16 GEMV, 1 token, K=2048 -> N=8192: us per call and achieved HBM GB/s",
        "value": f["us_per_call"], "unit": "us/call", "n_gpus": 1, "steps": f["calls"], "warmup": 3,
        "ms_per_step": f["us_per_call"] * 1e-3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-act/nvfp4-weight, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": "dense NVFP4 W4A16 GEMV (GatedDeltaNet in_proj_qkv shape), T=1, K=2048, N=8192, "
                               "FP16 per-16 scales; 16 rotating weight instances (168 MB)", "tokens_per_step": 1,
                   "l2": "inputs larger than L2: 16 rotating instances"},
        "roofline": {"bound": "hbm", "achieved": f["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": f["frac_of_hbm_peak"], "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": f["bytes_per_call"], "kernel": "gemv_kernel (one launch per call)"},
        "e4m3": res["e4m3"],
        "gpu_launches": f["calls"],
        "clocks": res.get("clocks"),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_lm_head(args, nv, wl, device):
    reps = max(4, -(-max(1, args.steps) // 2))
    res = measure_lm_head(nv, wl, device, reps)
    f = res["lm_head_fp16"]
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "NVFP4 lm_head GEMV, 1 token, K=2048 -> N=248320: us per call and achieved HBM GB/s",
        "value": f["us_per_call"], "unit": "us/call", "n_gpus": 1, "steps": f["calls"], "warmup": 3,
        "ms_per_step": f["us_per_call"] * 1e-3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-act/nvfp4-weight, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": "NVFP4 lm_head GEMV (vocabulary 248320 x hidden 2048), T=1, FP16 per-16 scales; "
                               "2 rotating weight instances (318 MB each)", "tokens_per_step": 1,
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": f["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": f["frac_of_hbm_peak"], "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": f["bytes_per_call"], "kernel": "gemv_kernel (one launch per call)"},
        "e4m3": res["lm_head_e4m3"],
        "gpu_launches": f["calls"],
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    global torch
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_w4a16_moe_gb300 as nv
    import workload as wl

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.workload == "prefill":
        if world > 1 and rank != 0:
            return 0
        return run_prefill(args, nv, wl, device)
    if args.workload == "batched":
        if world > 1 and rank != 0:
            return 0
        return run_batched(args, nv, wl, device)
    if args.workload == "gemv":
        if world > 1 and rank != 0:
            return 0
        return run_gemv(args, nv, wl, device)
    if args.workload == "lm_head":
        if world > 1 and rank != 0:
            return 0
        return run_lm_head(args, nv, wl, device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    extras = rank == 0 and not args.no_extras

    # layer instances: seeds 0..31 for the single-token steps; 40 stacked layers (seeds
    # 0..39) for the decode-step figures of the default run
    n_inst = max(1, min(args.seeds, N_SEEDS))
    layers, xs = build_layers(nv, wl, device, CHAIN_LAYERS if extras and n_inst == N_SEEDS else n_inst)
    T = 1
    ws = nv.Workspace(nv.moe_layer_workspace_size(layers[0], T), device=device)
    descs = [l.desc() for l in layers]
    ys = [torch.empty(T, layers[0].H, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
    stream = torch.cuda.current_stream()

    # routing of every instance, for the byte count of each step
    ids_all = []
    for i in range(n_inst):
        _, ids, _ = nv.moe_layer_forward(layers[i], xs[i], ws=ws, want_route=True, desc=descs[i])
        ids_all.append(ids.cpu().numpy()[0])
    bytes_per_step = [step_bytes(layers[i], ids_all[i]) for i in range(n_inst)]

    def step(i):
        j = i % n_inst
        nv.moe_layer_forward(layers[j], xs[j], ws=ws, y=ys[j], desc=descs[j])

    W = max(3, args.warmup)
    for i in range(W):
        step(i)
    torch.cuda.synchronize()

    # Exactly K steps, captured once as one CUDA graph: the timed region is one replay,
    # so the host's per-call cost (Python, ctypes) does not leave the GPU idle between
    # steps; consecutive kernels inside the graph keep their programmatic (PDL)
    # dependency. Steps rotate over the instances (14.5 GB >> L2).
    K = max(1, args.steps)
    cap = torch.cuda.Stream(device=device)
    cap.wait_stream(stream)
    graph = graph_of([(lambda i=i: step(i)) for i in range(K)], cap)
    graph.replay()       # untimed: warms the graph itself
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_local, clocks = time_graph(graph, 1, stream, device, clocks=True)
    ms, us_per_token = replicas_timing(ms_local, K, world, device)
    avg_bytes = sum(bytes_per_step[i % n_inst] for i in range(K)) / K
    achieved_gbs = avg_bytes / (us_per_token * world * 1e-6) / 1e9
    del graph

    # the same steps launched one by one from Python (host-bound; reported beside)
    Ks = min(K, 1000)
    es0 = torch.cuda.Event(enable_timing=True)
    es1 = torch.cuda.Event(enable_timing=True)
    es0.record(stream)
    for i in range(Ks):
        step(i)
    es1.record(stream)
    torch.cuda.synchronize()
    stream_us = 1e3 * es0.elapsed_time(es1) / Ks

    # end to end through the public API with host buffers: pinned x in, y out, every step
    xh = [x.cpu().pin_memory() for x in xs[:n_inst]]
    yh = torch.empty(T, layers[0].H, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(T, layers[0].H, dtype=torch.bfloat16, device=device)
    for i in range(5):
        xd.copy_(xh[i % n_inst], non_blocking=True)
        nv.moe_layer_forward(layers[i % n_inst], xd, ws=ws, y=ys[0], desc=descs[i % n_inst])
        yh.copy_(ys[0], non_blocking=True)
    torch.cuda.synchronize()
    Ke = min(K, 1000)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(Ke):
        j = i % n_inst
        xd.copy_(xh[j], non_blocking=True)
        nv.moe_layer_forward(layers[j], xd, ws=ws, y=ys[0], desc=descs[j])
        yh.copy_(ys[0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = 1e3 * e0.elapsed_time(e1) / Ke

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    line = {
        "metric": METRIC, "value": us_per_token, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms / K, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-act/nvfp4-weight, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1,
                   "l2": "inputs larger than L2: %d rotating layer instances (%.1f GB)" % (
                       n_inst, sum(l.gu_packed.numel() + l.dn_packed.numel() for l in layers[:n_inst]) * 1.125 / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": 1e6 / us_per_token,
        "achieved_gbs": achieved_gbs,
        "pct_of_8tbs": 100.0 * achieved_gbs / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak if peak else None, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(), "bytes_per_launch": avg_bytes,
                     "kernel": "moe_decode_t1_kernel (the whole step is this one launch)"},
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": 2 * layers[0].H * T,
                "d2h_bytes_per_step": 2 * layers[0].H * T},
        "gpu_launches": nv.launches_per_layer_call(T, layers[0].H) * K,
        "timing": {"mode": "one CUDA graph of exactly %d steps, replayed once" % K,
                   "stream_launch_us_per_token": stream_us},
        "clocks": clocks,
    }
    if extras:
        # the other measured configurations, each with its own CUDA-event timing
        line["batched_decode"] = [measure_batched(nv, wl, device, layers[:n_inst], descs[:n_inst], Tb, True, stream)
                                  for Tb in (8, 64)]
        if len(layers) == CHAIN_LAYERS:
            line["decode_step_40_layers"] = [measure_batched(nv, wl, device, layers, descs, Tb, False, stream)
                                             for Tb in (1, 8, 64)]
        del layers, xs, ys, ws, descs
        torch.cuda.empty_cache()
        line["gemv"] = measure_gemv(nv, wl, device)
        line["prefill"] = measure_prefill(nv, wl, device, steps=20, warmup=3)
    line["cpu_baseline"] = None
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_block(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
