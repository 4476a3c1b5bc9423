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
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seeds", type=int, default=N_SEEDS, help="layer instances to rotate over")
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "batched", "gemv"],
                    help="decode: the single-token layer (default, the headline); prefill: one "
                         "4096-token layer call with the skewed router; batched: one --tokens-token "
                         "decode call per step; gemv: the dense W4A16 GEMV, 1 token, K=2048 -> N=8192")
    ap.add_argument("--tokens", type=int, default=64, help="tokens per call of --workload batched (1..64)")
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
    src = open(os.path.join(ROOT, d["source"]), "rb").read()
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

def cpu_oracle_sample(budget_s: float, max_tokens: int = 64):
    """Time the CPU oracle on single tokens of the same workload (weights packed
    beforehand, as the GPU's are). Returns (us_per_token, tokens, cores)."""
    import oracle
    import workload as wl
    import numpy as np
    shape = wl.QWEN36_35B_A3B
    times = []
    t_start = time.time()
    seed = 0
    while len(times) < max_tokens and (time.time() - t_start) < budget_s:
        L = wl.LayerInputs(shape, seed=seed % N_SEEDS)
        x = wl.activations(seed % N_SEEDS, 1, shape.H)
        wg = L.router_w("cpu")
        ids, _, _ = oracle.route(oracle.router_logits(x, wg), shape.k)
        experts = {}
        for e in ids.ravel().tolist():
            g, u, d = L.expert_f32(e)
            experts[e] = (oracle.pack(g), oracle.pack(u), oracle.pack(d))
        sg, su, sd = L.shared_f32()
        shared = (oracle.pack(sg), oracle.pack(su), oracle.pack(sd))
        sgv = L.shared_sigmoid_w("cpu")
        t0 = time.perf_counter()
        oracle.moe_layer(x, wg, sgv, experts, shared, shape.k)
        times.append(time.perf_counter() - t0)
        seed += 1
    us = 1e6 * sum(times) / len(times)
    return us, len(times), sum(times)


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    us, n, tot = cpu_oracle_sample(max(5.0, args.cpu_seconds))
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": n, "warmup": 0, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "%d single-token layer calls" % n},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d tokens of the T=1 decode workload (seeds 0..%d), %.1f s of CPU" %
                                   (n, min(n, N_SEEDS) - 1, tot)},
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


def run_prefill(args, nv, wl, device):
    """One 4096-token call of the Qwen3.6-35B-A3B-shaped layer per step, router rows
    scaled by rank^-kappa (kappa from the committed calibration) so that per-expert
    token counts range from about 20 to 1000."""
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
    for _ in range(max(3, args.warmup)):
        nv.moe_layer_forward(layer, x, ws=ws, y=y, desc=d)
    torch.cuda.synchronize()
    K = max(1, args.steps)
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
    line = {
        "metric": "NVFP4 MoE-layer prefill: us per 4096-token layer call", "value": 1e3 * ms, "unit": "us/call",
        "n_gpus": 1, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-act/nvfp4-weight, bf16 MMA, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16, router rows scaled by rank^-%g)"
                % gold["kappa"],
        "config": {"workload": "qwen3.6-35b-a3b-shaped MoE layer prefill, T=%d tokens, H=2048 E=256 top-8 I=512 "
                               "Is=512, skewed router (per-expert entries %d..%d), seed %d"
                               % (T, gold["min_count"], gold["max_count"], seed),
                   "tokens_per_step": T,
                   "l2": "inputs larger than L2 (453 MB of NVFP4 weights per call)"},
        "tokens_per_s": T / (ms * 1e-3),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak if peak else None, "peak_kind": kind, "traffic": None,
                     "flops_per_launch": flops,
                     "kernel": "whole step (router GEMM, top-k, expert lists, grouped tcgen05 gate/up and down "
                               "GEMMs, combine): algorithmic FLOPs / step time"},
        "e2e": {"value": 1e3 * e2e_ms, "unit": "us/call", "h2d_bytes_per_step": 2 * T * shape.H,
                "d2h_bytes_per_step": 2 * T * shape.H},
        "gpu_launches": nv.launches_per_layer_call(T, shape.H) * K,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_batched(args, nv, wl, device):
    """One decode call of --tokens tokens per step through --seeds rotating layer
    instances (the multi-token kernels), CUDA-graph replayed in passes over the
    instances; bytes per call are the distinct active experts' weights plus the
    shared expert, the router and the activations."""
    Tb = args.tokens
    # one decode step through 40 stacked layers with independent weights (18.1 GB
    # resident): 40 layer calls in sequence on one stream, one graph replay
    n_inst = CHAIN_LAYERS if args.seeds == N_SEEDS else max(1, args.seeds)
    layers, _ = build_layers(nv, wl, device, n_inst)
    descs = [l.desc() for l in layers]
    xb = [wl.activations(100 + i, Tb, layers[0].H, device=device) for i in range(n_inst)]
    yb = [torch.empty(Tb, layers[0].H, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
    ws = nv.Workspace(nv.moe_layer_workspace_size(layers[0], Tb), device=device)
    ids = []
    for i in range(n_inst):
        _, ids_i, _ = nv.moe_layer_forward(layers[i], xb[i], ws=ws, want_route=True, desc=descs[i])
        ids.append(ids_i.cpu().numpy().ravel())
    bytes_call = sum(step_bytes(layers[i], ids[i], T=Tb) for i in range(n_inst)) / n_inst
    stream = torch.cuda.current_stream()
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        for i in range(n_inst):
            nv.moe_layer_forward(layers[i], xb[i], ws=ws, y=yb[i], desc=descs[i])
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            for i in range(n_inst):
                nv.moe_layer_forward(layers[i], xb[i], ws=ws, y=yb[i], desc=descs[i])
    torch.cuda.synchronize()
    W = max(3, args.warmup)
    for _ in range(-(-W // n_inst)):
        g.replay()
    torch.cuda.synchronize()
    passes = max(1, -(-max(1, args.steps) // n_inst))
    K = passes * n_inst
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index or 0) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(passes):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.2)
    us = 1e3 * ev0.elapsed_time(ev1) / K
    gbs = bytes_call / (us * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "NVFP4 MoE-layer decode, %d tokens per call: us/token and achieved HBM GB/s" % Tb,
        "value": us / Tb, "unit": "us/token", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": us * 1e-3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-act/nvfp4-weight, bf16 MMA, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": "qwen3.6-35b-a3b-shaped MoE layer decode, T=%d tokens per call, H=2048 E=256 "
                               "top-8 I=512 shared Is=512, NVFP4 E4M3 per-16 scales, %d stacked layers with "
                               "independent weights (%.1f GB resident)"
                               % (Tb, n_inst, n_inst * 0.4531), "tokens_per_step": Tb,
                   "l2": "inputs larger than L2: every layer's weights are read once per decode step"},
        "us_per_call": us, "achieved_gbs": gbs,
        "decode_step": {"layers": n_inst, "us": us * n_inst,
                        "note": "one graph replay = the layer calls of one decode step through the stacked "
                                "layers, in sequence on one stream; each layer gets its own seeded input "
                                "(the pages' layer has no norm, so a raw chain underflows within a few layers "
                                "and would route every token to the same experts)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak if peak else None, "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": bytes_call,
                     "kernel": "whole call (router, route, gate/up, down, combine): algorithmic bytes / call time"},
        "gpu_launches": nv.launches_per_layer_call(Tb, layers[0].H) * K,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gemv(args, nv, wl, device):
    """Dense NVFP4 W4A16 GEMV like a GatedDeltaNet in_proj_qkv: 1 token, K=2048 -> N=8192,
    FP16 block scales (the value) and E4M3 block scales (reported beside). 16 packed
    weight instances (168 MB) rotate so that every call reads cold weights; one CUDA
    graph replays a pass over them. Bytes per call: codes, scales, tensor scale, x, y."""
    N, K, T = 8192, 2048, 1
    n_inst = 16
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    res = {}
    clk_summary = None
    for kind, name in ((nv.SCALE_FP16, "fp16"), (nv.SCALE_E4M3, "e4m3")):
        Ws = []
        for i in range(n_inst):
            w = wl.dense_weight_f32(1 + i, N, K, device=device)
            Ws.append(nv.nvfp4_pack(w, kind))
            del w
        xs = [wl.activations(1 + i, T, K, device=device) for i in range(n_inst)]
        ys = [torch.empty(T, N, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
        sb = 2 if kind == nv.SCALE_FP16 else 1
        bytes_call = N * K // 2 + N * (K // 16) * sb + 4 + 2 * K * T + 2 * N * T
        cap = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            for i in range(n_inst):
                nv.nvfp4_gemv_w4a16(Ws[i], xs[i], y=ys[i])
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cap):
                for i in range(n_inst):
                    nv.nvfp4_gemv_w4a16(Ws[i], xs[i], y=ys[i])
        torch.cuda.synchronize()
        W = max(3, args.warmup)
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        passes = max(1, -(-max(1, args.steps) // n_inst))
        K_calls = passes * n_inst
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(device.index or 0) as clk:
            time.sleep(0.3)
            torch.cuda.synchronize()
            ev0.record(stream)
            for _ in range(passes):
                g.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            time.sleep(0.2)
        us = 1e3 * ev0.elapsed_time(ev1) / K_calls
        gbs = bytes_call / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": us, "bytes_per_call": bytes_call, "achieved_gbs": gbs,
                     "frac_of_hbm_peak": gbs / peak if peak else None, "calls": K_calls}
        if kind == nv.SCALE_FP16:
            clk_summary = clk.summary()
        del Ws, xs, ys, g
    f = res["fp16"]
    line = {
        "metric": "NVFP4 dense W4A16 GEMV, 1 token, K=2048 -> N=8192: us per call and achieved HBM GB/s",
        "value": f["us_per_call"], "unit": "us/call", "n_gpus": 1, "steps": f["calls"], "warmup": max(3, args.warmup),
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
        "clocks": clk_summary,
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
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    n_inst = max(1, min(args.seeds, N_SEEDS))
    layers, xs = build_layers(nv, wl, device, n_inst)
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

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()

    # One pass over every layer instance, captured once as a CUDA graph: the
    # timed region replays it, so the host's per-call cost (Python, ctypes) does
    # not leave the GPU idle between steps; consecutive kernels inside the graph
    # keep their programmatic (PDL) dependency.
    cap = torch.cuda.Stream(device=device)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        for i in range(n_inst):
            step(i)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(n_inst):
                step(i)
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup // n_inst + 1)):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    reps = max(1, (args.steps + n_inst - 1) // n_inst)
    K = reps * n_inst
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.2)
    ms, us_per_token = replicas_timing(ev0.elapsed_time(ev1), K, world, device)
    avg_bytes = sum(bytes_per_step) / n_inst
    achieved_gbs = avg_bytes / (1e3 * ms / K * 1e-6) / 1e9

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
    xh = [x.cpu().pin_memory() for x in xs]
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

    # batched decode: 8 and 64 tokens per call through the same rotating layers (the
    # multi-token kernels), graph-replayed like the single-token steps
    batched = []
    for Tb in (8, 64):
        xb = [wl.activations(100 + i, Tb, layers[0].H, device=device) for i in range(n_inst)]
        wsb = nv.Workspace(nv.moe_layer_workspace_size(layers[0], Tb), device=device)
        yb = [torch.empty(Tb, layers[0].H, dtype=torch.bfloat16, device=device) for _ in range(n_inst)]
        idsb = []
        for i in range(n_inst):
            _, ids_i, _ = nv.moe_layer_forward(layers[i], xb[i], ws=wsb, want_route=True, desc=descs[i])
            idsb.append(ids_i.cpu().numpy().ravel())
        bytes_b = sum(step_bytes(layers[i], idsb[i], T=Tb) for i in range(n_inst)) / n_inst
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            for i in range(n_inst):
                nv.moe_layer_forward(layers[i], xb[i], ws=wsb, y=yb[i], desc=descs[i])
            torch.cuda.synchronize()
            with torch.cuda.graph(gb, stream=cap):
                for i in range(n_inst):
                    nv.moe_layer_forward(layers[i], xb[i], ws=wsb, y=yb[i], desc=descs[i])
        torch.cuda.synchronize()
        for _ in range(3):
            gb.replay()
        torch.cuda.synchronize()
        rb = max(1, 200 // n_inst)
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(rb):
            gb.replay()
        b1.record(stream)
        torch.cuda.synchronize()
        us_call = 1e3 * b0.elapsed_time(b1) / (rb * n_inst)
        gbs = bytes_b / (us_call * 1e-6) / 1e9
        batched.append({"tokens": Tb, "us_per_call": us_call, "us_per_token": us_call / Tb,
                        "bytes_per_call": bytes_b, "achieved_gbs": gbs})
        del wsb

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    for b in batched:
        b["frac_of_hbm_peak"] = b["achieved_gbs"] / peak if peak else None
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        us, n, tot = cpu_oracle_sample(args.cpu_seconds)
        cpu = {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "%d single-token layer calls of the same workload (seeds 0..%d), %.1f s" %
                         (n, min(n, N_SEEDS) - 1, tot)}
    launches_per_step = nv.launches_per_layer_call(T, layers[0].H)
    line = {
        "metric": METRIC, "value": us_per_token, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms / K, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-act/nvfp4-weight, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights packed to NVFP4, x ~ N(0,1) bf16)",
        "config": {"workload": WORKLOAD, "tokens_per_step": 1,
                   "l2": "inputs larger than L2: %d rotating layer instances (%.1f GB)" % (
                       n_inst, sum(l.gu_packed.numel() + l.dn_packed.numel() for l in layers) * 1.125 / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "achieved_gbs": achieved_gbs,
        "pct_of_8tbs": 100.0 * achieved_gbs / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak if peak else None, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(), "bytes_per_launch": avg_bytes,
                     "kernel": "moe_decode_t1_kernel (the whole step is this one launch)"},
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": 2 * layers[0].H * T,
                "d2h_bytes_per_step": 2 * layers[0].H * T},
        "gpu_launches": launches_per_step * K,
        "timing": {"mode": "CUDA graph replay of %d-step passes" % n_inst,
                   "stream_launch_us_per_token": stream_us},
        "batched_decode": batched,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
