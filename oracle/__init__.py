"""Python view of the CPU oracle (``nvfp4_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg may use this module; the library under ``nvfp4_w4a16_moe_gb300``
never does. It shares no code with the CUDA path; the only thing both sides
import is the seeded input generator in ``workload``.

Every function converts arrays to contiguous numpy buffers, calls the C code
and returns numpy arrays. All results are fp64 unless they are codes/bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
LIB = os.path.join(HERE, "_liboracle.so")

SCALE_E4M3 = 0
SCALE_FP16 = 1
SCALE_FP32 = 2     # fp32 block scale per 16 elements, tensor scale 1
SCALE_UE8M0 = 3    # power-of-two E8M0 scale per 32 elements, tensor scale 1

# block length and numpy dtype of one block scale, per kind
SCALE_BLOCK = {SCALE_E4M3: 16, SCALE_FP16: 16, SCALE_FP32: 16, SCALE_UE8M0: 32}
SCALE_DTYPE = {SCALE_E4M3: np.uint8, SCALE_FP16: np.uint16, SCALE_FP32: np.float32, SCALE_UE8M0: np.uint8}

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        i32, f32 = ctypes.c_int, ctypes.c_float
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [i32]
        L.orc_e2m1_encode.restype = i32
        L.orc_e2m1_encode.argtypes = [f32]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [i32]
        L.orc_e4m3_encode.restype = i32
        L.orc_e4m3_encode.argtypes = [f32]
        L.orc_fp16_decode.restype = ctypes.c_double
        L.orc_fp16_decode.argtypes = [i32]
        L.orc_fp16_encode.restype = i32
        L.orc_fp16_encode.argtypes = [f32]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [i32]
        L.orc_pack.restype = i32
        L.orc_pack.argtypes = [P, i32, i32, i32, P, P, P]
        L.orc_dequant.restype = None
        L.orc_dequant.argtypes = [P, P, f32, i32, i32, i32, P]
        L.orc_gemv.restype = None
        L.orc_gemv.argtypes = [P, P, f32, i32, i32, i32, P, i32, P]
        L.orc_router_logits.restype = None
        L.orc_router_logits.argtypes = [P, i32, i32, P, i32, P]
        L.orc_route.restype = i32
        L.orc_route.argtypes = [P, i32, i32, i32, P, P, P]
        L.orc_swiglu.restype = None
        L.orc_swiglu.argtypes = [P, P, f32, P, P, f32, P, P, f32, i32, i32, i32, P, i32, P]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_rmsnorm.restype = None
        L.orc_rmsnorm.argtypes = [P, i32, i32, P, ctypes.c_double, P, P]
        L.orc_moe_layer.restype = i32
        L.orc_moe_layer.argtypes = ([i32] * 6 + [P, i32, P, P] + [P, P, P] * 3 +
                                    [P, P, f32] * 3 + [P, P, P, P, P])
        _lib = L
    return _lib


def _np(a, dtype):
    """Contiguous numpy copy/view of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.view(__import__("torch").int16).numpy().view(np.uint16)
        else:
            a = a.numpy()
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------- formats

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_decode(b: int) -> float:
    return lib().orc_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def fp16_decode(b: int) -> float:
    return lib().orc_fp16_decode(int(b))


def fp16_encode(v: float) -> int:
    return lib().orc_fp16_encode(float(v))


def e8m0_decode(b: int) -> float:
    return lib().orc_e8m0_decode(int(b))


@dataclass
class Packed:
    """One NVFP4 matrix: packed [N, K/2] u8, scales [N, K/B] (u8 E4M3, u16 FP16, f32 FP32 with B = 16;
    u8 E8M0 with B = 32), fp32 tensor scale."""
    packed: np.ndarray
    scales: np.ndarray
    tensor_scale: float
    kind: int
    N: int
    K: int


def pack(w, kind: int = SCALE_E4M3) -> Packed:
    w = _np(w, np.float32)
    N, K = w.shape
    packed = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // SCALE_BLOCK[kind]), SCALE_DTYPE[kind])
    ts = np.zeros(1, np.float32)
    rc = lib().orc_pack(_ptr(w), N, K, kind, _ptr(packed), _ptr(scales), _ptr(ts))
    if rc != 0:
        raise ValueError("oracle pack failed: code %d" % rc)
    return Packed(packed, scales, float(ts[0]), kind, N, K)


def dequant(p: Packed) -> np.ndarray:
    out = np.zeros((p.N, p.K), np.float64)
    lib().orc_dequant(_ptr(p.packed), _ptr(p.scales), p.tensor_scale, p.kind, p.N, p.K, _ptr(out))
    return out


def gemv(p: Packed, x) -> np.ndarray:
    """y[T, N] (fp64) = dequant(p) @ x[T, K] (bf16)."""
    xb = _np(x, np.uint16)
    T = xb.shape[0]
    y = np.zeros((T, p.N), np.float64)
    lib().orc_gemv(_ptr(p.packed), _ptr(p.scales), p.tensor_scale, p.kind, p.N, p.K, _ptr(xb), T,
                   _ptr(y))
    return y


def router_logits(x, router_w) -> np.ndarray:
    xb = _np(x, np.uint16)
    wb = _np(router_w, np.uint16)
    T, H = xb.shape
    E = wb.shape[0]
    out = np.zeros((T, E), np.float64)
    lib().orc_router_logits(_ptr(xb), T, H, _ptr(wb), E, _ptr(out))
    return out


def route(logits, k: int):
    """(ids [T,k] int32, w [T,k] fp64, p [T,E] fp64) from fp64 logits [T,E]."""
    lg = _np(logits, np.float64)
    T, E = lg.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    p = np.zeros((T, E), np.float64)
    rc = lib().orc_route(_ptr(lg), T, E, k, _ptr(ids), _ptr(w), _ptr(p))
    if rc != 0:
        raise ValueError("oracle route failed: code %d" % rc)
    return ids, w, p


def swiglu(g: Packed, u: Packed, d: Packed, x) -> np.ndarray:
    xb = _np(x, np.uint16)
    T, H = xb.shape
    I = g.N
    y = np.zeros((T, H), np.float64)
    lib().orc_swiglu(_ptr(g.packed), _ptr(g.scales), g.tensor_scale, _ptr(u.packed), _ptr(u.scales),
                     u.tensor_scale, _ptr(d.packed), _ptr(d.scales), d.tensor_scale, g.kind, H, I,
                     _ptr(xb), T, _ptr(y))
    return y


@dataclass
class LayerResult:
    y: np.ndarray        # [T, H] fp64
    ids: np.ndarray      # [T, k] int32
    w: np.ndarray        # [T, k] fp64
    sigmoid: np.ndarray  # [T] fp64


def moe_layer(x, router_w, sh_gate_vec, experts: dict, shared, k: int, kind: int = SCALE_E4M3,
              force_ids=None) -> LayerResult:
    """The full layer. ``experts`` maps expert id -> (gate, up, down) ``Packed``;
    only the experts that routing selects need to be present. ``shared`` is
    (gate, up, down) ``Packed`` or None for a layer without shared expert."""
    xb = _np(x, np.uint16)
    wg = _np(router_w, np.uint16)
    T, H = xb.shape
    E = wg.shape[0]
    any_e = next(iter(experts.values())) if experts else None
    I = any_e[0].N if any_e is not None else 1
    arrs = {n: (ctypes.c_void_p * E)() for n in ("gp", "gs", "up", "us", "dp", "ds")}
    ts = {n: np.zeros(E, np.float32) for n in ("g", "u", "d")}
    keep = []
    for e, (g, u, d) in experts.items():
        for name, p in (("g", g), ("u", u), ("d", d)):
            arrs[name + "p"][e] = p.packed.ctypes.data
            arrs[name + "s"][e] = p.scales.ctypes.data
            ts[name][e] = p.tensor_scale
            keep.append(p)
    if shared is not None:
        sg, su, sd = shared
        Is = sg.N
        sh = [(_ptr(m.packed), _ptr(m.scales), m.tensor_scale) for m in (sg, su, sd)]
        sgv = _np(sh_gate_vec, np.uint16)
    else:
        Is = 0
        sh = [(None, None, 0.0)] * 3
        sgv = np.zeros(H, np.uint16)
    y = np.zeros((T, H), np.float64)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    sig = np.zeros(T, np.float64)
    fi = None if force_ids is None else _np(force_ids, np.int32)
    rc = lib().orc_moe_layer(
        H, E, k, I, Is, kind, _ptr(xb), T, _ptr(wg), _ptr(sgv),
        arrs["gp"], arrs["gs"], _ptr(ts["g"]), arrs["up"], arrs["us"], _ptr(ts["u"]),
        arrs["dp"], arrs["ds"], _ptr(ts["d"]),
        sh[0][0], sh[0][1], sh[0][2], sh[1][0], sh[1][1], sh[1][2], sh[2][0], sh[2][1], sh[2][2],
        None if fi is None else _ptr(fi), _ptr(y), _ptr(ids), _ptr(w), _ptr(sig))
    if rc == 3:
        raise KeyError("routing selected an expert that was not provided")
    if rc != 0:
        raise ValueError("oracle moe_layer failed: code %d" % rc)
    return LayerResult(y, ids, w, sig)


def logit_gap(logits, k: int) -> np.ndarray:
    """Per token, the gap between the k-th and (k+1)-th largest logit (inf if E == k)."""
    lg = np.sort(_np(logits, np.float64), axis=1)[:, ::-1]
    if lg.shape[1] <= k:
        return np.full(lg.shape[0], np.inf)
    return lg[:, k - 1] - lg[:, k]


# ------------------------------------------------------- the layer for many tokens
#
# The same layer as moe_layer, evaluated expert by expert so that thousands of
# tokens take seconds instead of hours. Nothing is approximated: the dequantised
# matrices are the exact products code x block scale x tensor scale (fp64), each
# expert's SwiGLU is the definition written with numpy's fp64 matmul as the
# library step, and every token's output sums its k weighted expert rows in rank
# order, then the gated shared row, as moe_layer does (tutorials index, row 06;
# README P28/P29 notes). Pinned against moe_layer in tests/test_oracle_batched.py.

_TABLES = {}


def _decode_tables(kind: int):
    """E2M1 values of the 16 codes and the values of every scale code, from the C decoders."""
    t = _TABLES.get(kind)
    if t is None:
        e2m1 = np.array([e2m1_decode(c) for c in range(16)], np.float64)
        if kind == SCALE_E4M3:
            sc = np.array([e4m3_decode(b) for b in range(256)], np.float64)
        elif kind == SCALE_UE8M0:
            sc = np.array([e8m0_decode(b) for b in range(256)], np.float64)
        elif kind == SCALE_FP16:
            sc = np.array([fp16_decode(b) for b in range(65536)], np.float64)
        else:
            sc = None   # fp32 scales are their own values
        t = (e2m1, sc)
        _TABLES[kind] = t
    return t


def dequant_table(p: Packed) -> np.ndarray:
    """dequant(p) by table lookup: W[n, k] = E2M1(code) * scale(n, k // 16) * tensor_scale."""
    e2m1, sc = _decode_tables(p.kind)
    codes = np.empty((p.N, p.K), np.uint8)
    codes[:, 0::2] = p.packed & 15
    codes[:, 1::2] = p.packed >> 4
    vals = p.scales.astype(np.float64) if sc is None else sc[p.scales.astype(np.int64)]
    s = np.repeat(vals, SCALE_BLOCK[p.kind], axis=1)
    return e2m1[codes] * s * float(p.tensor_scale)


def _silu(z):
    return z / (1.0 + np.exp(-z))


def bf16_rows(x) -> np.ndarray:
    """bf16 [T, H] (torch tensor or uint16 bits) -> exact fp64 values."""
    xb = _np(x, np.uint16)
    return (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def swiglu_rows(g: Packed, u: Packed, d: Packed, xrows: np.ndarray) -> np.ndarray:
    """D (silu(G x) * (U x)) for every row x of xrows (fp64 [n, H]) -> fp64 [n, H]."""
    if xrows.shape[0] == 0:
        return np.zeros((0, d.N), np.float64)
    G, U, D = dequant_table(g), dequant_table(u), dequant_table(d)
    h = _silu(xrows @ G.T) * (xrows @ U.T)
    return h @ D.T


def route_tokens(x, router_w, k: int, force_ids=None):
    """(logits, ids, w, p) of moe_layer's router; with force_ids the weights are p over the
    forced set, renormalised (as moe_layer does for near-tie tokens)."""
    logits = router_logits(x, router_w)
    ids, w, p = route(logits, k)
    if force_ids is not None:
        ids = _np(force_ids, np.int32).copy()
        w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
        w = w / w.sum(axis=1, keepdims=True)
    return logits, ids, w, p


def shared_gate(x, sh_gate_vec) -> np.ndarray:
    """sigmoid(gs . x) per token (fp64)."""
    z = bf16_rows(x) @ bf16_rows(_np(sh_gate_vec, np.uint16)[None, :])[0]
    return 1.0 / (1.0 + np.exp(-z))


def combine(rows: np.ndarray, w: np.ndarray, shared_rows=None, sig=None) -> np.ndarray:
    """y[t] = sum_j w[t, j] rows[t, j] (j in rank order) + sig[t] * shared_rows[t]."""
    T, k, H = rows.shape
    y = np.zeros((T, H), np.float64)
    for j in range(k):
        y += w[:, j:j + 1] * rows[:, j, :]
    if shared_rows is not None:
        y += sig[:, None] * shared_rows
    return y


def moe_layer_batched(x, router_w, sh_gate_vec, experts: dict, shared, k: int, force_ids=None,
                      expert_rows=None, routing=None) -> LayerResult:
    """moe_layer for many tokens. ``experts`` maps expert id -> (gate, up, down) Packed (only the
    routed ones are needed). ``expert_rows(e, token_indices) -> fp64 [n, H]`` may replace the
    per-expert evaluation (the tests run it in worker processes); by default it is
    swiglu_rows on ``experts[e]``. ``routing`` = (ids, w) from route_tokens with the same
    arguments skips recomputing the router."""
    xr = bf16_rows(x)
    T = xr.shape[0]
    if routing is None:
        _, ids, w, _ = route_tokens(x, router_w, k, force_ids)
    else:
        ids, w = routing
    H = xr.shape[1]
    rows = np.zeros((T, k, H), np.float64)
    for e in np.unique(ids):
        tt, jj = np.nonzero(ids == e)
        if expert_rows is not None:
            out = expert_rows(int(e), tt)
        else:
            if int(e) not in experts:
                raise KeyError("routing selected an expert that was not provided")
            out = swiglu_rows(*experts[int(e)], xr[tt])
        rows[tt, jj] = out
    sig = np.zeros(T, np.float64)
    srows = None
    if shared is not None:
        sig = shared_gate(x, sh_gate_vec)
        srows = swiglu_rows(*shared, xr)
    y = combine(rows, w, srows, sig if shared is not None else None)
    return LayerResult(y, ids, w, sig)


# ------------------------------------------------- the layer in the residual stream

def bf16_from_double(v: float) -> int:
    """bits of the bf16 nearest to v (ties to even), rounded directly from fp64."""
    return int(lib().orc_bf16_from_double(float(v)))


def rmsnorm(h, w, eps: float):
    """(bf16 bits [T, H], fp64 values before rounding) of (1 + w) * h / sqrt(mean(h^2) + eps)
    (lynn-engine tutorials index, row 01)."""
    hb = _np(h, np.uint16)
    wb = _np(w, np.uint16)
    T, H = hb.shape
    out = np.zeros((T, H), np.uint16)
    f = np.zeros((T, H), np.float64)
    lib().orc_rmsnorm(_ptr(hb), T, H, _ptr(wb), float(eps), _ptr(out), _ptr(f))
    return out, f


def moe_layer_residual(h, norm_w, eps, router_w, sh_gate_vec, experts: dict, shared, k: int,
                       force_ids=None, batched: bool = False) -> LayerResult:
    """The MoE layer inside the residual stream: x = bf16(RMSNorm_(1+w)(h)), then
    y = h + moe_layer(x) in fp64 (README "decode launch-overhead campaign": fused RMSNorm;
    Lynn write-up, "Fused Kernels"). ``batched`` evaluates the layer with
    moe_layer_batched instead of the per-token C code."""
    xb, _ = rmsnorm(h, norm_w, eps)
    if batched:
        res = moe_layer_batched(xb, router_w, sh_gate_vec, experts, shared, k, force_ids=force_ids)
    else:
        kind = next(iter(experts.values()))[0].kind if experts else SCALE_E4M3
        res = moe_layer(xb, router_w, sh_gate_vec, experts, shared, k, kind=kind, force_ids=force_ids)
    res.y = res.y + bf16_rows(h)
    res.x = xb
    return res
