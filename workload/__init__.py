"""Seeded synthetic inputs shared by the tests, the bench and the oracle harness.

This module only draws numbers. It holds none of the layer's arithmetic: no
packing, no dequantisation, no router, no activation. Both sides of every
parity check (the CUDA library and the CPU oracle) receive their fp32 / bf16
inputs from here, so that they see identical bits.

Generator
---------
Every tensor is addressed by a *stream key* built from small integers
(seed, tensor kind, layer, expert, ...). Element ``i`` of a stream takes the
32-bit hash ``mix32((i >> 1) + key)`` and uses its high (odd ``i``) or low
(even ``i``) 16 bits as an index into a fixed table of 65536 standard-normal
quantiles, ``Phi^-1((j + 0.5) / 65536)`` rounded to fp32. The result is
multiplied by the requested standard deviation in fp32 (one correctly-rounded
IEEE multiply). The hash is the public-domain "lowbias32" integer finaliser
(xor-shift / multiply, constants 0x7feb352d and 0x846ca68b).

All of it is integer arithmetic plus one fp32 multiply, so the CPU and any
CUDA device produce bit-identical values: on a CUDA device it runs as int64
torch ops, on the CPU as uint64 numpy ops (the same operations, faster there).
The large weight sets for the bench are drawn directly on the GPU, and the
oracle redraws only the experts it needs on the CPU.
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass, field

import numpy as np
import torch

M32 = 0xFFFFFFFF

# tensor-kind ids used in stream keys
K_X = 1
K_ROUTER = 2
K_GATE = 3
K_UP = 4
K_DOWN = 5
K_SH_GATE = 6
K_SH_UP = 7
K_SH_DOWN = 8
K_SH_SIGMOID = 9
K_DENSE = 10
K_PERM = 11


def mix32_int(v: int) -> int:
    """lowbias32 finaliser on a Python int (exact, used for keys)."""
    v &= M32
    v ^= v >> 16
    v = (v * 0x7FEB352D) & M32
    v ^= v >> 15
    v = (v * 0x846CA68B) & M32
    v ^= v >> 16
    return v


def stream_key(*parts: int) -> int:
    """Fold small integers into one 32-bit stream key."""
    k = 0x9E3779B9
    for p in parts:
        k = mix32_int(k ^ mix32_int(int(p) + 0x632BE5AB))
    return k


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow: split x in halves.
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & M32


def mix32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 finaliser on an int64 tensor holding values in [0, 2^32)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


_TABLES: dict = {}


def _quantile_table(device) -> torch.Tensor:
    dev = torch.device(device)
    key = str(dev)
    t = _TABLES.get(key)
    if t is None:
        base = _TABLES.get("cpu")
        if base is None:
            nd = statistics.NormalDist()
            vals = [nd.inv_cdf((j + 0.5) / 65536.0) for j in range(65536)]
            base = torch.tensor(vals, dtype=torch.float64).to(torch.float32)
            _TABLES["cpu"] = base
        t = base.to(dev)
        _TABLES[key] = t
    return t


def _mix32_np(x: np.ndarray) -> np.ndarray:
    """lowbias32 finaliser on a uint64 array holding values in [0, 2^32)."""
    x = x ^ (x >> np.uint64(16))
    x = (x * np.uint64(0x7FEB352D)) & np.uint64(M32)
    x = x ^ (x >> np.uint64(15))
    x = (x * np.uint64(0x846CA68B)) & np.uint64(M32)
    x = x ^ (x >> np.uint64(16))
    return x


def _normal_np(key: int, n: int, std: float, start: int) -> torch.Tensor:
    # the same draws as _normal_torch, with numpy's uint64 arithmetic (faster on the CPU)
    idx = np.arange(start, start + n, dtype=np.uint64)
    h = _mix32_np(((idx >> np.uint64(1)) + np.uint64(key)) & np.uint64(M32))
    half = np.where((idx & np.uint64(1)) == 1, h >> np.uint64(16), h & np.uint64(0xFFFF))
    z = _quantile_table("cpu").numpy()[half.astype(np.int64)]
    return torch.from_numpy(z * np.float32(std))


def normal(key: int, n: int, std: float = 1.0, device="cpu", start: int = 0) -> torch.Tensor:
    """``n`` draws of N(0, std^2) (fp32) from stream ``key``, elements ``start..start+n``."""
    if n == 0:
        return torch.empty(0, dtype=torch.float32, device=device)
    if torch.device(device).type == "cpu":
        return _normal_np(key, n, std, start)
    return _normal_torch(key, n, std, device, start)


def _normal_torch(key: int, n: int, std: float, device, start: int) -> torch.Tensor:
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    h = mix32(((idx >> 1) + key) & M32)
    half = torch.where((idx & 1) == 1, h >> 16, h & 0xFFFF)
    z = _quantile_table(device)[half]
    return z * torch.tensor(std, dtype=torch.float32, device=device)


def uniform_u32(key: int, n: int, device="cpu") -> torch.Tensor:
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return mix32((idx + key) & M32)


def permutation(key: int, n: int) -> list:
    """Seeded permutation of range(n): sort by hash (ties impossible in practice; index breaks them)."""
    h = uniform_u32(key, n).tolist()
    return sorted(range(n), key=lambda i: (h[i], i))


# --------------------------------------------------------------------------------------
# Workload recipes (shapes and distributions of the layer these inputs feed)
# --------------------------------------------------------------------------------------

@dataclass(frozen=True)
class MoEShape:
    H: int      # hidden size
    E: int      # routed experts
    k: int      # experts per token
    I: int      # routed expert intermediate size
    Is: int     # shared expert intermediate size
    w_std: float = 0.02      # expert / router weight std
    router_kappa: float = 0.0  # >0: router row r scaled by rank^-kappa (skewed popularity)


TINY = MoEShape(H=256, E=16, k=2, I=128, Is=128)
# smallest shape whose prefill runs the grouped tensor-core path (H, I, Is multiples of 256)
SMALL256 = MoEShape(H=256, E=16, k=2, I=256, Is=256)
QWEN36_35B_A3B = MoEShape(H=2048, E=256, k=8, I=512, Is=512)


@dataclass
class LayerInputs:
    """fp32 master weights of one MoE layer, drawn from a seed (lazily per expert)."""
    shape: MoEShape
    seed: int
    layer: int = 0
    device: str = "cpu"
    _perm: list = field(default=None, repr=False)

    def _k(self, kind, *rest):
        return stream_key(self.seed, self.layer, kind, *rest)

    def router_w_f32(self, device=None) -> torch.Tensor:
        s = self.shape
        dev = device or self.device
        w = normal(self._k(K_ROUTER), s.E * s.H, s.w_std, dev).view(s.E, s.H)
        if s.router_kappa > 0.0:
            if self._perm is None:
                self._perm = permutation(self._k(K_PERM), s.E)
            rank = torch.tensor([1 + self._perm[e] for e in range(s.E)], dtype=torch.float64)
            f = rank.pow(-s.router_kappa).to(torch.float32).to(dev)
            w = w * f[:, None]
        return w

    def router_w(self, device=None) -> torch.Tensor:
        """Router gate weight [E, H] in bf16."""
        return self.router_w_f32(device).to(torch.bfloat16)

    def shared_sigmoid_w(self, device=None) -> torch.Tensor:
        """Shared-expert gate vector [H] in bf16."""
        s = self.shape
        return normal(self._k(K_SH_SIGMOID), s.H, s.w_std, device or self.device).to(torch.bfloat16)

    def expert_f32(self, e: int, device=None):
        """(gate [I,H], up [I,H], down [H,I]) fp32 for routed expert ``e``."""
        s = self.shape
        dev = device or self.device
        g = normal(self._k(K_GATE, e), s.I * s.H, s.w_std, dev).view(s.I, s.H)
        u = normal(self._k(K_UP, e), s.I * s.H, s.w_std, dev).view(s.I, s.H)
        d = normal(self._k(K_DOWN, e), s.H * s.I, s.w_std, dev).view(s.H, s.I)
        return g, u, d

    def shared_f32(self, device=None):
        """(gate [Is,H], up [Is,H], down [H,Is]) fp32 of the shared expert."""
        s = self.shape
        dev = device or self.device
        g = normal(self._k(K_SH_GATE), s.Is * s.H, s.w_std, dev).view(s.Is, s.H)
        u = normal(self._k(K_SH_UP), s.Is * s.H, s.w_std, dev).view(s.Is, s.H)
        d = normal(self._k(K_SH_DOWN), s.H * s.Is, s.w_std, dev).view(s.H, s.Is)
        return g, u, d


def activations(seed: int, T: int, H: int, device="cpu", layer: int = 0, attempts=None) -> torch.Tensor:
    """x [T, H] bf16 ~ N(0,1). ``attempts[t]`` selects a redraw of token t (default 0)."""
    rows = []
    for t in range(T):
        a = 0 if attempts is None else int(attempts[t])
        rows.append(normal(stream_key(seed, layer, K_X, t, a), H, 1.0, device))
    if T == 0:
        return torch.empty(0, H, dtype=torch.bfloat16, device=device)
    return torch.stack(rows).to(torch.bfloat16)


def dense_weight_f32(seed: int, N: int, K: int, std: float = 0.02, device="cpu") -> torch.Tensor:
    """Dense projection weight [N, K] fp32 ~ N(0, std^2)."""
    return normal(stream_key(seed, 0, K_DENSE), N * K, std, device).view(N, K)
