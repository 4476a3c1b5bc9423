"""Python binding of the GB300 NVFP4 W4A16 MoE library (``libnvfp4moe.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Output tensors are allocated with torch for convenience and their
device pointers handed to the C ABI together with the current CUDA stream.
There is no fallback: if the shared library is missing, importing this module
raises.

The function names are those of the C ABI in ``include/nvfp4moe.h``:
``nvfp4_pack``, ``nvfp4_gemv_w4a16``, ``moe_route_topk``, ``moe_layer_forward``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4moe.so")

SCALE_E4M3 = 0
SCALE_FP16 = 1
SCALE_FP32 = 2     # fp32 scale per 16 elements
SCALE_UE8M0 = 3    # E8M0 power-of-two scale per 32 elements


def scale_shape(rows: int, K: int, kind: int):
    """(shape, dtype) of the block scales of a [rows, K] matrix of the given kind."""
    if kind == SCALE_UE8M0:
        return (rows, K // 32), torch.uint8
    return (rows, K // 16), {SCALE_E4M3: torch.uint8, SCALE_FP16: torch.int16, SCALE_FP32: torch.float32}[kind]


def launches_per_layer_call(T: int, H: int = 2048, kind: int = 0, shared: bool = True, E: int = 256,
                            I: int = 512, Is: int = 512, k: int = 8) -> int:
    """Kernel launches one moe_layer_forward call enqueues (routing outputs not requested):
    one for the single-token fused kernel (E4M3 or FP16 scales); four for the tensor-core multi-token decode
    path (router + route, gate/up, down, combine; E4M3 scales, H, I, Is multiples of
    256 and at most 4096); five for the other multi-token shapes (router, top-k, lists,
    gate/up, down), per 64-token chunk for FP16-scaled layers above 64 tokens; and for
    the prefill path router (and the sum of its K-split partials), gate, top-k, three
    list passes, gate/up, down and combine (no gate launch without a shared expert)."""
    if (T == 1 and kind in (SCALE_E4M3, SCALE_FP16) and H % 256 == 0 and I % 256 == 0 and Is % 256 == 0
            and Is <= I and H <= 4096 and I <= 4096 and k * I + Is <= 8192):
        return 1
    mma = (kind == 0 and H % 256 == 0 and I % 256 == 0 and Is % 256 == 0 and
           H <= 4096 and I <= 4096 and Is <= 4096)
    if T <= 64:
        return 4 if mma else 5
    if kind == 0:
        return (9 if shared else 8) + (1 if (H // 32) % 2 == 0 and (T * E) % 4 == 0 else 0)
    return 5 * ((T + 63) // 64)


STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "pointer not 16-byte aligned",
    4: "workspace too small", 5: "CUDA error", 6: "bounded device wait ran out",
    7: "non-finite input", 8: "device is not sm_103",
}
NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED_SHAPE = 2
NVFP4_ERR_MISALIGNED = 3
NVFP4_ERR_WORKSPACE_TOO_SMALL = 4
NVFP4_ERR_CUDA = 5
NVFP4_ERR_DEVICE_TIMEOUT = 6
NVFP4_ERR_NONFINITE_INPUT = 7
NVFP4_ERR_ARCH = 8


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s: %s (status %d)" % (where, STATUS.get(status, "?"), status))
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError("libnvfp4moe.so is not built (run __graft_entry__.build() or "
                      "python nvfp4_w4a16_moe_gb300/build.py); there is no fallback path")

_P = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t


class NVFP4WeightC(ctypes.Structure):
    _fields_ = [("packed", _P), ("scales", _P), ("tensor_scale", _P), ("N", _i32), ("K", _i32),
                ("kind", _i32)]


class MoELayerDescC(ctypes.Structure):
    _fields_ = [("H", _i32), ("E", _i32), ("k", _i32), ("I", _i32), ("Is", _i32), ("kind", _i32),
                ("router_w", _P), ("gu_packed", _P), ("gu_scales", _P), ("gu_tscale", _P),
                ("dn_packed", _P), ("dn_scales", _P), ("dn_tscale", _P),
                ("sh_gu_packed", _P), ("sh_gu_scales", _P), ("sh_gu_tscale", _P),
                ("sh_dn_packed", _P), ("sh_dn_scales", _P), ("sh_dn_tscale", _P),
                ("sh_gate_w", _P)]


lib = ctypes.CDLL(LIB_PATH)
lib.nvfp4_pack.restype = _i32
lib.nvfp4_pack.argtypes = [_P, _i32, _i32, _i32, _P, _P, _P, _P, _sz, _P]
lib.nvfp4_pack_workspace_size.restype = _sz
lib.nvfp4_pack_workspace_size.argtypes = []
lib.nvfp4_gemv_w4a16.restype = _i32
lib.nvfp4_gemv_w4a16.argtypes = [ctypes.POINTER(NVFP4WeightC), _P, _i32, _P, _P, _sz, _P]
lib.moe_route_topk.restype = _i32
lib.moe_route_topk.argtypes = [_P, _i32, _i32, _i32, _P, _P, _P, _P, _P]
lib.moe_layer_forward.restype = _i32
lib.moe_layer_forward.argtypes = [ctypes.POINTER(MoELayerDescC), _P, _i32, _P, _P, _P, _P, _sz, _P]
lib.moe_layer_workspace_size.restype = _sz
lib.moe_layer_workspace_size.argtypes = [ctypes.POINTER(MoELayerDescC), _i32]
lib.nvfp4_scale_kind_of.restype = _i32
lib.nvfp4_scale_kind_of.argtypes = [_i32, _i32, _sz, _i32, ctypes.POINTER(_i32)]
lib.moe_layer_forward_residual.restype = _i32
lib.moe_layer_forward_residual.argtypes = [ctypes.POINTER(MoELayerDescC), _P, ctypes.c_float, _P, _i32, _P, _P, _P,
                                           _P, _sz, _P]
lib.moe_layer_residual_workspace_size.restype = _sz
lib.moe_layer_residual_workspace_size.argtypes = [ctypes.POINTER(MoELayerDescC), _i32]
lib.nvfp4_workspace_init.restype = _i32
lib.nvfp4_workspace_init.argtypes = [_P, _sz, _P]
lib.nvfp4_get_device_status.restype = _i32
lib.nvfp4_get_device_status.argtypes = [_P, _i32, _P]
lib.nvfp4_set_device_wait_limit.restype = None
lib.nvfp4_set_device_wait_limit.argtypes = [ctypes.c_uint64]
lib.nvfp4_set_single_token_form.restype = None
lib.nvfp4_set_single_token_form.argtypes = [ctypes.c_int32]
lib.nvfp4_single_token_form_used.restype = ctypes.c_int32
lib.nvfp4_single_token_form_used.argtypes = [ctypes.c_void_p, ctypes.c_int32]
lib.nvfp4_single_token_cluster_capacity.restype = ctypes.c_int32
lib.nvfp4_single_token_cluster_capacity.argtypes = [ctypes.c_void_p]
lib.nvfp4_status_string.restype = ctypes.c_char_p
lib.nvfp4_status_string.argtypes = [_i32]
lib.nvfp4_version.restype = _i32
lib.nvfp4_version.argtypes = []
lib.moe_layer_forward_noalloc.restype = _i32
lib.moe_layer_forward_noalloc.argtypes = [ctypes.POINTER(MoELayerDescC), _P, _i32, _P, _P, _P, _P]
lib.nvfp4_noalloc_status.restype = _i32
lib.nvfp4_noalloc_status.argtypes = [_i32, _P]


def _check(status: int, where: str):
    if status != NVFP4_OK:
        raise NVFP4Error(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _u16(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.bfloat16 and t.is_contiguous()
    return t


# ---------------------------------------------------------------- workspace

class Workspace:
    """Caller-owned device scratch for the library calls (zeroed once)."""

    def __init__(self, nbytes: int, device="cuda", stream=None):
        nbytes = max(256, (int(nbytes) + 255) // 256 * 256)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        _check(lib.nvfp4_workspace_init(_ptr(self.buf), nbytes, _stream(stream)), "nvfp4_workspace_init")

    def ptr(self):
        return _ptr(self.buf)

    def status(self, clear: bool = True, stream=None) -> int:
        return lib.nvfp4_get_device_status(_ptr(self.buf), 1 if clear else 0, _stream(stream))


_PACK_WS = {}


def _pack_ws(device) -> Workspace:
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    ws = _PACK_WS.get(key)
    if ws is None:
        ws = Workspace(lib.nvfp4_pack_workspace_size(), device=device)
        _PACK_WS[key] = ws
    return ws


# ---------------------------------------------------------------- pack

@dataclass
class NVFP4Weight:
    """One packed matrix on the device."""
    packed: torch.Tensor        # uint8 [N, K/2]
    scales: torch.Tensor        # uint8 [N, K/16] (E4M3) or int16 [N, K/16] (FP16 bits)
    tensor_scale: torch.Tensor  # float32 [1]
    N: int
    K: int
    kind: int

    def c(self) -> NVFP4WeightC:
        return NVFP4WeightC(self.packed.data_ptr(), self.scales.data_ptr(), self.tensor_scale.data_ptr(),
                            self.N, self.K, self.kind)


def nvfp4_pack(w: torch.Tensor, kind: int = SCALE_E4M3, out: Optional[NVFP4Weight] = None,
               ws: Optional[Workspace] = None, check: bool = False, stream=None) -> NVFP4Weight:
    """Quantise fp32 W[N, K] (CUDA) to NVFP4 with the library's packer."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous() and w.dim() == 2
    N, K = w.shape
    if out is None:
        sshape, sdt = scale_shape(N, K, kind)
        out = NVFP4Weight(torch.empty(N, K // 2, dtype=torch.uint8, device=w.device),
                          torch.empty(*sshape, dtype=sdt, device=w.device),
                          torch.empty(1, dtype=torch.float32, device=w.device), N, K, kind)
    ws = ws or _pack_ws(w.device)
    _check(lib.nvfp4_pack(_ptr(w), N, K, kind, _ptr(out.packed), _ptr(out.scales), _ptr(out.tensor_scale),
                          ws.ptr(), ws.nbytes, _stream(stream)), "nvfp4_pack")
    if check:
        _check(ws.status(clear=True, stream=stream), "nvfp4_pack (device)")
    return out


def nvfp4_pack_into(w: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, tensor_scale: torch.Tensor,
                    kind: int = SCALE_E4M3, ws: Optional[Workspace] = None, stream=None):
    """Pack fp32 W[N, K] into caller-provided (contiguous) views, e.g. slices of a grouped buffer."""
    N, K = w.shape
    assert packed.is_contiguous() and scales.is_contiguous()
    ws = ws or _pack_ws(w.device)
    _check(lib.nvfp4_pack(_ptr(w), N, K, kind, _ptr(packed), _ptr(scales), _ptr(tensor_scale),
                          ws.ptr(), ws.nbytes, _stream(stream)), "nvfp4_pack")


def nvfp4_scale_kind_of(N: int, K: int, scales) -> int:
    """The scale contract of an [N, K] NVFP4 matrix from its scale tensor's metadata (element
    count and size); raises NVFP4Error when it matches none."""
    out = _i32(-1)
    _check(lib.nvfp4_scale_kind_of(N, K, scales.numel(), scales.element_size(), ctypes.byref(out)),
           "nvfp4_scale_kind_of")
    return out.value


# ---------------------------------------------------------------- GEMV

def nvfp4_gemv_w4a16(W: NVFP4Weight, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None):
    """y[T, N] bf16 = W x for x bf16 [T, K] (1 <= T <= 64)."""
    x = _u16(x)
    T = x.shape[0]
    if y is None:
        y = torch.empty(T, W.N, dtype=torch.bfloat16, device=x.device)
    wc = W.c()
    _check(lib.nvfp4_gemv_w4a16(ctypes.byref(wc), _ptr(x), T, _ptr(y), None, 0, _stream(stream)),
           "nvfp4_gemv_w4a16")
    return y


# ---------------------------------------------------------------- route

def moe_route_topk(logits: torch.Tensor, k: int, stream=None):
    """(ids [T,k] int32, w [T,k] fp32, offsets [E+1] int32, token_list [T*k] int32)."""
    assert logits.dtype == torch.float32 and logits.is_contiguous()
    T, E = logits.shape
    dev = logits.device
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    tl = torch.empty(max(T * k, 4), dtype=torch.int32, device=dev)
    _check(lib.moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(tl),
                              _stream(stream)), "moe_route_topk")
    return ids, w, offsets, tl[:T * k]


# ---------------------------------------------------------------- layer

@dataclass
class MoELayer:
    """Device buffers of one layer in the library's canonical layout."""
    H: int
    E: int
    k: int
    I: int
    Is: int
    kind: int
    router_w: torch.Tensor      # bf16 [E, H]
    gu_packed: torch.Tensor     # u8 [E, 2I, H/2]
    gu_scales: torch.Tensor     # [E, 2I, H/16]
    gu_tscale: torch.Tensor     # f32 [E, 2]
    dn_packed: torch.Tensor     # u8 [E, H, I/2]
    dn_scales: torch.Tensor     # [E, H, I/16]
    dn_tscale: torch.Tensor     # f32 [E]
    sh_gu_packed: Optional[torch.Tensor] = None
    sh_gu_scales: Optional[torch.Tensor] = None
    sh_gu_tscale: Optional[torch.Tensor] = None
    sh_dn_packed: Optional[torch.Tensor] = None
    sh_dn_scales: Optional[torch.Tensor] = None
    sh_dn_tscale: Optional[torch.Tensor] = None
    sh_gate_w: Optional[torch.Tensor] = None

    @staticmethod
    def allocate(H, E, k, I, Is, kind=SCALE_E4M3, device="cuda") -> "MoELayer":
        z = dict(device=device)
        (_, gcols), sdt = scale_shape(1, H, kind)
        (_, dcols), _ = scale_shape(1, I, kind)
        L = MoELayer(H, E, k, I, Is, kind,
                     torch.empty(E, H, dtype=torch.bfloat16, **z),
                     torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, **z),
                     torch.empty(E, 2 * I, gcols, dtype=sdt, **z),
                     torch.empty(E, 2, dtype=torch.float32, **z),
                     torch.empty(E, H, I // 2, dtype=torch.uint8, **z),
                     torch.empty(E, H, dcols, dtype=sdt, **z),
                     torch.empty(E, dtype=torch.float32, **z))
        if Is > 0:
            (_, scols), _ = scale_shape(1, Is, kind)
            L.sh_gu_packed = torch.empty(2 * Is, H // 2, dtype=torch.uint8, **z)
            L.sh_gu_scales = torch.empty(2 * Is, gcols, dtype=sdt, **z)
            L.sh_gu_tscale = torch.empty(4, dtype=torch.float32, **z)   # 2 used, 16-byte aligned
            L.sh_dn_packed = torch.empty(H, Is // 2, dtype=torch.uint8, **z)
            L.sh_dn_scales = torch.empty(H, scols, dtype=sdt, **z)
            L.sh_dn_tscale = torch.empty(4, dtype=torch.float32, **z)
            L.sh_gate_w = torch.empty(H, dtype=torch.bfloat16, **z)
        return L

    def pack_expert(self, e: int, gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor, stream=None):
        """Pack fp32 gate [I,H], up [I,H], down [H,I] (CUDA) into expert slot e."""
        I = self.I
        nvfp4_pack_into(gate.contiguous(), self.gu_packed[e, :I], self.gu_scales[e, :I], self.gu_tscale[e, 0:1],
                        self.kind, stream=stream)
        nvfp4_pack_into(up.contiguous(), self.gu_packed[e, I:], self.gu_scales[e, I:], self.gu_tscale[e, 1:2],
                        self.kind, stream=stream)
        nvfp4_pack_into(down.contiguous(), self.dn_packed[e], self.dn_scales[e], self.dn_tscale[e:e + 1],
                        self.kind, stream=stream)

    def pack_shared(self, gate, up, down, gate_vec: torch.Tensor, stream=None):
        Is = self.Is
        nvfp4_pack_into(gate.contiguous(), self.sh_gu_packed[:Is], self.sh_gu_scales[:Is], self.sh_gu_tscale[0:1],
                        self.kind, stream=stream)
        nvfp4_pack_into(up.contiguous(), self.sh_gu_packed[Is:], self.sh_gu_scales[Is:], self.sh_gu_tscale[1:2],
                        self.kind, stream=stream)
        nvfp4_pack_into(down.contiguous(), self.sh_dn_packed, self.sh_dn_scales, self.sh_dn_tscale[0:1],
                        self.kind, stream=stream)
        self.sh_gate_w.copy_(gate_vec)

    def desc(self) -> MoELayerDescC:
        d = MoELayerDescC()
        d.H, d.E, d.k, d.I, d.Is, d.kind = self.H, self.E, self.k, self.I, self.Is, self.kind
        for name in ("router_w", "gu_packed", "gu_scales", "gu_tscale", "dn_packed", "dn_scales", "dn_tscale",
                     "sh_gu_packed", "sh_gu_scales", "sh_gu_tscale", "sh_dn_packed", "sh_dn_scales",
                     "sh_dn_tscale", "sh_gate_w"):
            t = getattr(self, name)
            setattr(d, name, None if t is None else t.data_ptr())
        return d

    def weight_bytes_per_expert(self) -> int:
        H, I = self.H, self.I
        (_, gc), gdt = scale_shape(1, H, self.kind)
        (_, dc), _ = scale_shape(1, I, self.kind)
        sb = torch.tensor([], dtype=gdt).element_size()
        return 2 * I * H // 2 + 2 * I * gc * sb + H * I // 2 + H * dc * sb + 12


def moe_layer_workspace_size(layer: MoELayer, T: int) -> int:
    d = layer.desc()
    return int(lib.moe_layer_workspace_size(ctypes.byref(d), T))


def moe_layer_forward(layer: MoELayer, x: torch.Tensor, ws: Optional[Workspace] = None,
                      y: Optional[torch.Tensor] = None, ids_out: Optional[torch.Tensor] = None,
                      w_out: Optional[torch.Tensor] = None, want_route: bool = False, stream=None,
                      desc: Optional[MoELayerDescC] = None):
    """y [T, H] bf16 (and optionally the routing) for x [T, H] bf16."""
    x = _u16(x)
    T = x.shape[0]
    d = desc if desc is not None else layer.desc()
    if ws is None:
        ws = Workspace(lib.moe_layer_workspace_size(ctypes.byref(d), T), device=x.device, stream=stream)
    if y is None:
        y = torch.empty(T, layer.H, dtype=torch.bfloat16, device=x.device)
    if want_route and ids_out is None:
        ids_out = torch.empty(T, layer.k, dtype=torch.int32, device=x.device)
        w_out = torch.empty(T, layer.k, dtype=torch.float32, device=x.device)
    _check(lib.moe_layer_forward(ctypes.byref(d), _ptr(x), T, _ptr(y), _ptr(ids_out), _ptr(w_out),
                                 ws.ptr(), ws.nbytes, _stream(stream)), "moe_layer_forward")
    if want_route:
        return y, ids_out, w_out
    return y


def moe_layer_forward_residual(layer: MoELayer, h: torch.Tensor, norm_w: torch.Tensor, eps: float = 1e-6,
                               ws: Optional[Workspace] = None, h_out: Optional[torch.Tensor] = None,
                               want_route: bool = False, stream=None, desc: Optional[MoELayerDescC] = None):
    """h_out = h + layer(RMSNorm_(1+w)(h)) [T, H] bf16 (and optionally the routing) for the
    residual stream h [T, H] bf16; h_out may be h itself."""
    h = _u16(h)
    T = h.shape[0]
    d = desc if desc is not None else layer.desc()
    if ws is None:
        ws = Workspace(lib.moe_layer_residual_workspace_size(ctypes.byref(d), T), device=h.device, stream=stream)
    if h_out is None:
        h_out = torch.empty(T, layer.H, dtype=torch.bfloat16, device=h.device)
    ids_out = w_out = None
    if want_route:
        ids_out = torch.empty(T, layer.k, dtype=torch.int32, device=h.device)
        w_out = torch.empty(T, layer.k, dtype=torch.float32, device=h.device)
    _check(lib.moe_layer_forward_residual(ctypes.byref(d), _ptr(_u16(norm_w)), float(eps), _ptr(h), T, _ptr(h_out),
                                          _ptr(ids_out), _ptr(w_out), ws.ptr(), ws.nbytes, _stream(stream)),
           "moe_layer_forward_residual")
    if want_route:
        return h_out, ids_out, w_out
    return h_out


def moe_layer_forward_noalloc(layer: MoELayer, x: torch.Tensor, y: Optional[torch.Tensor] = None,
                              ids_out: Optional[torch.Tensor] = None, w_out: Optional[torch.Tensor] = None,
                              want_route: bool = False, stream=None):
    """moe_layer_forward with the library's static scratch instead of a workspace
    (for callers that cannot allocate device memory where they run the layer)."""
    x = _u16(x)
    T = x.shape[0]
    d = layer.desc()
    if y is None:
        y = torch.empty(T, layer.H, dtype=torch.bfloat16, device=x.device)
    if want_route and ids_out is None:
        ids_out = torch.empty(T, layer.k, dtype=torch.int32, device=x.device)
        w_out = torch.empty(T, layer.k, dtype=torch.float32, device=x.device)
    _check(lib.moe_layer_forward_noalloc(ctypes.byref(d), _ptr(x), T, _ptr(y), _ptr(ids_out), _ptr(w_out),
                                         _stream(stream)), "moe_layer_forward_noalloc")
    if want_route:
        return y, ids_out, w_out
    return y


def noalloc_status(clear: bool = True, stream=None) -> int:
    """The status word a kernel of the last moe_layer_forward_noalloc call on the current
    device recorded (NVFP4_OK, or NVFP4_ERR_DEVICE_TIMEOUT when a bounded wait ran out);
    synchronises the stream first."""
    return lib.nvfp4_noalloc_status(1 if clear else 0, _stream(stream))


def set_device_wait_limit(spins: int):
    lib.nvfp4_set_device_wait_limit(int(spins))


SINGLE_TOKEN_AUTO = 0
SINGLE_TOKEN_GRID = 1
SINGLE_TOKEN_CLUSTER = 2


def set_single_token_form(form: int):
    """0: automatic (the persistent-grid form), 1: the grid form, 2: the cluster form
    where supported."""
    lib.nvfp4_set_single_token_form(int(form))


def single_token_form_used(layer: "MoELayer", T: int = 1) -> int:
    """2: the cluster form runs a T-token call of this layer, 1: the grid form, 0: neither."""
    d = layer.desc()
    return int(lib.nvfp4_single_token_form_used(ctypes.byref(d), int(T)))


def single_token_cluster_capacity(layer: "MoELayer") -> int:
    """Resident 16-CTA clusters of the cluster form on this device for this layer."""
    d = layer.desc()
    return int(lib.nvfp4_single_token_cluster_capacity(ctypes.byref(d)))


def version() -> int:
    return lib.nvfp4_version()
