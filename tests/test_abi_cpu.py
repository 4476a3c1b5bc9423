"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments before it
touches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_w4a16_moe_gb300 as nv
    return nv


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"NVFP4_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for n in ("nvfp4_pack", "nvfp4_gemv_w4a16", "moe_route_topk", "moe_layer_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(nv):
    lib = ctypes.CDLL(nv.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(nv):
    assert nv.version() == 1
    for code in range(9):
        s = nv.lib.nvfp4_status_string(code).decode()
        assert s and s != "unknown status"


def test_null_and_misaligned_arguments_rejected(nv):
    lib = nv.lib
    fake = ctypes.c_void_p(0x100000)        # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x100008)
    assert lib.nvfp4_pack(None, 4, 32, 0, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_pack(fake, 4, 30, 0, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_pack(fake, 4, 32, 5, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_pack(odd, 4, 32, 0, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_MISALIGNED
    assert lib.nvfp4_pack(fake, 4, 32, 0, fake, fake, fake, fake, 16, None) == nv.NVFP4_ERR_WORKSPACE_TOO_SMALL
    W = nv.NVFP4WeightC(0x100000, 0x100000, 0x100000, 64, 2048, 0)
    assert lib.nvfp4_gemv_w4a16(ctypes.byref(W), fake, 0, fake, None, 0, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemv_w4a16(ctypes.byref(W), fake, 65, fake, None, 0, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    W.K = 48
    assert lib.nvfp4_gemv_w4a16(ctypes.byref(W), fake, 1, fake, None, 0, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    W.K = 2048
    assert lib.nvfp4_gemv_w4a16(ctypes.byref(W), odd, 1, fake, None, 0, None) == nv.NVFP4_ERR_MISALIGNED
    assert lib.moe_route_topk(fake, 4, 16, 9, fake, fake, fake, fake, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_route_topk(fake, 4, 300, 2, fake, fake, fake, fake, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_route_topk(None, 4, 16, 2, fake, fake, fake, fake, None) == nv.NVFP4_ERR_INVALID_ARG


def _desc(nv, **kw):
    d = nv.MoELayerDescC()
    d.H, d.E, d.k, d.I, d.Is, d.kind = 2048, 256, 8, 512, 512, 0
    for name in ("router_w", "gu_packed", "gu_scales", "gu_tscale", "dn_packed", "dn_scales", "dn_tscale",
                 "sh_gu_packed", "sh_gu_scales", "sh_gu_tscale", "sh_dn_packed", "sh_dn_scales", "sh_dn_tscale",
                 "sh_gate_w"):
        setattr(d, name, 0x200000)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_layer_argument_checks(nv):
    lib = nv.lib
    fake = ctypes.c_void_p(0x100000)
    d = _desc(nv)
    ws = lib.moe_layer_workspace_size(ctypes.byref(d), 1)
    assert ws > 0
    assert lib.moe_layer_workspace_size(ctypes.byref(d), 64) > ws
    bad = [
        (_desc(nv, k=9), nv.NVFP4_ERR_UNSUPPORTED_SHAPE),
        (_desc(nv, E=4, k=5), nv.NVFP4_ERR_UNSUPPORTED_SHAPE),
        (_desc(nv, E=257), nv.NVFP4_ERR_UNSUPPORTED_SHAPE),
        (_desc(nv, H=2040), nv.NVFP4_ERR_UNSUPPORTED_SHAPE),
        (_desc(nv, I=500), nv.NVFP4_ERR_UNSUPPORTED_SHAPE),
        (_desc(nv, kind=7), nv.NVFP4_ERR_INVALID_ARG),
        (_desc(nv, gu_packed=None), nv.NVFP4_ERR_INVALID_ARG),
        (_desc(nv, dn_scales=0x200004), nv.NVFP4_ERR_MISALIGNED),
        (_desc(nv, sh_gate_w=None), nv.NVFP4_ERR_INVALID_ARG),
    ]
    for dd, want in bad:
        assert lib.moe_layer_forward(ctypes.byref(dd), fake, 1, fake, None, None, fake, ws, None) == want
    # Is = 0: shared pointers may be NULL; then the workspace check is reached
    d0 = _desc(nv, Is=0, sh_gate_w=None, sh_gu_packed=None)
    assert lib.moe_layer_forward(ctypes.byref(d0), fake, 1, fake, None, None, fake, 16, None) == \
        nv.NVFP4_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_layer_forward(ctypes.byref(d), fake, 1, fake, None, None, None, ws, None) == \
        nv.NVFP4_ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(d), ctypes.c_void_p(0x100002), 1, fake, None, None, fake, ws,
                                 None) == nv.NVFP4_ERR_MISALIGNED


def test_residual_and_kind_argument_checks(nv):
    """Host-side checks of moe_layer_forward_residual and of the scale-kind tag (nothing is
    enqueued when a check fails, so no GPU is needed)."""
    lib = nv.lib
    fake = ctypes.c_void_p(0x100000)
    d = _desc(nv)
    ws = lib.moe_layer_residual_workspace_size(ctypes.byref(d), 1)
    assert ws > lib.moe_layer_workspace_size(ctypes.byref(d), 1)
    call = lambda dd, nw=fake, eps=1e-6, h=fake, out=fake, wsb=ws: lib.moe_layer_forward_residual(
        ctypes.byref(dd), nw, eps, h, 1, out, None, None, fake, wsb, None)
    assert call(d, nw=None) == nv.NVFP4_ERR_INVALID_ARG
    assert call(d, eps=-1.0) == nv.NVFP4_ERR_INVALID_ARG
    assert call(d, eps=float("nan")) == nv.NVFP4_ERR_INVALID_ARG
    assert call(d, nw=ctypes.c_void_p(0x100008)) == nv.NVFP4_ERR_MISALIGNED
    assert call(d, wsb=16) == nv.NVFP4_ERR_WORKSPACE_TOO_SMALL
    assert call(_desc(nv, kind=9)) == nv.NVFP4_ERR_INVALID_ARG
    # pack: E8M0 blocks are 32 elements
    assert lib.nvfp4_pack(fake, 4, 48, 3, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_pack(fake, 4, 48, 5, fake, fake, fake, fake, 256, None) == nv.NVFP4_ERR_INVALID_ARG


def test_scale_kind_classifier(nv):
    """Metadata-only classification of the stored scale contract (README P59): every kind
    is recognised from (count, element size), everything else is refused."""
    import torch
    N, K = 12, 256
    cases = [((N, K // 16), torch.uint8, nv.SCALE_E4M3), ((N, K // 16), torch.int16, nv.SCALE_FP16),
             ((N, K // 16), torch.float32, nv.SCALE_FP32), ((N, K // 32), torch.uint8, nv.SCALE_UE8M0)]
    for shape, dt, want in cases:
        assert nv.nvfp4_scale_kind_of(N, K, torch.empty(shape, dtype=dt)) == want
        shp, sdt = nv.scale_shape(N, K, want)
        assert tuple(shp) == shape and sdt == dt
    for shape, dt in [((N, K // 32), torch.int16), ((N, K // 8), torch.uint8), ((N, K // 16 + 1), torch.uint8),
                      ((N, K // 32), torch.float32)]:
        with pytest.raises(nv.NVFP4Error):
            nv.nvfp4_scale_kind_of(N, K, torch.empty(shape, dtype=dt))
    # K = 48 has no per-32 reading
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_scale_kind_of(4, 48, torch.empty(4, 1, dtype=torch.uint8))
