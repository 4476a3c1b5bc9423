"""nvfp4_pack on the GPU against the oracle's packer: bytes, scales and tensor
scale bit-exact (both scale kinds), including zeros, signed zeros, midpoints,
E4M3-subnormal block scales, ragged shapes and the non-finite error path."""
import numpy as np
import pytest
import torch

import oracle
import workload as wl

pytestmark = pytest.mark.gpu


def _compare(nv, w_cpu, kind):
    w = w_cpu.contiguous().cuda()
    p = nv.nvfp4_pack(w, kind, check=True)
    torch.cuda.synchronize()
    ref = oracle.pack(w_cpu, kind)
    got_packed = p.packed.cpu().numpy()
    got_scales = p.scales.cpu().numpy().view(np.uint8 if kind == 0 else np.uint16)
    assert np.array_equal(got_scales, ref.scales), "scales differ"
    assert np.float32(p.tensor_scale.item()) == np.float32(ref.tensor_scale)
    if not np.array_equal(got_packed, ref.packed):
        bad = np.argwhere(got_packed != ref.packed)[:5]
        raise AssertionError("packed bytes differ at %s: gpu %s oracle %s" % (
            bad.tolist(), got_packed[tuple(bad.T)], ref.packed[tuple(bad.T)]))


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (7, 256), (512, 2048), (2048, 512), (33, 8192)])
def test_pack_bit_exact_random(nv, kind, N, K):
    w = wl.normal(wl.stream_key(100, N, K), N * K, 0.02).view(N, K)
    _compare(nv, w, kind)


@pytest.mark.parametrize("kind", [0, 1])
def test_pack_bit_exact_special_values(nv, kind):
    rng = np.random.default_rng(7)
    N, K = 64, 256
    w = rng.normal(0, 1, size=(N, K)).astype(np.float32)
    w[0] = 0.0                                   # all-zero block rows
    w[1, :16] = -0.0                             # signed zeros
    w[2] *= 1e-6                                 # tiny blocks (E4M3 subnormal scales)
    w[3] *= 1e6
    w[4, ::3] = 0.0
    # exact E2M1 midpoints relative to a block amax of 6
    mids = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, -6],
                    np.float32)
    w[5, :16] = mids
    w[6, :16] = mids * 2.0 ** -12
    w[7] = rng.normal(0, 1e-3, K).astype(np.float32) * (np.arange(K) % 16 == 0)
    w[8, 0] = 3.0e4                              # a large outlier sets the tensor scale
    _compare(nv, torch.from_numpy(w), kind)


def test_pack_full_expert_matrices(nv):
    L = wl.LayerInputs(wl.QWEN36_35B_A3B, seed=0)
    g, u, d = L.expert_f32(17)
    for m in (g, u, d):
        _compare(nv, m, 0)
    _compare(nv, L.shared_f32()[2], 0)


def test_pack_nonfinite_reports_status(nv):
    w = torch.zeros(4, 32)
    w[2, 5] = float("nan")
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.nvfp4_pack(w.cuda(), 0, check=True)
    assert ei.value.status == nv.NVFP4_ERR_NONFINITE_INPUT
    w[2, 5] = float("-inf")
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_pack(w.cuda(), 1, check=True)
    # the status was cleared: a finite matrix packs cleanly again
    nv.nvfp4_pack(torch.ones(4, 32).cuda(), 0, check=True)
