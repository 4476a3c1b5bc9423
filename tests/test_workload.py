"""Pins for the seeded input generator (shared by both sides of every parity check)."""
import numpy as np
import torch

import workload as wl


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    # the published finaliser, written with wrapping uint32 arithmetic
    x = x.astype(np.uint32)
    x ^= x >> np.uint32(16)
    x = (x * np.uint32(0x7FEB352D)).astype(np.uint32)
    x ^= x >> np.uint32(15)
    x = (x * np.uint32(0x846CA68B)).astype(np.uint32)
    x ^= x >> np.uint32(16)
    return x


def test_mix32_matches_uint32_definition():
    rng = np.random.default_rng(0)
    v = rng.integers(0, 2**32, size=100000, dtype=np.uint64)
    v[:4] = [0, 1, 0xFFFFFFFF, 0x80000000]
    got = wl.mix32(torch.from_numpy(v.astype(np.int64))).numpy()
    with np.errstate(over="ignore"):
        want = _lowbias32_np(v)
    assert np.array_equal(got.astype(np.uint32), want)
    assert wl.mix32_int(12345) == int(_lowbias32_np(np.array([12345]))[0])


def test_normal_moments_and_determinism():
    a = wl.normal(wl.stream_key(1, 2, 3), 1 << 20, 1.0)
    b = wl.normal(wl.stream_key(1, 2, 3), 1 << 20, 1.0)
    assert torch.equal(a, b)
    assert abs(a.mean().item()) < 5e-3
    assert abs(a.std().item() - 1.0) < 5e-3
    # fourth moment of a normal is 3
    assert abs((a.double() ** 4).mean().item() - 3.0) < 0.05
    c = wl.normal(wl.stream_key(1, 2, 4), 1 << 20, 1.0)
    assert not torch.equal(a, c)
    # correlation between different streams is negligible
    assert abs(torch.corrcoef(torch.stack([a, c]))[0, 1].item()) < 5e-3


def test_normal_offset_window():
    k = wl.stream_key(7)
    full = wl.normal(k, 1000, 0.02)
    part = wl.normal(k, 300, 0.02, start=501)
    assert torch.equal(full[501:801], part)


def test_std_scaling_is_one_fp32_multiply():
    k = wl.stream_key(9)
    z = wl.normal(k, 4096, 1.0)
    w = wl.normal(k, 4096, 0.02)
    assert torch.equal(w, z * torch.tensor(0.02, dtype=torch.float32))


def test_layer_inputs_shapes():
    L = wl.LayerInputs(wl.TINY, seed=0)
    g, u, d = L.expert_f32(3)
    assert g.shape == (128, 256) and u.shape == (128, 256) and d.shape == (256, 128)
    assert L.router_w().dtype == torch.bfloat16 and L.router_w().shape == (16, 256)
    x = wl.activations(0, 3, 256)
    assert x.shape == (3, 256) and x.dtype == torch.bfloat16
    x2 = wl.activations(0, 3, 256, attempts=[0, 1, 0])
    assert torch.equal(x[0], x2[0]) and not torch.equal(x[1], x2[1])


def test_cpu_and_torch_draws_are_bit_identical():
    """The CPU path (numpy uint64) and the torch int64 path draw the same bits."""
    for key, n, std, start in [(wl.stream_key(1, 2, 3), 100003, 0.02, 0), (wl.stream_key(5), 4097, 1.0, 1),
                               (0xFFFFFFFF, 1000, 0.5, (1 << 31) - 7), (0, 33, 3.0, 12)]:
        a = wl.normal(key, n, std, "cpu", start)
        b = wl._normal_torch(key, n, std, "cpu", start)
        assert a.dtype == torch.float32 and torch.equal(a, b)
