"""Pins for the oracle's number formats and packer.

Each check ties the oracle to something outside itself: the printed E2M1
magnitude set, IEEE/OCP conversions done by numpy and torch, brute-force
nearest-value search on tiny inputs, exact on-grid round trips, and the packed
size printed for the P1 projection.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table(orc):
    # NVFP4 element: 4-bit E2M1, magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign
    for c in range(16):
        v = orc.e2m1_decode(c)
        mag = E2M1_MAGS[c & 7]
        assert v == (-mag if c & 8 else mag)
        assert np.signbit(v) == bool(c & 8)


def test_e2m1_roundtrip_every_code(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_decode(c)) == c


@pytest.mark.parametrize("v,want", [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0),
                                    (2.5, 2.0), (3.5, 4.0), (5.0, 4.0), (5.0001, 6.0),
                                    (7.0, 6.0), (1e30, 6.0), (0.2499, 0.0), (0.2501, 0.5)])
def test_e2m1_midpoints_ties_to_even(orc, v, want):
    for s in (1.0, -1.0):
        code = orc.e2m1_encode(s * v)
        assert orc.e2m1_decode(code) == s * want
        assert bool(code & 8) == (s < 0)


def test_e2m1_encode_is_nearest_brute_force(orc):
    grid = np.array(E2M1_MAGS)
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), rng.uniform(-1, 1, 2000)]).astype(np.float32)
    for v in vals:
        a = min(abs(float(v)), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        # a tie picks the code with an even (zero) mantissa bit
        idx = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        code = orc.e2m1_encode(float(v))
        assert (code & 7) == idx, (v, code, idx)


def test_e4m3_decode_matches_torch_all_bytes(orc):
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for i in range(256):
        got = orc.e4m3_decode(i)
        if np.isnan(ref[i]):
            assert np.isnan(got)
        else:
            assert got == ref[i], i


def test_e4m3_roundtrip_and_encode_matches_torch(orc):
    for i in range(256):
        if i & 0x7F == 0x7F:
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(i)) == i
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-0.03, 0.03, 3000),
                           np.exp(rng.uniform(-14, 6, 3000)) * rng.choice([-1, 1], 3000)])
    vals = vals.astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in vals])
    assert np.array_equal(got, ref)


def test_e4m3_saturates(orc):
    assert orc.e4m3_encode(449.0) == 0x7E
    assert orc.e4m3_encode(1e20) == 0x7E
    assert orc.e4m3_encode(-1e20) == 0xFE
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9


def test_fp16_matches_numpy(orc):
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-5, 3000),
                           np.exp(rng.uniform(-20, 11, 3000))]).astype(np.float32)
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.fp16_encode(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    for bits in range(0, 65536, 7):
        r = np.array([bits], np.uint16).view(np.float16)[0]
        g = orc.fp16_decode(bits)
        if np.isnan(r):
            assert np.isnan(g)
        else:
            assert g == float(r)
    assert orc.fp16_encode(1e6) == 0x7BFF


def _e4m3_values():
    return [(b, torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).item())
            for b in range(1, 0x7F)]


@pytest.mark.parametrize("kind", [0, 1])
def test_pack_on_grid_roundtrip_exact(orc, kind):
    """W built exactly as code * scale * tensor_scale packs back to the same bytes."""
    rng = np.random.default_rng(4)
    N, K = 12, 64
    nb = K // 16
    codes = rng.integers(0, 16, size=(N, K))
    # every block holds one +-6 so its amax is 6 * scale
    codes[:, ::16] = rng.choice([7, 15], size=(N, nb))
    if kind == 0:
        s_t = 2.0 ** -10
        table = _e4m3_values()
        sel = rng.integers(0, len(table), size=(N, nb))
        sbytes = np.array([[table[s][0] for s in row] for row in sel], np.uint8)
        sbytes[0, 0] = 0x7E           # one block at 448 fixes amax_t = 6*448*s_t
        svals = np.array([[orc.e4m3_decode(int(b)) for b in row] for row in sbytes])
    else:
        s_t = 1.0
        sbits = rng.integers(0x0400, 0x5000, size=(N, nb)).astype(np.uint16)  # normal fp16
        sbytes = sbits
        svals = sbits.view(np.float16).astype(np.float64)
    mags = np.array([orc.e2m1_decode(int(c)) for c in codes.ravel()]).reshape(N, K)
    W = mags * np.repeat(svals, 16, axis=1) * s_t
    Wf = W.astype(np.float32)
    assert np.array_equal(Wf.astype(np.float64), W)           # exactly representable
    p = orc.pack(Wf, kind)
    assert p.tensor_scale == s_t
    assert np.array_equal(p.scales, sbytes)
    # element 2j -> low nibble, 2j+1 -> high nibble
    want_bytes = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    # signed zeros keep their sign bit, so every byte matches
    assert np.array_equal(p.packed, want_bytes)
    assert np.array_equal(orc.dequant(p), W)


@pytest.mark.parametrize("kind", [0, 1])
def test_pack_random_codes_are_nearest(orc, kind):
    """Brute force: every code is the nearest grid point to w / (decoded block scale)."""
    w = wl.normal(wl.stream_key(5), 6 * 96, 0.02).view(6, 96).numpy()
    p = orc.pack(w, kind)
    nb = 96 // 16
    dec_scale = np.zeros((6, nb))
    for n in range(6):
        for b in range(nb):
            sv = orc.e4m3_decode(int(p.scales[n, b])) if kind == 0 else orc.fp16_decode(int(p.scales[n, b]))
            dec_scale[n, b] = np.float32(np.float32(sv) * np.float32(p.tensor_scale))
    grid = np.array(E2M1_MAGS)
    for n in range(6):
        for k in range(96):
            byte = int(p.packed[n, k // 2])
            code = (byte >> 4) if k & 1 else (byte & 15)
            d = dec_scale[n, k // 16]
            u = np.float32(np.float32(w[n, k]) / np.float32(d))
            dist = np.abs(grid - min(abs(float(u)), 6.0))
            assert dist[code & 7] == dist.min()
            assert bool(code & 8) == bool(np.signbit(w[n, k]))


def test_pack_scale_tracks_block_amax(orc):
    w = wl.normal(wl.stream_key(6), 64 * 256, 0.02).view(64, 256).numpy()
    p = orc.pack(w, 0)
    assert p.tensor_scale == np.float32(np.abs(w).max()) / np.float32(2688.0)
    amax_b = np.abs(w.reshape(64, 16, 16)).max(axis=2)
    dec = np.array([[orc.e4m3_decode(int(b)) for b in row] for row in p.scales]) * p.tensor_scale
    # E4M3 keeps 3 mantissa bits: relative rounding error of the scale <= 2^-4 (normal range)
    rel = np.abs(dec - amax_b / 6) / (amax_b / 6)
    assert rel.max() <= 2.0 ** -4 + 1e-6
    # dequantisation error bounded by one decoded scale per element; overall rel. error ~ 10 %
    deq = orc.dequant(p)
    assert np.all(np.abs(deq - w) <= np.repeat(dec, 16, axis=1) * 1.0 + 1e-12)
    assert np.linalg.norm(deq - w) / np.linalg.norm(w) < 0.15


def test_pack_zero_and_nonfinite(orc):
    z = np.zeros((2, 32), np.float32)
    p = orc.pack(z, 0)
    assert p.tensor_scale == 1.0 and not p.scales.any() and not p.packed.any()
    bad = z.copy()
    bad[1, 3] = np.nan
    with pytest.raises(ValueError):
        orc.pack(bad, 0)
    bad[1, 3] = np.inf
    with pytest.raises(ValueError):
        orc.pack(bad, 1)


def test_p1_packed_footprint(orc):
    """Packed E2M1 + FP16 per-16 scale for the [8192, 2048] projection: 10.00 MiB vs 32.00 MiB bf16."""
    g = json.load(open(os.path.join(GOLDEN, "p1_packed_footprint.json")))
    N, K = g["N"], g["K"]
    w = np.zeros((N, 32), np.float32)   # only the byte layout per element matters here
    p = orc.pack(w, 1)
    bytes_per_elem = (p.packed.nbytes + p.scales.nbytes) / (N * 32)
    packed_mib = bytes_per_elem * N * K / 2 ** 20
    assert packed_mib == pytest.approx(g["packed_mib"], abs=0.005)
    assert 2 * N * K / 2 ** 20 == pytest.approx(g["bf16_mib"], abs=0.005)


# ------------------------------------------------------------------ other scale contracts
# README P52 (Lynn-native fp32 scale per 16 elements) and P17/P18 (the e8m0 scale per 32
# elements of the vendor MX layout, neutral byte 127).

def test_e8m0_decode_all_bytes(orc):
    for b in range(255):
        assert orc.e8m0_decode(b) == 2.0 ** (b - 127)
    assert np.isnan(orc.e8m0_decode(255))
    assert orc.e8m0_decode(127) == 1.0


def test_fp32_scale_on_grid_round_trip(orc):
    """codes x an fp32 block scale whose block holds a +-6: the packer recovers both exactly."""
    rng = np.random.default_rng(11)
    N, K = 6, 64
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, ::16] = 7                                   # a 6 in every block
    s = (rng.integers(1, 2 ** 10, size=(N, K // 16)) * 2.0 ** rng.integers(-20, 5, size=(N, K // 16)))
    s = s.astype(np.float32)
    mags = np.array([orc.e2m1_decode(int(c)) for c in codes.ravel()]).reshape(N, K)
    W = (mags * np.repeat(s.astype(np.float64), 16, axis=1)).astype(np.float32)
    p = orc.pack(W, orc.SCALE_FP32)
    assert p.tensor_scale == 1.0 and p.scales.dtype == np.float32
    assert np.array_equal(p.scales, s)
    got = np.empty((N, K), np.int64)
    got[:, 0::2] = p.packed & 15
    got[:, 1::2] = p.packed >> 4
    zero = mags == 0
    assert np.array_equal(got[~zero], codes[~zero])
    assert np.array_equal(orc.dequant(p), W.astype(np.float64))


def test_ue8m0_scale_on_grid_round_trip(orc):
    """codes x 2^e per 32-element block whose largest magnitude is 4 or 6: the scale byte is
    e + 127 (floor(log2 amax) - 2 = e) and every code comes back."""
    rng = np.random.default_rng(12)
    N, K = 5, 96
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, ::32] = rng.choice([6, 7, 14, 15], size=(N, K // 32))   # largest magnitude 4 or 6
    codes[:, 1::32] = 6
    e = rng.integers(-30, 20, size=(N, K // 32))
    mags = np.array([orc.e2m1_decode(int(c)) for c in codes.ravel()]).reshape(N, K)
    W = (mags * np.repeat(2.0 ** e, 32, axis=1)).astype(np.float32)
    p = orc.pack(W, orc.SCALE_UE8M0)
    assert p.tensor_scale == 1.0 and p.scales.shape == (N, K // 32)
    assert np.array_equal(p.scales.astype(np.int64), e + 127)
    got = np.empty((N, K), np.int64)
    got[:, 0::2] = p.packed & 15
    got[:, 1::2] = p.packed >> 4
    zero = mags == 0
    assert np.array_equal(got[~zero], codes[~zero])
    assert np.array_equal(orc.dequant(p), W.astype(np.float64))


@pytest.mark.parametrize("kind", [2, 3])
def test_new_kinds_codes_are_nearest(orc, kind):
    """Random matrices: every code is the E2M1 point nearest to w / decoded block scale (ties
    to the even code), and for UE8M0 the block's amax / scale lies in [4, 8)."""
    B = 32 if kind == 3 else 16
    w = wl.normal(wl.stream_key(13, kind), 20 * 128, 0.3).view(20, 128).numpy()
    p = orc.pack(w, kind)
    grid = np.array([orc.e2m1_decode(c) for c in range(8)])
    sc = p.scales.astype(np.float64) if kind == 2 else 2.0 ** (p.scales.astype(np.float64) - 127)
    full = np.repeat(sc, B, axis=1)
    u = np.abs(w.astype(np.float64)) / full
    codes = np.empty(w.shape, np.int64)
    codes[:, 0::2] = p.packed & 15
    codes[:, 1::2] = p.packed >> 4
    for (n, k), uv in np.ndenumerate(u):
        d = np.abs(grid - min(uv, 6.0))
        best = np.flatnonzero(d == d.min())
        m = codes[n, k] & 7
        assert m in best, (n, k, uv, m)
        if len(best) > 1:
            assert m % 2 == 0
    if kind == 3:
        amax = np.abs(w).reshape(20, 128 // 32, 32).max(axis=2)
        ratio = amax / sc
        assert np.all((ratio >= 4) & (ratio < 8))
