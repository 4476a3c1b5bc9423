"""nvfp4_gemv_w4a16 on the GPU against the oracle's fp64 GEMV.

Tolerance: max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 per output tensor (the
layer's stated bound; the kernel accumulates in fp32 and rounds to bf16 once).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workload as wl
from harness import tol_ok

pytestmark = pytest.mark.gpu


def _run(nv, N, K, T, kind, seed):
    w = wl.dense_weight_f32(seed, N, K)
    x = wl.activations(seed, T, K)
    W = nv.nvfp4_pack(w.cuda(), kind, check=True)
    y = nv.nvfp4_gemv_w4a16(W, x.cuda())
    torch.cuda.synchronize()
    ref = oracle.gemv(oracle.pack(w, kind), x)
    got = y.float().cpu().numpy().astype(np.float64)
    ok, err, bound = tol_ok(got, ref)
    assert ok, (N, K, T, kind, err, bound)
    # fp32 accumulation + one bf16 rounding: far inside the bound in practice
    assert err <= 2.0 ** -7 * np.abs(ref).max() + 1e-6
    return y


@pytest.mark.parametrize("kind", [1, 0])
def test_gemv_in_proj_qkv_shape(nv, kind):
    """1 token, K=2048 -> N=8192 (FP16 scales, and the E4M3 variant)."""
    _run(nv, 8192, 2048, 1, kind, seed=1)


@pytest.mark.parametrize("T", [2, 3, 8, 9, 17, 64])
def test_gemv_tokens(nv, T):
    _run(nv, 301, 1024, T, 0, seed=T)


@pytest.mark.parametrize("N,K", [(1, 32), (5, 96), (4099, 64), (17, 8192), (64, 4096)])
def test_gemv_ragged_shapes(nv, N, K):
    _run(nv, N, K, 3, 1, seed=N + K)


def test_gemv_dyadic_exact(nv):
    """On-grid weights, power-of-two scales, integer activations: exact sums."""
    rng = np.random.default_rng(3)
    N, K = 40, 256
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, ::16] = 7
    sexp = rng.integers(-2, 3, size=(N, K // 16))
    mags = np.array([oracle.e2m1_decode(int(c)) for c in codes.ravel()]).reshape(N, K)
    W = (mags * np.repeat(2.0 ** sexp, 16, axis=1)).astype(np.float32)
    xi = rng.integers(-4, 5, size=(2, K))
    x = torch.tensor(xi, dtype=torch.bfloat16)
    Wd = nv.nvfp4_pack(torch.from_numpy(W).cuda(), 1, check=True)
    y = nv.nvfp4_gemv_w4a16(Wd, x.cuda()).float().cpu().numpy()
    for t in range(2):
        for n in range(N):
            exact = sum(Fraction(float(W[n, k])) * int(xi[t, k]) for k in range(K))
            # exact fp32 sum, then one bf16 rounding of it
            want = torch.tensor(float(exact), dtype=torch.float32).to(torch.bfloat16).float().item()
            assert y[t, n] == want


def test_gemv_deterministic(nv):
    w = wl.dense_weight_f32(9, 8192, 2048)
    x = wl.activations(9, 4, 2048).cuda()
    W = nv.nvfp4_pack(w.cuda(), 0)
    y0 = nv.nvfp4_gemv_w4a16(W, x)
    for _ in range(9):
        assert torch.equal(nv.nvfp4_gemv_w4a16(W, x), y0)


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_lm_head_vocab(nv, T):
    """The NVFP4 lm_head of Qwen3.6-35B-A3B (lynn-engine tutorials index, Qwen 3.6 config
    block: vocab_size 248320, hidden 2048) as one dense W4A16 GEMV, FP16 block scales
    (the P1 stage's format; a row's bytes depend on that row only, so the oracle packs just
    the rows it checks). 512 rows spread over the vocabulary, the first and the last, are
    compared with the oracle; all rows must be finite."""
    N, K, seed = 248320, 2048, 17
    w = wl.dense_weight_f32(seed, N, K, device="cuda")
    W = nv.nvfp4_pack(w, 1, check=True)
    del w
    x = wl.activations(seed, T, K)
    y = nv.nvfp4_gemv_w4a16(W, x.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 510, replace=False)]))
    key = wl.stream_key(seed, 0, wl.K_DENSE)
    wr = torch.stack([wl.normal(key, K, 0.02, start=int(r) * K) for r in rows])
    ref = oracle.gemv(oracle.pack(wr, 1), x)
    got = y.float().cpu().numpy().astype(np.float64)[:, rows]
    ok, err, bound = tol_ok(got, ref)
    assert ok, (err, bound)
    assert err <= 2.0 ** -7 * np.abs(ref).max() + 1e-6


def test_gemv_lm_head_e4m3_scales(nv):
    """E4M3 block scales at a 32768-row vocabulary slice (the tensor scale depends on the whole
    matrix, so the oracle packs all of it)."""
    _run(nv, 32768, 2048, 1, 0, seed=18)


@pytest.mark.parametrize("kind", [2, 3])
@pytest.mark.parametrize("N,K,T", [(8192, 2048, 1), (301, 1024, 3), (77, 64, 9), (5000, 8192, 2)])
def test_gemv_other_scale_contracts(nv, kind, N, K, T):
    """FP32 per-16 and E8M0 per-32 block scales (README P52, P17/P18): packer bytes and scales
    bit-exact against the oracle's, GEMV within the bar."""
    w = wl.dense_weight_f32(50 + kind, N, K)
    W = nv.nvfp4_pack(w.cuda(), kind, check=True)
    ref_p = oracle.pack(w, kind)
    assert np.array_equal(W.packed.cpu().numpy(), ref_p.packed)
    gs = W.scales.cpu().numpy().view(ref_p.scales.dtype)
    assert np.array_equal(gs, ref_p.scales)
    assert float(W.tensor_scale.cpu()[0]) == ref_p.tensor_scale == 1.0
    x = wl.activations(50 + kind, T, K)
    y = nv.nvfp4_gemv_w4a16(W, x.cuda())
    torch.cuda.synchronize()
    ok, err, bound = tol_ok(y.float().cpu().numpy().astype(np.float64), oracle.gemv(ref_p, x))
    assert ok, (err, bound)


def test_gemv_ue8m0_needs_k_multiple_of_64(nv):
    w = wl.dense_weight_f32(60, 16, 96)
    W = nv.nvfp4_pack(w.cuda(), 3)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.nvfp4_gemv_w4a16(W, wl.activations(60, 1, 96).cuda())
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
