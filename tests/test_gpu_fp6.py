"""FP6 E2M3 block-scaled weights on the GPU vs the oracle: the quantiser
byte-exact, the products (skinny N <= 16 and tensor-core prefill N > 16, plain
and gate/up + SwiGLU) within the library's accuracy bound."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, swiglu_tol, to_np

pytestmark = pytest.mark.gpu


def quantize_both(w_cpu: torch.Tensor):
    W = g.nvfp4_fp6_quantize(w_cpu.to(DEV).contiguous())
    torch.cuda.synchronize()
    return W, oracle.fp6_quantize(w_cpu.numpy())


def assert_bytes_equal(W, ref, what):
    c, s = ref
    gc, gs = W.codes.cpu().numpy(), W.scales.cpu().numpy()
    if not np.array_equal(gs, s):
        bad = np.argwhere(gs != s)[:5]
        raise AssertionError(f"{what}: scales differ at {bad.tolist()}")
    if not np.array_equal(gc, c):
        bad = np.argwhere(gc != c)[:5]
        raise AssertionError(f"{what}: codes differ at {bad.tolist()}")


@pytest.mark.parametrize("M,K", [(1, 128), (3, 256), (17, 384), (100, 4096), (255, 1024), (4096, 4096)])
def test_quantize_bit_exact(M, K):
    W, ref = quantize_both(inputs.weights(M, K, seed=M + 5 * K))
    assert_bytes_equal(W, ref, f"fp6 {M}x{K}")


def test_quantize_heavy_tail_and_extreme_ranges():
    w = inputs.weights(64, 1024, seed=41, heavy_tail=True)
    w[1] *= 1e30        # scale bytes above 128: the two-step multiplier
    w[2] *= 1e-36       # tiny scales
    w[3] = 0.0          # zero blocks
    w[4, :128] = -0.0
    w[5] *= 1e-7
    w[5, 128:256] = 0.0
    w[5, 200] = 2.0 ** -140  # block 1 of row 5: a subnormal amax
    W, ref = quantize_both(w)
    assert_bytes_equal(W, ref, "extreme")
    s = W.scales.cpu().numpy()
    assert s.max() > 128 and s.min() == 0


def test_quantize_bf16_bit_exact_and_same_as_fp32():
    w = inputs.weights(777, 2048, seed=43, heavy_tail=True).to(torch.bfloat16)
    A = g.nvfp4_fp6_quantize_bf16(w.to(DEV))
    B = g.nvfp4_fp6_quantize(w.float().to(DEV))
    torch.cuda.synchronize()
    assert_bytes_equal(A, oracle.fp6_quantize_bf16(inputs.bf16_bits(w)), "fp6 bf16")
    assert torch.equal(A.codes, B.codes) and torch.equal(A.scales, B.scales)


def test_quantize_rejects_bad_shapes():
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_fp6_quantize(torch.zeros(4, 192, device=DEV))
    with pytest.raises(ValueError):
        g.nvfp4_fp6_quantize(torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("N", [1, 3, 8, 9, 16, 17, 100, 300])
@pytest.mark.parametrize("M,K", [(1000, 2048), (129, 384), (4096, 1024)])
def test_gemm_vs_oracle(N, M, K):
    w = inputs.weights(M, K, seed=M + N)
    x = inputs.activations(N, K, seed=N + K, outlier_rows=True)
    W = g.nvfp4_fp6_quantize(w.to(DEV))
    y = g.nvfp4_fp6_gemm(x.to(DEV), W)
    torch.cuda.synchronize()
    codes, scales = oracle.fp6_quantize(w.numpy())
    rows = np.unique(np.r_[0, M - 1, np.random.default_rng(N).integers(0, M, 200)])
    y_ref, A = oracle.fp6_gemv(bf16_bits(x), codes, scales, rows=rows)
    assert_close(to_np(y)[:, rows], y_ref, gemv_tol(y_ref, A), f"fp6 N={N} M={M} K={K}")


@pytest.mark.parametrize("N", [4, 600])
def test_gemm_bf16_output_and_wide_scales(N):
    M, K = 384, 1024
    w = inputs.weights(M, K, seed=51)
    w[0:64] *= 1e30
    w[64:128] *= 1e-30
    x = inputs.activations(N, K, seed=52)
    W = g.nvfp4_fp6_quantize(w.to(DEV))
    codes, scales = oracle.fp6_quantize(w.numpy())
    assert np.array_equal(W.scales.cpu().numpy(), scales)
    y_ref, A = oracle.fp6_gemv(bf16_bits(x), codes, scales)
    for dt in (torch.float32, torch.bfloat16):
        y = g.nvfp4_fp6_gemm(x.to(DEV), W, out_dtype=dt)
        torch.cuda.synchronize()
        assert_close(to_np(y), y_ref, gemv_tol(y_ref, A, dt), f"fp6 N={N} {dt}")


@pytest.mark.parametrize("N", [1, 5, 16, 64, 300])
def test_gateup_swiglu_vs_oracle(N):
    M, K = 640, 2048
    wg, wu = inputs.weights(M, K, seed=61), inputs.weights(M, K, seed=62)
    x = inputs.activations(N, K, seed=63)
    Wg, Wu = g.nvfp4_fp6_quantize(wg.to(DEV)), g.nvfp4_fp6_quantize(wu.to(DEV))
    h = g.nvfp4_fp6_gateup_swiglu(x.to(DEV), Wg, Wu)
    torch.cuda.synchronize()
    gate, up = oracle.fp6_quantize(wg.numpy()), oracle.fp6_quantize(wu.numpy())
    rows = np.unique(np.r_[0, M - 1, np.random.default_rng(N).integers(0, M, 150)])
    h_ref, g_ref, u_ref, Ag, Au = oracle.fp6_swiglu(bf16_bits(x), gate, up, rows=rows)
    assert_close(to_np(h)[:, rows], h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au), f"fp6 swiglu N={N}")


def test_27b_shapes_sampled():
    """Full-size 27B-class down projection (5120 x 17408) and gate/up
    (17408 x 5120) at decode and prefill widths, checked on sampled rows."""
    shapes = inputs.LAYER_27B.shapes()
    Md, Kd = shapes["down"]
    wd = inputs.weights(Md, Kd, seed=inputs.matrix_seed("down"), device=DEV)
    Wd = g.nvfp4_fp6_quantize(wd)
    cd, sd = oracle.fp6_quantize(wd.cpu().numpy())
    assert np.array_equal(Wd.scales.cpu().numpy(), sd) and np.array_equal(Wd.codes.cpu().numpy(), cd)
    rng = np.random.default_rng(3)
    for N in (1, 16, 512):
        x = inputs.activations(N, Kd, seed=N, device=DEV)
        y = g.nvfp4_fp6_gemm(x, Wd)
        torch.cuda.synchronize()
        rows = np.unique(rng.integers(0, Md, 48))
        toks = np.unique(rng.integers(0, N, 8))
        y_ref, A = oracle.fp6_gemv(bf16_bits(x.cpu()), cd, sd, rows=rows, tokens=toks)
        assert_close(to_np(y)[np.ix_(toks, rows)], y_ref, gemv_tol(y_ref, A), f"fp6 down N={N}")
    Mg, Kg = shapes["gate"]
    wg = inputs.weights(Mg, Kg, seed=inputs.matrix_seed("gate"), device=DEV)
    wu = inputs.weights(Mg, Kg, seed=inputs.matrix_seed("up"), device=DEV)
    Wg, Wu = g.nvfp4_fp6_quantize(wg), g.nvfp4_fp6_quantize(wu)
    gate, up = oracle.fp6_quantize(wg.cpu().numpy()), oracle.fp6_quantize(wu.cpu().numpy())
    for N in (1, 9, 600):
        x = inputs.activations(N, Kg, seed=N + 1, device=DEV)
        h = g.nvfp4_fp6_gateup_swiglu(x, Wg, Wu)
        torch.cuda.synchronize()
        rows = np.unique(rng.integers(0, Mg, 48))
        toks = np.unique(rng.integers(0, N, 6))
        h_ref, g_ref, u_ref, Ag, Au = oracle.fp6_swiglu(bf16_bits(x.cpu()), gate, up, rows=rows, tokens=toks)
        assert_close(to_np(h)[np.ix_(toks, rows)], h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au),
                     f"fp6 gateup N={N}")


def test_deterministic_and_token_independent():
    M, K = 2048, 4096
    W = g.nvfp4_fp6_quantize(inputs.weights(M, K, seed=71, device=DEV))
    x = inputs.activations(9, K, seed=72, device=DEV)
    y9 = g.nvfp4_fp6_gemm(x, W)
    y9b = g.nvfp4_fp6_gemm(x, W)
    y1 = g.nvfp4_fp6_gemm(x[4:5].contiguous(), W)
    torch.cuda.synchronize()
    assert torch.equal(y9, y9b)
    assert torch.equal(y9[4], y1[0])


def test_empty_and_zero_k():
    W = g.nvfp4_fp6_quantize(torch.zeros(8, 128, device=DEV))
    y = g.nvfp4_fp6_gemm(torch.zeros(0, 128, dtype=torch.bfloat16, device=DEV), W)
    assert y.shape == (0, 8)
    W0 = g.FP6Weight(torch.zeros(8, 0, dtype=torch.uint8, device=DEV), torch.zeros(8, 0, dtype=torch.uint8,
                                                                                    device=DEV))
    y = g.nvfp4_fp6_gemm(torch.zeros(3, 0, dtype=torch.bfloat16, device=DEV), W0)
    torch.cuda.synchronize()
    assert y.shape == (3, 8) and not y.any()
