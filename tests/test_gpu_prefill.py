"""Prefill product (N > 16) through the C ABI vs the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, swiglu_tol, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,M,K", [(17, 48, 272), (40, 130, 512), (200, 256, 1024), (300, 500, 2064)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_small(N, M, K, out_dtype):
    w = inputs.weights(M, K, seed=N + M)
    x = inputs.activations(N, K, seed=N + K)
    W = g.nvfp4_quantize(w.to(DEV))
    y = g.nvfp4_gemm_prefill(x.to(DEV), W, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref_w = oracle.quantize(w.numpy())
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w)
    assert_close(to_np(y), y_ref, gemv_tol(y_ref, A, out_dtype), f"prefill N={N} M={M} K={K}")


def test_prefill_forwards_small_n():
    w = inputs.weights(64, 256, seed=3)
    x = inputs.activations(5, 256, seed=4)
    W = g.nvfp4_quantize(w.to(DEV))
    y = g.nvfp4_gemm_prefill(x.to(DEV), W)
    y2 = g.nvfp4_gemv_skinny(x.to(DEV), W)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("N", [64, 300])
def test_gateup_prefill_small(N):
    M, K = 160, 1024
    wg, wu = inputs.weights(M, K, seed=7), inputs.weights(M, K, seed=8)
    x = inputs.activations(N, K, seed=9)
    Wg, Wu = g.nvfp4_quantize(wg.to(DEV)), g.nvfp4_quantize(wu.to(DEV))
    h = g.nvfp4_gateup_swiglu(x.to(DEV), Wg, Wu)
    torch.cuda.synchronize()
    h_ref, g_ref, u_ref, Ag, Au = oracle.swiglu(bf16_bits(x), oracle.quantize(wg.numpy()),
                                                oracle.quantize(wu.numpy()))
    assert_close(to_np(h), h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au), f"gate/up prefill N={N}")


def test_prefill_deterministic():
    w = inputs.weights(256, 1024, seed=1).to(DEV)
    x = inputs.activations(100, 1024, seed=2).to(DEV)
    W = g.nvfp4_quantize(w)
    a, b = g.nvfp4_gemm_prefill(x, W), g.nvfp4_gemm_prefill(x, W)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
