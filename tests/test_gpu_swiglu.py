"""Fused gate/up + SwiGLU through the C ABI vs the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, swiglu_tol, to_np

pytestmark = pytest.mark.gpu


def run(M, K, N, seed=0, out_dtype=torch.float32, rows=None, device_gen=False, heavy=False, outliers=False):
    dev = DEV if device_gen else "cpu"
    wg = inputs.weights(M, K, seed=seed, heavy_tail=heavy, device=dev)
    wu = inputs.weights(M, K, seed=seed + 100, heavy_tail=heavy, device=dev)
    x = inputs.activations(N, K, seed=seed + 1, outlier_rows=outliers, device=dev)
    Wg, Wu = g.nvfp4_quantize(wg.to(DEV)), g.nvfp4_quantize(wu.to(DEV))
    h = g.nvfp4_gateup_swiglu(x.to(DEV), Wg, Wu, out_dtype=out_dtype)
    torch.cuda.synchronize()
    gref = oracle.quantize(wg.cpu().numpy())
    uref = oracle.quantize(wu.cpu().numpy())
    h_ref, g_ref, u_ref, Ag, Au = oracle.swiglu(bf16_bits(x), gref, uref, rows=rows)
    got = to_np(h) if rows is None else to_np(h)[:, rows]
    assert_close(got, h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au, out_dtype), f"swiglu M={M} K={K} N={N}")
    return h


@pytest.mark.parametrize("N", [1, 4, 9, 16])
@pytest.mark.parametrize("M,K", [(16, 64), (100, 1024), (333, 4112)])
def test_small(M, K, N):
    run(M, K, N, seed=M + K)


def test_bf16_output():
    run(200, 2048, 3, seed=5, out_dtype=torch.bfloat16)


def test_9b_gate_up_n1_sampled():
    M, K = inputs.LAYER_9B.shapes()["gate"]
    rows = np.unique(np.random.default_rng(1).integers(0, M, 48))
    run(M, K, 1, seed=200, rows=rows, device_gen=True)


@pytest.mark.parametrize("N", [4, 16])
def test_27b_gate_up_sampled(N):
    M, K = inputs.LAYER_27B.shapes()["gate"]
    rows = np.unique(np.random.default_rng(N).integers(0, M, 40))
    run(M, K, N, seed=200, rows=rows, device_gen=True, heavy=(N == 16), outliers=(N == 16))


def test_cross_n_identity():
    wg = inputs.weights(256, 2048, seed=1).to(DEV)
    wu = inputs.weights(256, 2048, seed=2).to(DEV)
    Wg, Wu = g.nvfp4_quantize(wg), g.nvfp4_quantize(wu)
    x = inputs.activations(16, 2048, seed=3).to(DEV)
    h = g.nvfp4_gateup_swiglu(x, Wg, Wu)
    h1 = g.nvfp4_gateup_swiglu(x[5:6].contiguous(), Wg, Wu)
    torch.cuda.synchronize()
    assert torch.equal(h[5], h1[0])
