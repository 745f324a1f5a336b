"""Device-side failure reporting (nvfp4_device_status, nvfp4_selftest_wait_timeout).

Every wait inside the tensor-core kernels is bounded: a pipeline that stops
making progress gives up after 2 s, stores a code in the status word of the
call's workspace and returns, so the GPU never hangs.  These tests check that
ordinary product calls leave the word clean, that a wait which runs out (the
self-test waits on a barrier that nothing completes, which faults nothing) is
reported to the host, that no later kernel hides it, and that the context
still computes correct products afterwards.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, to_np

pytestmark = pytest.mark.gpu


def _skinny_ws(M, K):
    need = max(g.nvfp4_workspace_bytes(g.NVFP4_OP_GATEUP_SWIGLU, 16, M, K),
               g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, 16, M, K))
    return torch.zeros(need, dtype=torch.uint8, device=DEV)


def _check_rows(y, x, ref_w, what):
    rows = np.arange(0, y.shape[1], 7)
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    assert_close(to_np(y)[:, rows], y_ref, gemv_tol(y_ref, A), what)


def test_status_clean_after_every_kind_of_product():
    M, K = 1024, 4096  # K % 256 == 0: the tensor-core skinny kernel and the TMA-fed prefill
    W = g.nvfp4_quantize(inputs.weights(M, K, seed=5, device=DEV))
    Wu = g.nvfp4_quantize(inputs.weights(M, K, seed=6, device=DEV))
    F = g.nvfp4_fp6_quantize(inputs.weights(M, K, seed=7, device=DEV))
    ws = _skinny_ws(M, K)
    for N in (1, 4, 16):
        x = inputs.activations(N, K, seed=N, device=DEV)
        g.nvfp4_gemv_skinny(x, W, workspace=ws)
        g.nvfp4_gateup_swiglu(x, W, Wu, workspace=ws)
        g.nvfp4_fp6_gemm(x, F, workspace=ws)
    assert g.nvfp4_device_status(ws) == (g.NVFP4_OK, 0)
    # one workspace for every prefill call below: the largest they need (a
    # single NVFP4 matrix may split K, which needs partial slots)
    pws = torch.zeros(max(g.nvfp4_workspace_bytes(op, N, M, K) for N in (40, 600)
                          for op in (g.NVFP4_OP_GEMM_PREFILL, g.NVFP4_OP_GATEUP_SWIGLU, g.NVFP4_OP_FP6_GEMM)),
                      dtype=torch.uint8, device=DEV)
    for N in (40, 600):
        x = inputs.activations(N, K, seed=N, device=DEV)
        g.nvfp4_gemm_prefill(x, W, workspace=pws)
        g.nvfp4_gateup_swiglu(x, W, Wu, workspace=pws)
        g.nvfp4_fp6_gemm(x, F, workspace=pws)
    assert g.nvfp4_device_status(pws) == (g.NVFP4_OK, 0)


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    M, K, N = 512, 4096, 4
    w = inputs.weights(M, K, seed=11, device=DEV)
    x = inputs.activations(N, K, seed=12, device=DEV)
    W = g.nvfp4_quantize(w)
    ref_w = oracle.quantize(w.cpu().numpy())
    ws = _skinny_ws(M, K)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.nvfp4_selftest_wait_timeout(ws)
    st, code = g.nvfp4_device_status(ws, clear=False)  # synchronises: the wait has given up
    waited = time.perf_counter() - t0
    assert (st, code) == (g.NVFP4_ERR_DEVICE_TIMEOUT, 127)
    assert 1.5 < waited < 60.0, f"the bounded wait took {waited:.2f} s"

    # No kernel clears the word: products on the same workspace (with and
    # without the skinny prep kernel) leave the failure visible, and compute
    # correct results.
    y4 = g.nvfp4_gemv_skinny(x, W, workspace=ws)
    y1 = g.nvfp4_gemv_skinny(x[:1].contiguous(), W, workspace=ws)
    assert g.nvfp4_device_status(ws, clear=True) == (g.NVFP4_ERR_DEVICE_TIMEOUT, 127)
    assert g.nvfp4_device_status(ws) == (g.NVFP4_OK, 0)
    _check_rows(y4, x, ref_w, "skinny N=4 after a reported timeout")
    _check_rows(y1, x[:1], ref_w, "skinny N=1 after a reported timeout")

    # a prefill workspace (status word, and split-mode partial slots) and the
    # prefill kernel afterwards
    pws = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, 300, M, K), dtype=torch.uint8,
                      device=DEV)
    g.nvfp4_selftest_wait_timeout(pws)
    xp = inputs.activations(300, K, seed=13, device=DEV)
    yp = g.nvfp4_gemm_prefill(xp, W, workspace=pws)
    assert g.nvfp4_device_status(pws) == (g.NVFP4_ERR_DEVICE_TIMEOUT, 127)
    assert g.nvfp4_device_status(pws) == (g.NVFP4_OK, 0)
    _check_rows(yp, xp, ref_w, "prefill after a reported timeout")
