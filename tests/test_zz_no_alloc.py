"""The no-allocation skinny product (nvfp4_gemv_skinny_noalloc).

It serves callers that cannot allocate device memory (a host program without a
device allocator, or a loop that must not call cudaMalloc because it
synchronises the device): its scratch is a fixed array inside the library.
This file is collected last so that, if it fails, a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process.  Each case calls the entry point twice in a row through the C ABI and
checks both outputs against the regular workspace-taking entry point, within
the accuracy bound the other parity tests use.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N", [(4096, 4096, 1), (1000, 5120, 16), (333, 4112, 4), (17408, 5120, 4)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(M, K, N):
    w = inputs.weights(M, K, seed=M + K, device=DEV)
    x = inputs.activations(N, K, seed=N, device=DEV)
    W = g.nvfp4_quantize(w)
    y_ws = g.nvfp4_gemv_skinny(x, W)
    y1 = g.nvfp4_gemv_skinny_noalloc(x, W)
    y2 = g.nvfp4_gemv_skinny_noalloc(x, W)
    torch.cuda.synchronize()
    ref_w = oracle.quantize(w.cpu().numpy())
    rows = np.unique(np.random.default_rng(M).integers(0, M, 64))
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    tol = gemv_tol(y_ref, A)
    base = to_np(y_ws)
    for y in (y1, y2):
        got = to_np(y)
        # within the accuracy bound of the regular entry point's result, everywhere
        assert (np.abs(got - base) <= 2e-5 * np.abs(base) + 1e-6).all()
        # and within the oracle bound on the sampled rows
        assert_close(got[:, rows], y_ref, tol, f"noalloc M={M} K={K} N={N}")


def test_noalloc_rejects_bad_arguments():
    W = g.nvfp4_quantize(inputs.weights(32, 64, seed=1, device=DEV))
    x = inputs.activations(17, 64, seed=2, device=DEV)
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_gemv_skinny_noalloc(x, W)  # N = 17 is outside 1..16
