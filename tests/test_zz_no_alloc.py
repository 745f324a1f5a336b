"""The no-allocation skinny product (nvfp4_gemv_skinny_noalloc).

It serves callers that cannot allocate device memory (a host program without a
device allocator, or a loop that must not call cudaMalloc because it
synchronises the device): its scratch is a fixed array inside the library.
This file is collected last so that, if it fails, a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process.  Each case calls the entry point twice in a row through the C ABI and
checks that both outputs are the same bits as the regular workspace-taking
entry point's (the same kernels run with the same split), and against the
oracle within the accuracy bound the other parity tests use.  The failure path
(a wait that runs out in the array's status word) is read and cleared through
nvfp4_noalloc_status, since the caller never sees the array's address.
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
    # same kernels, shapes and split as the workspace entry point: the same bits
    assert torch.equal(y1, y_ws) and torch.equal(y2, y_ws)
    # the calls left the array's status word clean (and nothing to clear)
    assert g.nvfp4_noalloc_status(clear=False) == (g.NVFP4_OK, 0)
    ref_w = oracle.quantize(w.cpu().numpy())
    rows = np.unique(np.random.default_rng(M).integers(0, M, 64))
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    assert_close(to_np(y1)[:, rows], y_ref, gemv_tol(y_ref, A), f"noalloc M={M} K={K} N={N}")


def test_noalloc_rejects_bad_arguments():
    W = g.nvfp4_quantize(inputs.weights(32, 64, seed=1, device=DEV))
    x = inputs.activations(17, 64, seed=2, device=DEV)
    with pytest.raises(g.NVFP4Error) as e:
        g.nvfp4_gemv_skinny_noalloc(x, W)  # N = 17 is outside 1..16
    assert e.value.status == g.binding.NVFP4_ERR_UNSUPPORTED_SHAPE


def test_noalloc_failure_path_is_reported_and_cleared():
    """A bounded wait that runs out in the array's status word (the self-test:
    it faults nothing) is reported by nvfp4_noalloc_status; clearing it
    zero-fills the array, and the next calls are bit-exact again."""
    M, K, N = 5120, 17408, 4   # a split-K shape: counters in the array are used
    W = g.nvfp4_quantize(inputs.weights(M, K, seed=77, device=DEV))
    x = inputs.activations(N, K, seed=78, device=DEV)
    y_ws = g.nvfp4_gemv_skinny(x, W)
    g.nvfp4_noalloc_selftest_wait_timeout()
    assert g.nvfp4_noalloc_status(clear=False) == (g.NVFP4_ERR_DEVICE_TIMEOUT, 127)
    assert g.nvfp4_noalloc_status(clear=True) == (g.NVFP4_ERR_DEVICE_TIMEOUT, 127)
    assert g.nvfp4_noalloc_status() == (g.NVFP4_OK, 0)
    for _ in range(2):
        assert torch.equal(g.nvfp4_gemv_skinny_noalloc(x, W), y_ws)
    assert g.nvfp4_noalloc_status(clear=False) == (g.NVFP4_OK, 0)
