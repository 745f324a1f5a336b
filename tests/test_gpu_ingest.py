"""Ingest on the GPU vs the oracle: the bf16-input quantiser and the import of
block scales from the blocked (128 x 4) layout, both byte-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV
from test_gpu_quantize import assert_bit_exact

pytestmark = pytest.mark.gpu


def bf16_weights(M, K, seed, heavy_tail=False):
    return inputs.weights(M, K, seed=seed, heavy_tail=heavy_tail).to(torch.bfloat16)


def quantize_bf16_both(w_bf16: torch.Tensor):
    W = g.nvfp4_quantize_bf16(w_bf16.to(DEV).contiguous())
    torch.cuda.synchronize()
    ref = oracle.quantize_bf16(inputs.bf16_bits(w_bf16))
    return W, ref


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (17, 272), (100, 4112), (255, 1024), (4096, 4096)])
def test_quantize_bf16_bit_exact(M, K):
    W, ref = quantize_bf16_both(bf16_weights(M, K, seed=M * 7 + K))
    assert_bit_exact(W, ref, f"bf16 {M}x{K}")


def test_quantize_bf16_heavy_tail_and_27b_rows():
    W, ref = quantize_bf16_both(bf16_weights(1024, 5120, seed=5, heavy_tail=True))
    assert_bit_exact(W, ref, "bf16 heavy tail")


def test_quantize_bf16_equals_fp32_quantise_of_same_values():
    w = bf16_weights(2048, 5120, seed=9, heavy_tail=True)
    a = g.nvfp4_quantize_bf16(w.to(DEV))
    b = g.nvfp4_quantize(w.float().to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    assert torch.equal(a.tensor_scale, b.tensor_scale)


def test_quantize_bf16_zero_and_empty():
    W = g.nvfp4_quantize_bf16(torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert W.tensor_scale.item() == 0.0 and not W.codes.any() and not W.scales.any()
    g.nvfp4_quantize_bf16(torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_quantize_bf16(torch.zeros(4, 24, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        g.nvfp4_quantize_bf16(torch.zeros(4, 64, dtype=torch.float32, device=DEV))


@pytest.mark.parametrize("M,K", [(1, 16), (130, 80), (128, 64), (257, 1040), (300, 4000 // 16 * 16),
                                 (17408, 5120), (4096, 12288), (200, 768)])
def test_import_blocked_scales_matches_oracle(M, K):
    rng = np.random.default_rng(M + 3 * K)
    # random bytes everywhere, padding included: the import must ignore padding
    blocked = rng.integers(0, 256, oracle.blocked_scale_bytes(M, K), dtype=np.uint8)
    assert g.nvfp4_blocked_scale_bytes(M, K) == blocked.size
    got = g.nvfp4_import_blocked_scales(torch.from_numpy(blocked).to(DEV), M, K)
    torch.cuda.synchronize()
    ref = oracle.deinterleave_scales(blocked, M, K)
    if not np.array_equal(got.cpu().numpy(), ref):
        bad = np.argwhere(got.cpu().numpy() != ref)[:5]
        raise AssertionError(f"{M}x{K}: scales differ at {bad.tolist()}")


def test_imported_weights_give_the_same_products():
    """A synthetic external checkpoint: quantise, export the scales to the blocked
    layout with the oracle, import on the GPU, run the skinny product with both."""
    M, K = 1000, 2064
    w = bf16_weights(M, K, seed=12)
    W = g.nvfp4_quantize_bf16(w.to(DEV))
    torch.cuda.synchronize()
    blocked = oracle.interleave_scales(W.scales.cpu().numpy())
    scales = g.nvfp4_import_blocked_scales(torch.from_numpy(blocked).to(DEV), M, K)
    torch.cuda.synchronize()
    assert torch.equal(scales, W.scales)
    Wi = g.NVFP4Weight(W.codes, scales, W.tensor_scale)
    x = inputs.activations(3, K, seed=4).to(DEV)
    y0 = g.nvfp4_gemv_skinny(x, W)
    y1 = g.nvfp4_gemv_skinny(x, Wi)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_import_rejects_bad_arguments():
    b = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_import_blocked_scales(b, 16, 24)
    with pytest.raises(ValueError):
        g.nvfp4_import_blocked_scales(b, 1024, 4096)  # buffer too small
    out = g.nvfp4_import_blocked_scales(b, 0, 64)
    assert out.shape == (0, 4)
