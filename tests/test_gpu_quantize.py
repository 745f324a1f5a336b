"""GPU quantiser vs the oracle: codes, scales and tensor scale bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV
from test_oracle_pins import read_golden_block, rounding_order_matrix

pytestmark = pytest.mark.gpu


def quantize_both(w_cpu: torch.Tensor):
    W = g.nvfp4_quantize(w_cpu.to(DEV).contiguous())
    torch.cuda.synchronize()
    c, s, ts = oracle.quantize(w_cpu.numpy())
    return W, (c, s, ts)


def assert_bit_exact(W, ref, what=""):
    c, s, ts = ref
    gc, gs, gt = W.codes.cpu().numpy(), W.scales.cpu().numpy(), W.tensor_scale.cpu().numpy()[0]
    assert gt.view(np.uint32) == np.float32(ts).view(np.uint32), f"{what}: tensor scale {gt} vs {ts}"
    if not np.array_equal(gs, s):
        bad = np.argwhere(gs != s)[:5]
        raise AssertionError(f"{what}: scales differ at {bad.tolist()}: {gs[tuple(bad.T)]} vs {s[tuple(bad.T)]}")
    if not np.array_equal(gc, c):
        bad = np.argwhere(gc != c)[:5]
        raise AssertionError(f"{what}: codes differ at {bad.tolist()}: {gc[tuple(bad.T)]} vs {c[tuple(bad.T)]}")


def test_hand_block():
    w, sb, codes = read_golden_block()
    W, ref = quantize_both(torch.from_numpy(w.reshape(1, 16)))
    assert_bit_exact(W, ref, "hand block")
    got = []
    for byte in W.codes.cpu().numpy()[0]:
        got += [int(byte) & 0xF, int(byte) >> 4]
    assert got == codes and W.scales.cpu().item() == sb


def test_single_matrix_4096():
    w = inputs.weights(4096, 4096, seed=0)
    W, ref = quantize_both(w)
    assert_bit_exact(W, ref, "4096x4096")


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (17, 272), (100, 4112), (255, 1024)])
def test_ragged_shapes(M, K):
    W, ref = quantize_both(inputs.weights(M, K, seed=M + K))
    assert_bit_exact(W, ref, f"{M}x{K}")


def test_heavy_tailed_blocks():
    W, ref = quantize_both(inputs.weights(512, 5120, seed=300, heavy_tail=True))
    assert_bit_exact(W, ref, "heavy tail")


def test_rounding_order_sensitive_blocks():
    w, extra = rounding_order_matrix()
    W, ref = quantize_both(torch.from_numpy(w))
    assert_bit_exact(W, ref, "rounding order")


def test_extreme_ranges():
    rng = np.random.default_rng(0)
    cases = {
        "zeros": np.zeros((4, 64), np.float32),
        "tiny_blocks": (rng.standard_normal((8, 64)) * np.logspace(-12, 0, 8)[:, None]).astype(np.float32),
        "huge": (rng.standard_normal((4, 64)) * 1e30).astype(np.float32),
        "subnormal_amax": (rng.standard_normal((4, 64)) * 1e-39).astype(np.float32),
        "near_underflow_ts": (rng.standard_normal((4, 64)) * 1e-36).astype(np.float32),
        "signed_tiny": np.tile(np.array([1.0, -1e-3, -0.0, 2e-3] * 4, np.float32), (2, 1)),
        "e2m1_midpoints": np.tile(np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5] * 2, np.float32) * 0.1, (3, 1)),
    }
    for name, w in cases.items():
        W, ref = quantize_both(torch.from_numpy(w))
        assert_bit_exact(W, ref, name)


def test_deterministic_and_empty():
    w = inputs.weights(64, 256, seed=5).to(DEV)
    a, b = g.nvfp4_quantize(w), g.nvfp4_quantize(w)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    e = g.nvfp4_quantize(torch.empty(0, 64, device=DEV))
    torch.cuda.synchronize()
    assert e.codes.numel() == 0 and e.tensor_scale.item() == 0.0


def test_bad_shape_raises():
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_quantize(torch.zeros(4, 40, device=DEV))
