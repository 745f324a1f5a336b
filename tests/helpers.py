"""Shared helpers for the parity tests (device results vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gemm_nvfp4_gb300 import inputs

DEV = "cuda:0"

# |y - y_ref| <= REL * sum_k |w x| + ABS  (the accuracy bound of the library)
REL, ABS = 1e-5, 1e-7
# bf16 outputs additionally carry the round-to-nearest-even of the fp32 result
BF16_REL = 2.0 ** -8


def oracle_weight(w_cpu: torch.Tensor):
    return oracle.quantize(w_cpu.numpy())


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.double().numpy()


def gemv_tol(y_ref, A, out_dtype=torch.float32):
    tol = REL * A + ABS
    if out_dtype == torch.bfloat16:
        tol = tol + BF16_REL * np.abs(y_ref)
    return tol


def swiglu_tol(h_ref, g_ref, u_ref, Ag, Au, out_dtype=torch.float32):
    # |d silu/dg| <= 1.1; errors of g and u propagate through h = silu(g) * u,
    # plus a few ulps of fp32 for exp and the division.
    tg = REL * Ag + ABS
    tu = REL * Au + ABS
    silu = g_ref / (1.0 + np.exp(-g_ref))
    tol = 1.1 * np.abs(u_ref) * tg + np.abs(silu) * tu + 1.1 * tg * tu + 2e-6 * np.abs(h_ref) + ABS
    if out_dtype == torch.bfloat16:
        tol = tol + BF16_REL * np.abs(h_ref)
    return tol


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()}: "
                             f"got {got[bad][:5]}, ref {ref[bad][:5]}, tol {np.asarray(tol)[bad][:5]}")


def bf16_bits(x):
    return inputs.bf16_bits(x)
