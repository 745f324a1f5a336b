"""Skinny product (N = 1..16) through the C ABI vs the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, to_np

pytestmark = pytest.mark.gpu


def make_case(M, K, N, seed=0, heavy=False, outliers=False):
    w = inputs.weights(M, K, seed=seed, heavy_tail=heavy)
    x = inputs.activations(N, K, seed=seed + 1, outlier_rows=outliers)
    W = g.nvfp4_quantize(w.to(DEV))
    ref_w = oracle.quantize(w.numpy())
    return W, ref_w, x


def check(W, ref_w, x, out_dtype=torch.float32, rows=None, what=""):
    y = g.nvfp4_gemv_skinny(x.to(DEV), W, out_dtype=out_dtype)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    got = to_np(y) if rows is None else to_np(y[:, torch.as_tensor(rows)])
    assert_close(got, y_ref, gemv_tol(y_ref, A, out_dtype), what)
    return y


def test_single_matrix_4096_n1():
    W, ref, x = make_case(4096, 4096, 1)
    check(W, ref, x, what="4096x4096 N=1")


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8, 9, 12, 16])
@pytest.mark.parametrize("M,K", [(16, 128), (48, 272), (100, 1024), (333, 4112), (1000, 2048)])
def test_shapes_and_token_counts(M, K, N):
    W, ref, x = make_case(M, K, N, seed=M * 7 + K)
    check(W, ref, x, what=f"M={M} K={K} N={N}")


@pytest.mark.parametrize("K", [16, 32, 48, 112, 144])
def test_short_k(K):
    W, ref, x = make_case(40, K, 5, seed=K)
    check(W, ref, x, what=f"K={K}")


def test_outliers_and_heavy_tail():
    W, ref, x = make_case(512, 5120, 16, seed=300, heavy=True, outliers=True)
    check(W, ref, x, what="heavy tail + outlier rows")


def test_bf16_output():
    W, ref, x = make_case(300, 2048, 4, seed=11)
    check(W, ref, x, out_dtype=torch.bfloat16, what="bf16 out")


def test_cross_n_identity_and_determinism():
    """Token n of an N-token call equals the same token alone, bit for bit, and
    repeated calls are bit-identical (fixed reduction order)."""
    W, ref, x = make_case(1000, 5120, 16, seed=21)
    xd = x.to(DEV)
    y16 = g.nvfp4_gemv_skinny(xd, W)
    y16b = g.nvfp4_gemv_skinny(xd, W)
    singles = [g.nvfp4_gemv_skinny(xd[n:n + 1].contiguous(), W) for n in range(16)]
    y4 = g.nvfp4_gemv_skinny(xd[4:8].contiguous(), W)
    torch.cuda.synchronize()
    assert torch.equal(y16, y16b)
    for n in range(16):
        assert torch.equal(y16[n], singles[n][0]), n
    assert torch.equal(y16[4:8], y4)


def test_k_zero_gives_zeros_and_empty_calls():
    W = g.NVFP4Weight(torch.empty(8, 0, dtype=torch.uint8, device=DEV),
                      torch.empty(8, 0, dtype=torch.uint8, device=DEV),
                      torch.ones(1, device=DEV))
    x = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    y = torch.full((3, 8), 7.0, device=DEV)
    g.nvfp4_gemv_skinny(x, W, out=y)
    torch.cuda.synchronize()
    assert (y == 0).all()


def test_n_out_of_range_raises():
    W, _, x = make_case(32, 64, 17)
    with pytest.raises(g.NVFP4Error) as e:
        g.nvfp4_gemv_skinny(x.to(DEV), W)
    assert e.value.status == 2


@pytest.mark.parametrize("name", ["qkv", "o", "gate", "down"])
@pytest.mark.parametrize("N", [1, 4])
def test_27b_layer_shapes_sampled(name, N):
    """Full 27B-class layer shapes, device-generated weights, sampled rows."""
    M, K = inputs.LAYER_27B.shapes()[name]
    seed = inputs.matrix_seed(name)
    w = inputs.weights(M, K, seed=seed, device=DEV)
    x = inputs.activations(N, K, seed=seed + 1, device=DEV)
    W = g.nvfp4_quantize(w)
    y = g.nvfp4_gemv_skinny(x, W)
    torch.cuda.synchronize()
    ref_w = oracle.quantize(w.cpu().numpy())
    assert np.array_equal(W.codes.cpu().numpy(), ref_w[0])
    assert np.array_equal(W.scales.cpu().numpy(), ref_w[1])
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.integers(0, M, 48), [0, 15, 16, M - 17, M - 1]]))
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    assert_close(to_np(y)[:, rows], y_ref, gemv_tol(y_ref, A), f"{name} N={N}")


@pytest.mark.parametrize("N", [9, 16])
def test_27b_deep_verify_sampled(N):
    """The deep-verify workload: heavy-tailed weights and x8 outlier token rows."""
    M, K = inputs.LAYER_27B.shapes()["down"]
    w = inputs.weights(M, K, seed=400, heavy_tail=True, device=DEV)
    x = inputs.activations(N, K, seed=401, outlier_rows=True, device=DEV)
    W = g.nvfp4_quantize(w)
    y = g.nvfp4_gemv_skinny(x, W)
    torch.cuda.synchronize()
    ref_w = oracle.quantize(w.cpu().numpy())
    assert np.array_equal(W.codes.cpu().numpy(), ref_w[0])
    rows = np.unique(np.random.default_rng(N).integers(0, M, 40))
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows)
    assert_close(to_np(y)[:, rows], y_ref, gemv_tol(y_ref, A), f"deep verify N={N}")


def test_activations_not_exact_in_f16_fall_back_exactly():
    """A token whose elements span more than the f16 window after scaling
    (here 1e4 next to 1e-12) makes the call use bf16 operands; results stay
    within the bound for every token, including the wide-range one."""
    M, K, N = 512, 4096, 4
    w = inputs.weights(M, K, seed=77)
    x = inputs.activations(N, K, seed=78).float()
    x[2, 5] = 1.0e4
    x[2, 6:200] = 1.0e-12
    xb = x.to(torch.bfloat16)
    W = g.nvfp4_quantize(w.to(DEV))
    ref = oracle.quantize(w.numpy())
    y = g.nvfp4_gemv_skinny(xb.to(DEV), W)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(bf16_bits(xb), *ref)
    assert_close(to_np(y), y_ref, gemv_tol(y_ref, A), "wide-range token")


def test_zero_and_tiny_token_rows():
    M, K, N = 256, 2048, 3
    w = inputs.weights(M, K, seed=79)
    x = inputs.activations(N, K, seed=80).float()
    x[0] = 0.0
    x[1] *= 1e-30
    xb = x.to(torch.bfloat16)
    W = g.nvfp4_quantize(w.to(DEV))
    ref = oracle.quantize(w.numpy())
    y = g.nvfp4_gemv_skinny(xb.to(DEV), W)
    torch.cuda.synchronize()
    y_ref, A = oracle.gemv(bf16_bits(xb), *ref)
    assert_close(to_np(y), y_ref, gemv_tol(y_ref, A), "zero / tiny rows")
    assert (to_np(y)[0] == 0).all()


@pytest.mark.parametrize("M", [1, 100, 127, 129, 4224])
def test_ragged_rows_tensor_core_path(M):
    """M not a multiple of the 128-row tile on the tcgen05 path (K % 256 == 0)."""
    W, ref, x = make_case(M, 1280, 5, seed=M)
    check(W, ref, x, what=f"M={M}")


def test_workspace_reuse_back_to_back():
    """Two different shapes sharing one workspace, queued back to back."""
    W1, r1, x1 = make_case(4096, 4096, 1, seed=1)
    W2, r2, x2 = make_case(12288, 4096, 4, seed=2)
    need = max(g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 1, 4096, 4096),
               g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 4, 12288, 4096))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)  # zero-filled once, kept zero by every call
    outs = []
    for _ in range(3):
        outs.append(g.nvfp4_gemv_skinny(x1.to(DEV), W1, workspace=ws))
        outs.append(g.nvfp4_gemv_skinny(x2.to(DEV), W2, workspace=ws))
    torch.cuda.synchronize()
    for o in outs[2::2]:
        assert torch.equal(o, outs[0])
    for o in outs[3::2]:
        assert torch.equal(o, outs[1])
    y_ref, A = oracle.gemv(bf16_bits(x2), *r2, rows=np.arange(0, 12288, 97))
    assert_close(to_np(outs[1])[:, ::97], y_ref, gemv_tol(y_ref, A), "reuse")


def test_workspace_left_zero_across_paths():
    """The skinny calls keep split-K counters in a fixed region of the
    workspace (bytes 256 .. 256 + 1 MiB) and leave it zero: one zeroing
    serves a mixed sequence of shapes and paths (prep kernel or not, gate/up,
    the mma.sync path for K % 256 != 0), and each result equals the same call
    on a fresh workspace."""
    cases = [(4096, 4096, 1, 1), (12288, 4096, 4, 1), (4096, 4096, 2, 2), (300, 4000, 3, 1),
             (5120, 17408, 16, 1), (640, 2048, 7, 1), (12288, 4096, 1, 2)]
    need = 0
    for M, K, N, nw in cases:
        op = g.NVFP4_OP_GEMV_SKINNY if nw == 1 else g.NVFP4_OP_GATEUP_SWIGLU
        need = max(need, g.nvfp4_workspace_bytes(op, N, M, K))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for i, (M, K, N, nw) in enumerate(cases):
        Ws = [g.nvfp4_quantize(inputs.weights(M, K, seed=50 + 10 * i + j).to(DEV)) for j in range(nw)]
        x = inputs.activations(N, K, seed=7 + i).to(DEV)
        call = (lambda w: g.nvfp4_gemv_skinny(x, Ws[0], workspace=w)) if nw == 1 else \
            (lambda w: g.nvfp4_gateup_swiglu(x, Ws[0], Ws[1], workspace=w))
        got = call(ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws[256:256 + (1 << 20)]).item()) == 0, f"counters not left zero after case {i}"
        ref = call(None)  # fresh zero-filled workspace from the binding
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"case {i}"


def test_workspace_shared_with_fp6_and_prefill_calls():
    """FP6 skinny calls (split-K partials in the same region, zeroed after
    use) and prefill calls (word 0 only) on a workspace shared with NVFP4
    skinny calls leave the counter region zero, and the NVFP4 results stay
    those of a fresh workspace."""
    M, K = 5120, 4096
    need = max(g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 16, M, K),
               g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GATEUP_SWIGLU, 16, M, K),
               g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, 300, M, K))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    w = inputs.weights(M, K, seed=91).to(DEV)
    W, W6 = g.nvfp4_quantize(w), g.nvfp4_fp6_quantize(w)
    x = inputs.activations(300, K, seed=92).to(DEV)
    for step in range(3):
        g.nvfp4_fp6_gemm(x[:9].contiguous(), W6, workspace=ws)
        g.nvfp4_fp6_gateup_swiglu(x[:3].contiguous(), W6, W6, workspace=ws)
        g.nvfp4_gemm_prefill(x, W, workspace=ws)
        y = g.nvfp4_gemv_skinny(x[:5].contiguous(), W, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws[256:256 + (1 << 20)]).item()) == 0, step
        assert torch.equal(y, g.nvfp4_gemv_skinny(x[:5].contiguous(), W))
