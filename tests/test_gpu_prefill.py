"""Prefill product (N > 16, tcgen05 tensor cores) through the C ABI vs the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, swiglu_tol, to_np

pytestmark = pytest.mark.gpu


def workspace(op, N, M, K):
    """A prefill workspace filled with garbage (the call needs no initialised
    workspace) except for the device status word, zeroed so it can be read."""
    n = g.nvfp4_workspace_bytes(op, N, M, K)
    ws = torch.full((max(n, 256),), 0xAB, dtype=torch.uint8, device=DEV)
    ws[g.NVFP4_STATUS_WORD_OFFSET:g.NVFP4_STATUS_WORD_OFFSET + 4] = 0
    return ws


def timeout_flag(ws):
    """The device status word: nonzero if a pipeline wait gave up."""
    st, code = g.nvfp4_device_status(ws, clear=False)
    assert (st == g.NVFP4_OK) == (code == 0)
    return code


@pytest.mark.parametrize("N,M,K", [(17, 48, 272), (40, 130, 512), (256, 128, 64), (257, 256, 1024),
                                   (300, 500, 2064), (600, 384, 4096)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_small(N, M, K, out_dtype):
    w = inputs.weights(M, K, seed=N + M)
    x = inputs.activations(N, K, seed=N + K)
    W = g.nvfp4_quantize(w.to(DEV))
    ws = workspace(g.NVFP4_OP_GEMM_PREFILL, N, M, K)
    y = g.nvfp4_gemm_prefill(x.to(DEV), W, out_dtype=out_dtype, workspace=ws)
    torch.cuda.synchronize()
    assert timeout_flag(ws) == 0
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
    ws = workspace(g.NVFP4_OP_GATEUP_SWIGLU, N, M, K)
    h = g.nvfp4_gateup_swiglu(x.to(DEV), Wg, Wu, workspace=ws)
    torch.cuda.synchronize()
    assert timeout_flag(ws) == 0
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


def _sample(n, total, seed, edges):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, total, n), edges]))


@pytest.mark.parametrize("N", [512, 2048, 8192])
def test_prefill_gateup_full_size_sampled(N):
    """Full-size prefill gate/up (5120 -> 17408 each, SwiGLU), sampled outputs."""
    M, K = inputs.LAYER_27B.shapes()["gate"]
    wg = inputs.weights(M, K, seed=200, device=DEV)
    wu = inputs.weights(M, K, seed=300, device=DEV)
    x = inputs.activations(N, K, seed=201, device=DEV)
    Wg, Wu = g.nvfp4_quantize(wg), g.nvfp4_quantize(wu)
    ws = workspace(g.NVFP4_OP_GATEUP_SWIGLU, N, M, K)
    h = g.nvfp4_gateup_swiglu(x, Wg, Wu, workspace=ws)
    torch.cuda.synchronize()
    assert timeout_flag(ws) == 0
    gref, uref = oracle.quantize(wg.cpu().numpy()), oracle.quantize(wu.cpu().numpy())
    rows = _sample(24, M, N, [0, 127, 128, M - 1])
    toks = _sample(6, N, N + 1, [0, 255, 256, N - 1])
    h_ref, g_ref, u_ref, Ag, Au = oracle.swiglu(bf16_bits(x), gref, uref, rows=rows, tokens=toks)
    got = to_np(h)[np.ix_(toks, rows)]
    assert_close(got, h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au), f"gate/up prefill N={N}")


@pytest.mark.parametrize("N", [512, 2048, 8192])
def test_prefill_down_full_size_sampled(N):
    """Full-size prefill down projection (17408 -> 5120), fresh bf16 inputs, at
    every token count the benchmark times: N = 512 splits every tile's K
    across the SMs; N = 2048 and 8192 run whole-tile waves, then k slices of
    the tiles left (split mode's two forms), each followed by its reduction."""
    M, K = inputs.LAYER_27B.shapes()["down"]
    w = inputs.weights(M, K, seed=400, device=DEV)
    x = inputs.activations(N, K, seed=401, device=DEV)
    W = g.nvfp4_quantize(w)
    ws = workspace(g.NVFP4_OP_GEMM_PREFILL, N, M, K)
    y = g.nvfp4_gemm_prefill(x, W, workspace=ws, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert timeout_flag(ws) == 0
    ref_w = oracle.quantize(w.cpu().numpy())
    rows = _sample(24, M, N, [0, 127, 128, M - 1])
    toks = _sample(8, N, N + 2, [0, 191, 192, 255, 256, N - 1])
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows, tokens=toks)
    got = to_np(y)[np.ix_(toks, rows)]
    assert_close(got, y_ref, gemv_tol(y_ref, A, torch.bfloat16), f"down prefill N={N}")


@pytest.mark.parametrize("fmt", ["nvfp4", "fp6"])
def test_token_rows_independent_of_tile_choice(fmt):
    """The launch picks 192- or 256-token tiles from N and the SM count
    (N = 600 and N = 4096 over 64 row tiles take different tiles on a 152-SM
    GPU; N = 300 fills two token tiles); a token's row is the same bits either
    way.  The operations here never split K (an NVFP4 gate/up pair, one FP6
    matrix), so the contract is bit identity."""
    M, K = 8192, 1024
    w = inputs.weights(M, K, seed=81, device=DEV)
    x = inputs.activations(4096, K, seed=82, device=DEV)
    if fmt == "nvfp4":
        Wg = g.nvfp4_quantize(w)
        Wu = g.nvfp4_quantize(inputs.weights(M, K, seed=83, device=DEV))
        run = lambda xx: g.nvfp4_gateup_swiglu(xx, Wg, Wu)
    else:
        W = g.nvfp4_fp6_quantize(w)
        run = lambda xx: g.nvfp4_fp6_gemm(xx, W)
    y_all = run(x)
    y_600 = run(x[:600].contiguous())
    y_300 = run(x[100:400].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(y_600, y_all[:600])
    assert torch.equal(y_300, y_all[100:400])


@pytest.mark.parametrize("N,M,K", [(40, 130, 512), (600, 384, 4096), (700, 1300, 3072), (2100, 640, 8192),
                                   (4096, 4096, 512), (4096, 1280, 16384)])
def test_split_k_prefill_deterministic(N, M, K):
    """Single matrices whose tiles fill the SMs' last wave poorly split K
    across CTAs: with operands that fit in L2, contiguous unit ranges (a part
    of one tile, parts of two, or whole tiles between two parts); with larger
    operands (the last shape: 134 MB of activations), whole-tile waves and
    then equal k slices of the tiles left.  fp32 partials are added by a
    reduction launch, in CTA order.  Repeated calls give the same
    bits, and the result matches the oracle.  Ragged row and token tiles
    included."""
    w = inputs.weights(M, K, seed=N + 5, device=DEV)
    x = inputs.activations(N, K, seed=N + 6, device=DEV)
    W = g.nvfp4_quantize(w)
    ws = workspace(g.NVFP4_OP_GEMM_PREFILL, N, M, K)
    y1 = g.nvfp4_gemm_prefill(x, W, workspace=ws)
    y2 = g.nvfp4_gemm_prefill(x, W, workspace=ws)
    torch.cuda.synchronize()
    assert timeout_flag(ws) == 0
    assert torch.equal(y1, y2)
    ref_w = oracle.quantize(w.cpu().numpy())
    rows = _sample(24, M, N + 7, [0, 127, 128, M - 1])
    toks = _sample(6, N, N + 8, [0, N - 1])
    y_ref, A = oracle.gemv(bf16_bits(x), *ref_w, rows=rows, tokens=toks)
    assert_close(to_np(y1)[np.ix_(toks, rows)], y_ref, gemv_tol(y_ref, A), f"split prefill N={N}")


def test_dependent_prefill_chain_eager_and_graph():
    """Three prefill calls back to back on one stream, each reading the output
    of the one before: gate/up + SwiGLU with bf16 h, a down projection that
    splits K (stream-K launch, then its reduction launch), and a product over
    the down output (K % 256 != 0: the plain-load kernel).  Every prefill
    launch is a programmatic dependent launch that waits for the kernel
    before it before any global access, so each stage must agree with the
    oracle run on the input that stage actually received, complete.  The
    chain captured in a CUDA graph and replayed gives the eager bits."""
    N, K0, M1, M2, M3 = 600, 512, 4096, 384, 256
    wg = inputs.weights(M1, K0, seed=41, device=DEV)
    wu = inputs.weights(M1, K0, seed=42, device=DEV)
    wd = inputs.weights(M2, M1, seed=43, device=DEV)
    w3 = inputs.weights(M3, M2, seed=44, device=DEV)
    Wg, Wu, Wd, W3 = (g.nvfp4_quantize(w) for w in (wg, wu, wd, w3))
    x = inputs.activations(N, K0, seed=45, device=DEV)
    h = torch.empty(N, M1, dtype=torch.bfloat16, device=DEV)
    y = torch.empty(N, M2, dtype=torch.bfloat16, device=DEV)
    z = torch.empty(N, M3, dtype=torch.float32, device=DEV)
    ws1 = workspace(g.NVFP4_OP_GATEUP_SWIGLU, N, M1, K0)
    ws2 = workspace(g.NVFP4_OP_GEMM_PREFILL, N, M2, M1)
    ws3 = workspace(g.NVFP4_OP_GEMM_PREFILL, N, M3, M2)

    def chain(stream=None):
        g.nvfp4_gateup_swiglu(x, Wg, Wu, out=h, workspace=ws1, stream=stream)
        g.nvfp4_gemm_prefill(h, Wd, out=y, workspace=ws2, stream=stream)
        g.nvfp4_gemm_prefill(y, W3, out=z, workspace=ws3, stream=stream)

    chain()
    torch.cuda.synchronize()
    for ws in (ws1, ws2, ws3):
        assert timeout_flag(ws) == 0
    ref = [t.clone() for t in (h, y, z)]
    toks = _sample(8, N, 46, [0, 255, 256, N - 1])
    r1, r2, r3 = (_sample(24, M, 47 + i, [0, 127, 128, M - 1]) for i, M in enumerate((M1, M2, M3)))
    h_ref, g_ref, u_ref, Ag, Au = oracle.swiglu(bf16_bits(x), oracle.quantize(wg.cpu().numpy()),
                                                oracle.quantize(wu.cpu().numpy()), rows=r1, tokens=toks)
    assert_close(to_np(h)[np.ix_(toks, r1)], h_ref,
                 swiglu_tol(h_ref, g_ref, u_ref, Ag, Au, torch.bfloat16), "chain stage 1 (gate/up)")
    y_ref, A = oracle.gemv(bf16_bits(h), *oracle.quantize(wd.cpu().numpy()), rows=r2, tokens=toks)
    assert_close(to_np(y)[np.ix_(toks, r2)], y_ref, gemv_tol(y_ref, A, torch.bfloat16), "chain stage 2 (down)")
    z_ref, A = oracle.gemv(bf16_bits(y), *oracle.quantize(w3.cpu().numpy()), rows=r3, tokens=toks)
    assert_close(to_np(z)[np.ix_(toks, r3)], z_ref, gemv_tol(z_ref, A), "chain stage 3")

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain(stream=s)
    for _ in range(3):
        for t in (h, y, z):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for t, t0 in zip((h, y, z), ref):
            assert torch.equal(t, t0)
    for ws in (ws1, ws2, ws3):
        assert timeout_flag(ws) == 0
