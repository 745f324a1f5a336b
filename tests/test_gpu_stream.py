"""Product lists in one launch (nvfp4_stream_plan / nvfp4_stream_run) vs the oracle.

Every job's output is compared with the oracle evaluated on the job's actual
input: a caller buffer, or, for a job that reads an earlier job's output, that
output as the launch left it (bf16).  A job that read its input before the
producing job had finished would not match, so the chained cases also check
the ordering inside the launch.  Repeated runs, and replays of a captured CUDA
graph, must give the same bits.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_nvfp4_gb300 as g
import oracle
from gemm_nvfp4_gb300 import inputs
from helpers import DEV, assert_close, bf16_bits, gemv_tol, swiglu_tol, to_np

pytestmark = pytest.mark.gpu


def quantize_pair(M, K, seed, heavy=False):
    w = inputs.weights(M, K, seed=seed, heavy_tail=heavy, device=DEV)
    return g.nvfp4_quantize(w), w


def oracle_weight(W: g.NVFP4Weight):
    return W.codes.cpu().numpy(), W.scales.cpu().numpy(), float(W.tensor_scale.cpu().numpy()[0])


def check_jobs(jobs, rows_per_job=None, what=""):
    """Each job against the oracle on its actual input (all rows, or a sample)."""
    for i, job in enumerate(jobs):
        x = job.x if job.x is not None else jobs[job.input].y
        xb = bf16_bits(x.contiguous() if x.stride(1) == 1 else x)
        ws = job.weights()
        M = ws[0].M
        rows = None
        if rows_per_job is not None and M > rows_per_job:
            rng = np.random.default_rng(M + i)
            rows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.integers(0, M, rows_per_job)]))
        got = to_np(job.y)
        if rows is not None:
            got = got[:, rows]
        if len(ws) == 1:
            y_ref, A = oracle.gemv(xb, *oracle_weight(ws[0]), rows=rows)
            assert_close(got, y_ref, gemv_tol(y_ref, A, job.y.dtype), f"{what} job {i} (M={M})")
        else:
            h_ref, g_ref, u_ref, Ag, Au = oracle.swiglu(xb, oracle_weight(ws[0]), oracle_weight(ws[1]), rows=rows)
            assert_close(got, h_ref, swiglu_tol(h_ref, g_ref, u_ref, Ag, Au, job.y.dtype),
                         f"{what} gate/up job {i} (M={M})")


def status_clean(plan):
    assert g.nvfp4_device_status(plan.buffer, clear=False) == (g.NVFP4_OK, 0)


@pytest.mark.parametrize("N", [1, 4, 16])
def test_independent_list_mixed_shapes(N):
    """Single matrices and gate/up pairs of several shapes (ragged row tiles,
    jobs smaller than one unit per SM, one job with more tiles than SMs),
    fp32 and bf16 outputs, caller-provided activations (one with a row stride)."""
    shapes = [(200, 512, 1, torch.float32), (64, 256, 1, torch.bfloat16), (1000, 1024, 2, torch.float32),
              (4096, 768, 1, torch.float32), (384, 2048, 2, torch.bfloat16), (20000, 256, 1, torch.float32),
              (136, 4352, 1, torch.bfloat16)]
    jobs = []
    for i, (M, K, nw, dt) in enumerate(shapes):
        Ws = tuple(quantize_pair(M, K, seed=10 * i + k)[0] for k in range(nw))
        if i == 3:  # strided rows: a view into a wider buffer
            xx = inputs.activations(N, K + 64, seed=100 + i, outlier_rows=True, device=DEV)[:, :K]
        else:
            xx = inputs.activations(N, K, seed=100 + i, outlier_rows=(i % 2 == 1), device=DEV)
        y = torch.empty(N, M, dtype=dt, device=DEV)
        jobs.append(g.SkinnyJob(Ws if nw == 2 else Ws[0], y, x=xx))
    plan = g.nvfp4_stream_plan(jobs, N)
    g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    first = [j.y.clone() for j in jobs]
    status_clean(plan)
    check_jobs(jobs, rows_per_job=400, what=f"independent N={N}")
    # runs of one plan are deterministic (and the run state resets itself)
    for _ in range(2):
        g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    for j, y0 in zip(jobs, first):
        assert torch.equal(j.y, y0)
    status_clean(plan)


def small_layers(n_layers, hidden, qkv, ffn, N, seed, heavy=False, outliers=False):
    """A dependent decode chain: per layer QKV (input: the previous layer's
    down output), O (a caller buffer standing in for attention's output),
    gate/up + SwiGLU (input: O's output) and down (input: the SwiGLU output)."""
    jobs = []
    x0 = inputs.activations(N, hidden, seed=seed, outlier_rows=outliers, device=DEV)
    prev_down = None
    for li in range(n_layers):
        s = seed + 1000 * (li + 1)
        Wqkv = quantize_pair(qkv, hidden, s + 0, heavy)[0]
        Wo = quantize_pair(hidden, hidden, s + 100, heavy)[0]
        Wg = quantize_pair(ffn, hidden, s + 200, heavy)[0]
        Wu = quantize_pair(ffn, hidden, s + 300, heavy)[0]
        Wd = quantize_pair(hidden, ffn, s + 400, heavy)[0]
        y_qkv = torch.empty(N, qkv, dtype=torch.float32, device=DEV)
        if prev_down is None:
            jobs.append(g.SkinnyJob(Wqkv, y_qkv, x=x0))
        else:
            jobs.append(g.SkinnyJob(Wqkv, y_qkv, input=prev_down))
        x_attn = inputs.activations(N, hidden, seed=s + 7, outlier_rows=outliers, device=DEV)
        jobs.append(g.SkinnyJob(Wo, torch.empty(N, hidden, dtype=torch.bfloat16, device=DEV), x=x_attn))
        o_idx = len(jobs) - 1
        jobs.append(g.SkinnyJob((Wg, Wu), torch.empty(N, ffn, dtype=torch.bfloat16, device=DEV), input=o_idx))
        jobs.append(g.SkinnyJob(Wd, torch.empty(N, hidden, dtype=torch.bfloat16, device=DEV), input=len(jobs) - 1))
        prev_down = len(jobs) - 1
    return jobs


@pytest.mark.parametrize("N", [1, 4, 9, 16])
def test_dependent_chain_small(N):
    jobs = small_layers(3, hidden=512, qkv=768, ffn=1536, N=N, seed=N, outliers=True)
    plan = g.nvfp4_stream_plan(jobs, N)
    g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    status_clean(plan)
    check_jobs(jobs, what=f"chain N={N}")
    first = [j.y.clone() for j in jobs]
    g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    for j, y0 in zip(jobs, first):
        assert torch.equal(j.y, y0)


def test_dependent_chain_in_a_cuda_graph():
    """The chain captured once and replayed: every replay gives the eager bits."""
    N = 4
    jobs = small_layers(2, hidden=1024, qkv=1536, ffn=2048, N=N, seed=33)
    plan = g.nvfp4_stream_plan(jobs, N)
    g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    ref = [j.y.clone() for j in jobs]
    check_jobs(jobs, what="graph chain (eager)")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.nvfp4_stream_run(plan, stream=s)
    for _ in range(3):
        for j in jobs:
            j.y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for j, y0 in zip(jobs, ref):
            assert torch.equal(j.y, y0)
    status_clean(plan)


@pytest.mark.parametrize("shape,N,heavy", [(inputs.LAYER_9B, 1, False), (inputs.LAYER_27B, 4, False),
                                           (inputs.LAYER_27B, 16, True)])
def test_full_size_chain_sampled(shape, N, heavy):
    """Two full-size decoder layers chained (the benchmark's shapes), sampled rows."""
    jobs = small_layers(2, hidden=shape.hidden, qkv=shape.qkv_out, ffn=shape.ffn, N=N, seed=5, heavy=heavy,
                        outliers=heavy)
    plan = g.nvfp4_stream_plan(jobs, N)
    g.nvfp4_stream_run(plan)
    torch.cuda.synchronize()
    status_clean(plan)
    check_jobs(jobs, rows_per_job=48, what=f"{shape.name} chain N={N}")


def test_plan_rejects_bad_lists():
    W = quantize_pair(256, 512, 1)[0]
    x = inputs.activations(2, 512, seed=2, device=DEV)
    y32 = torch.empty(2, 256, dtype=torch.float32, device=DEV)
    ybf = torch.empty(2, 256, dtype=torch.bfloat16, device=DEV)
    W2 = quantize_pair(256, 256, 3)[0]
    bad = [
        [g.SkinnyJob(W2, y32, input=0)],                                   # a job reading itself
        [g.SkinnyJob(W, y32, x=x), g.SkinnyJob(W2, ybf, input=0)],         # input is fp32
        [g.SkinnyJob(W, ybf, x=x), g.SkinnyJob(W, y32, input=0)],          # input narrower than K
    ]
    for jobs in bad:
        assert g.nvfp4_stream_plan_bytes(jobs, 2) == 0
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_stream_plan([g.SkinnyJob(W, y32, x=x)], 17)
    W3 = quantize_pair(64, 272, 4)[0]  # K % 256 != 0
    with pytest.raises(g.NVFP4Error):
        g.nvfp4_stream_plan([g.SkinnyJob(W3, torch.empty(2, 64, device=DEV),
                                         x=inputs.activations(2, 272, seed=5, device=DEV))], 2)
