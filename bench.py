"""Benchmark of the NVFP4 x bf16 decode path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense9b-n1|dense27b-n1|dense27b-n4|dense27b-n9|dense27b-n16]

A step is one pass of the decode hot path over a rotating stream of dense
decoder layers (weights larger than L2): per layer the fused QKV projection,
the O projection, the fused gate/up + SwiGLU, and the down projection, all
NVFP4 weights x bf16 activations, fp32 out.  The default workload is the dense
9B-class layer stream at N = 1 (36 distinct layers, 3.9 GB of NVFP4 weights).
The whole stream is captured once as a CUDA graph (one replay per step, as a
CUDA-graph decode replays one graph per token) and timed with CUDA events.

Printed: one JSON line with the HBM GB/s of the stream (algorithmic bytes:
codes + scales + x + y), the roofline of the dominant kernel, an end-to-end
number with host<->device copies, the oracle timed on host cores, and the SM
clocks sampled during the timed region.

--impl reference times the CPU oracle (no other reference implementation of
this path exists) on a bounded sample of the same workload, in the same unit,
on all host cores.
Under torchrun every rank runs its own replica (no collective on the data
path; the path does not shard), rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMV achieved HBM GB/s (% of ~8 TB/s) at N=1/4/9; prefill GEMM TFLOPS"

WORKLOADS = {
    # name: (layer shape, N, layers, heavy-tailed weights, outlier token rows)
    "dense9b-n1": ("LAYER_9B", 1, 36, False, False),
    "dense27b-n1": ("LAYER_27B", 1, 64, False, False),
    "dense27b-n4": ("LAYER_27B", 4, 64, False, False),
    "dense27b-n9": ("LAYER_27B", 9, 64, True, True),
    "dense27b-n16": ("LAYER_27B", 16, 64, True, True),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dense9b-n1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-ingest", action="store_true")
    ap.add_argument("--no-fp6", action="store_true")
    ap.add_argument("--no-streams", action="store_true",
                    help="skip the other decode workloads, the single-matrix stream and the chains")
    ap.add_argument("--fp6-only", action="store_true",
                    help="print the FP6 measurement (27B-class MLP stream and prefill) and exit")
    ap.add_argument("--ingest-only", action="store_true",
                    help="print the ingest measurement (quantise fp32 / bf16, scale import) and exit")
    # for profiling one call kind on a short stream (ncu captures): not a bench line
    ap.add_argument("--layers", type=int, default=None, help="override the number of layers in the stream")
    ap.add_argument("--only", choices=["qkv", "o", "gateup", "down"], default=None,
                    help="time only this call kind of every layer")
    ap.add_argument("--profile-stream", action="store_true",
                    help="three launches of the workload's product list over --layers layers (default 4) and exit "
                         "(for ncu captures)")
    ap.add_argument("--prefill-profile", default=None, metavar="gateup:N|down:N",
                    help="run three prefill calls of one 27B-class shape and exit (for ncu captures)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in rows]
        smax = max(r[1] for r in rows)
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2][1:5]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# the decode layer stream
# ---------------------------------------------------------------------------

class LayerStream:
    """Rotating NVFP4 layers + per-layer activations and outputs on one GPU."""

    def __init__(self, workload: str, device, n_layers=None, layers_from=None):
        import gemm_nvfp4_gb300 as g
        from gemm_nvfp4_gb300 import inputs
        self.g = g
        shape_name, self.N, self.n_layers, heavy, outliers = WORKLOADS[workload]
        if n_layers is not None:
            self.n_layers = n_layers
        self.shape = getattr(inputs, shape_name)
        self.workload = workload
        shapes = self.shape.shapes()
        self.shapes = shapes
        self.device = device
        if layers_from is not None:
            # same weights as another stream of this layer shape (another N)
            self.layers = layers_from.layers
            self.n_layers = layers_from.n_layers
        else:
            # base layer: quantise each matrix once on the GPU, then replicate
            base = {}
            for name, (M, K) in shapes.items():
                w = inputs.weights(M, K, seed=inputs.matrix_seed(name), heavy_tail=heavy, device=device)
                base[name] = g.nvfp4_quantize(w)
                del w
            torch.cuda.synchronize()
            self.layers = []
            for _ in range(self.n_layers):
                layer = {}
                for name, W in base.items():
                    layer[name] = g.NVFP4Weight(W.codes.clone(), W.scales.clone(), W.tensor_scale.clone())
                self.layers.append(layer)
            del base
        # activations per layer and matrix (bf16 N(0,1), the step's inputs) and
        # outputs, as views into one input and one output buffer so the
        # end-to-end run moves each with a single copy
        N = self.N
        names = ("qkv", "o", "gate", "down")
        x_sizes = [N * shapes[n][1] for n in names]
        y_sizes = [N * shapes[n][0] for n in names]
        self.x_all = torch.empty(self.n_layers * sum(x_sizes), dtype=torch.bfloat16, device=device)
        self.y_all = torch.empty(self.n_layers * sum(y_sizes), dtype=torch.float32, device=device)
        self.x, self.y = [], []
        xo = yo = 0
        for li in range(self.n_layers):
            xs, ys = {}, {}
            for name, xsz, ysz in zip(names, x_sizes, y_sizes):
                M, K = shapes[name]
                xs[name] = self.x_all[xo:xo + xsz].view(N, K)
                xs[name].copy_(inputs.activations(N, K, seed=1000 * li + inputs.matrix_seed(name) + 1,
                                                  outlier_rows=outliers, device=device))
                ys[name] = self.y_all[yo:yo + ysz].view(N, M)
                xo += xsz
                yo += ysz
            self.x.append(xs)
            self.y.append(ys)
        ws_need = max(g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, N, M, K) for M, K in shapes.values())
        ws_need = max(ws_need, g.nvfp4_workspace_bytes(g.NVFP4_OP_GATEUP_SWIGLU, N, *shapes["gate"]))
        self.ws = torch.zeros(ws_need, dtype=torch.uint8, device=device)  # skinny workspace: zero-filled once

    # algorithmic bytes (codes + scales + x + y) of each call kind
    def call_bytes(self, name):
        N = self.N
        if name == "gateup":
            M, K = self.shapes["gate"]
            return 2 * (M * K // 2 + M * K // 16) + N * K * 2 + N * M * 4
        M, K = self.shapes[name]
        return M * K // 2 + M * K // 16 + N * K * 2 + N * M * 4

    def step_bytes(self, only=None):
        names = ("qkv", "o", "gateup", "down") if only is None else (only,)
        return self.n_layers * sum(self.call_bytes(n) for n in names)

    def weight_bytes(self):
        return self.n_layers * sum(M * K // 2 + M * K // 16 for M, K in self.shapes.values())

    def run_layer(self, li, only=None):
        g, L, X, Y, ws = self.g, self.layers[self.layer_index(li)], self.x[li], self.y[li], self.ws
        if only in (None, "qkv"):
            g.nvfp4_gemv_skinny(X["qkv"], L["qkv"], out=Y["qkv"], workspace=ws)
        if only in (None, "o"):
            g.nvfp4_gemv_skinny(X["o"], L["o"], out=Y["o"], workspace=ws)
        if only in (None, "gateup"):
            g.nvfp4_gateup_swiglu(X["gate"], L["gate"], L["up"], out=Y["gate"], workspace=ws)
        if only in (None, "down"):
            g.nvfp4_gemv_skinny(X["down"], L["down"], out=Y["down"], workspace=ws)

    def layer_index(self, li):
        return li

    def run_all(self, only=None):
        for li in range(self.n_layers):
            self.run_layer(li, only)

    def launches_per_call(self, name):
        """Our kernels per call: the activation prep kernel and the main kernel
        (split-K partials are reduced inside the main kernel); a single matrix
        with N >= 2 skips the prep kernel (the main kernel reads x itself)."""
        single = name != "gateup"
        return 1 if (single and self.N >= 2) else 2

    def launches_per_step(self, only=None):
        names = ["qkv", "o", "gateup", "down"] if only is None else [only]
        return self.n_layers * sum(self.launches_per_call(n) for n in names)

    def capture(self, only=None):
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run_all(only)  # warm (not captured)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            self.run_all(only)
        torch.cuda.synchronize()
        return graph

    def stream_jobs(self):
        """The step as one product list: every call of every layer on its own
        activations and outputs (the same buffers as the per-call step)."""
        g, jobs = self.g, []
        for li in range(self.n_layers):
            L, X, Y = self.layers[li], self.x[li], self.y[li]
            jobs.append(g.SkinnyJob(L["qkv"], Y["qkv"], x=X["qkv"]))
            jobs.append(g.SkinnyJob(L["o"], Y["o"], x=X["o"]))
            jobs.append(g.SkinnyJob((L["gate"], L["up"]), Y["gate"], x=X["gate"]))
            jobs.append(g.SkinnyJob(L["down"], Y["down"], x=X["down"]))
        return jobs

    def chain_jobs(self):
        """The step as a dependent decode chain: per layer QKV reads the previous
        layer's down output (layer 0: its own input), O reads a caller buffer
        (attention's output, which this library does not compute), gate/up +
        SwiGLU reads O's output and down reads the SwiGLU output; the outputs a
        later job reads are bf16."""
        g, jobs = self.g, []
        N, dev = self.N, self.device
        hidden, ffn = self.shapes["o"][0], self.shapes["gate"][0]
        self.chain_out = []
        prev = None
        for li in range(self.n_layers):
            L, X, Y = self.layers[li], self.x[li], self.y[li]
            o_out = torch.empty(N, hidden, dtype=torch.bfloat16, device=dev)
            h_out = torch.empty(N, ffn, dtype=torch.bfloat16, device=dev)
            d_out = torch.empty(N, hidden, dtype=torch.bfloat16, device=dev)
            self.chain_out += [o_out, h_out, d_out]
            if prev is None:
                jobs.append(g.SkinnyJob(L["qkv"], Y["qkv"], x=X["qkv"]))
            else:
                jobs.append(g.SkinnyJob(L["qkv"], Y["qkv"], input=prev))
            jobs.append(g.SkinnyJob(L["o"], o_out, x=X["o"]))
            jobs.append(g.SkinnyJob((L["gate"], L["up"]), h_out, input=len(jobs) - 1))
            jobs.append(g.SkinnyJob(L["down"], d_out, input=len(jobs) - 1))
            prev = len(jobs) - 1
        return jobs

    def chain_bytes(self):
        """Algorithmic bytes of the chain step: the weights once, every job's
        activations read and outputs written (bf16 where a later job reads them)."""
        N = self.N
        hidden, ffn, qkv = self.shapes["o"][0], self.shapes["gate"][0], self.shapes["qkv"][0]
        per_layer = (sum(M * K // 2 + M * K // 16 for M, K in self.shapes.values())
                     + N * hidden * 2 + N * qkv * 4          # QKV: x in, fp32 out
                     + N * hidden * 2 + N * hidden * 2       # O
                     + N * hidden * 2 + N * ffn * 2          # gate/up
                     + N * ffn * 2 + N * hidden * 2)         # down
        return self.n_layers * per_layer

    def host_io(self):
        """Pinned host copies of the step's inputs and outputs (for e2e)."""
        return ([(self.x_all, self.x_all.cpu().pin_memory())],
                [(self.y_all, torch.empty_like(self.y_all, device="cpu").pin_memory())])


def time_graph(graph, steps, warmup, world, stream=None):
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        graph.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(stop) / steps  # ms per replay


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


KERNEL_SOURCES = ("stream.cu", "skinny.cuh", "tcgen05.cuh", "common.cuh")


def kernel_source_hash():
    """Hash of the stream kernel's sources (the ncu traffic summary records it)."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "gemm_nvfp4_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (the summary records the source hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash()
    for line in open(path):
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        if len(parts) >= 4 and parts[0] == kernel_key and parts[1] == h:
            try:
                return float(parts[2])
            except ValueError:
                return None
    return None


def time_calls(fn, reps):
    """Mean milliseconds of `reps` back-to-back calls on the current stream,
    CUDA events, after one warm-up call."""
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def prefill_tflops(dev, reps=10):
    """Prefill GEMM throughput on the 27B-class gate/up (SwiGLU) and down
    matrices at N = 512, 2048, 8192 (dense bf16-equivalent FLOPs, 2*N*M*K per
    matrix), timed with CUDA events after one warm-up call each; outputs and
    workspaces are allocated before the timed calls."""
    import gemm_nvfp4_gb300 as g
    from gemm_nvfp4_gb300 import inputs
    shapes = inputs.LAYER_27B.shapes()
    out = {"unit": "TFLOP/s", "peak_bf16": read_peaks()[1], "shapes": {}}
    Mg, Kg = shapes["gate"]
    Md, Kd = shapes["down"]
    Wg = g.nvfp4_quantize(inputs.weights(Mg, Kg, seed=inputs.matrix_seed("gate"), device=dev))
    Wu = g.nvfp4_quantize(inputs.weights(Mg, Kg, seed=inputs.matrix_seed("up"), device=dev))
    Wd = g.nvfp4_quantize(inputs.weights(Md, Kd, seed=inputs.matrix_seed("down"), device=dev))
    for N in (512, 2048, 8192):
        xg = inputs.activations(N, Kg, seed=N, device=dev)
        xd = inputs.activations(N, Kd, seed=N + 1, device=dev)
        h = torch.empty(N, Mg, dtype=torch.float32, device=dev)
        y = torch.empty(N, Md, dtype=torch.float32, device=dev)
        wsg = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_GATEUP_SWIGLU, N, Mg, Kg), dtype=torch.uint8,
                          device=dev)
        wsd = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, N, Md, Kd), dtype=torch.uint8,
                          device=dev)
        for name, fn, flops in (
                ("gateup", lambda: g.nvfp4_gateup_swiglu(xg, Wg, Wu, out=h, workspace=wsg), 2 * 2.0 * N * Mg * Kg),
                ("down", lambda: g.nvfp4_gemm_prefill(xd, Wd, out=y, workspace=wsd), 2.0 * N * Md * Kd)):
            ms = time_calls(fn, reps)
            tf = flops / (ms * 1e-3) / 1e12
            out["shapes"][f"{name} N={N}"] = {"ms": ms, "tflops": tf,
                                               "frac": tf / out["peak_bf16"] if out["peak_bf16"] else None}
        del xg, xd, h, y
    torch.cuda.empty_cache()
    return out


def ingest_gbs(dev, reps=5):
    """Load-time ingest on the 27B-class gate matrix (17408 x 5120): quantise
    from fp32 and from bf16, and import of blocked scales.  HBM-bound; the
    algorithmic bytes are two reads of the input (the tensor amax must be known
    before any block is quantised and the matrix is larger than L2) plus the
    NVFP4 writes (0.5625 B per weight); the import reads the blocked scales and
    writes the row-major ones once.  L2 is flushed by reading a 256 MB buffer
    before every timed call."""
    import gemm_nvfp4_gb300 as g
    from gemm_nvfp4_gb300 import inputs
    M, K = inputs.LAYER_27B.shapes()["gate"]
    peak = read_peaks()[0]
    flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    w32 = inputs.weights(M, K, seed=inputs.matrix_seed("gate"), device=dev)
    w16 = w32.to(torch.bfloat16)
    W = g.nvfp4_quantize(w32)
    ws = torch.empty(g.nvfp4_workspace_bytes(g.NVFP4_OP_QUANTIZE, 0, M, K), dtype=torch.uint8, device=dev)
    blocked = torch.randint(0, 256, (g.nvfp4_blocked_scale_bytes(M, K),), dtype=torch.uint8, device=dev)
    scales = torch.empty(M, K // 16, dtype=torch.uint8, device=dev)
    out_bytes = M * K // 2 + M * K // 16 + 4
    ops = {
        "quantize fp32": (lambda: g.nvfp4_quantize(w32, workspace=ws, out=W), 2 * 4 * M * K + out_bytes),
        "quantize bf16": (lambda: g.nvfp4_quantize_bf16(w16, workspace=ws, out=W), 2 * 2 * M * K + out_bytes),
        "import scales": (lambda: g.nvfp4_import_blocked_scales(blocked, M, K, out=scales),
                          blocked.numel() + M * K // 16),
    }
    out = {"unit": "GB/s", "peak_hbm": peak, "matrix": f"{M}x{K}", "l2": "flushed before each call", "ops": {}}
    for name, (fn, nbytes) in ops.items():
        fn()
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(reps):
            torch.amax(flush)  # a read-only flush: leaves no dirty lines to write back
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        ms = total / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["ops"][name] = {"us": ms * 1e3, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak if peak else None}
    del flush, w32, w16, W, blocked, scales
    torch.cuda.empty_cache()
    return out


def fp6_measure(dev, layers=4, reps=10):
    """FP6 E2M3 weights on the 27B-class MLP matrices: the skinny product
    streaming `layers` rotating copies of gate/up (SwiGLU) and down (larger
    than L2 together) at N = 1, 4, 16, as one CUDA graph per N (algorithmic
    bytes: codes + scales + x + outputs), and the prefill GEMMs at N = 2048
    (dense bf16-equivalent FLOPs)."""
    import gemm_nvfp4_gb300 as g
    from gemm_nvfp4_gb300 import inputs
    shapes = inputs.LAYER_27B.shapes()
    Mg, Kg = shapes["gate"]
    Md, Kd = shapes["down"]
    peak_hbm, peak_tf, _ = read_peaks()
    Ws = []
    for li in range(layers):
        ws = [g.nvfp4_fp6_quantize(inputs.weights(M, K, seed=inputs.matrix_seed(n) + 7 * li, device=dev))
              for n, (M, K) in (("gate", (Mg, Kg)), ("up", (Mg, Kg)), ("down", (Md, Kd)))]
        Ws.append(ws)
    torch.cuda.synchronize()
    out = {"unit_stream": "GB/s", "unit_prefill": "TFLOP/s", "peak_hbm": peak_hbm, "peak_bf16": peak_tf,
           "layers": layers, "weight_bytes": sum(W.nbytes() for ws in Ws for W in ws), "stream": {}, "prefill": {}}
    for N in (1, 4, 16):
        xg = inputs.activations(N, Kg, seed=N, device=dev)
        xd = inputs.activations(N, Kd, seed=N + 1, device=dev)
        h = torch.empty(N, Mg, dtype=torch.float32, device=dev)
        y = torch.empty(N, Md, dtype=torch.float32, device=dev)
        wsg = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GATEUP_SWIGLU, N, Mg, Kg), dtype=torch.uint8,
                          device=dev)
        wsd = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, N, Md, Kd), dtype=torch.uint8, device=dev)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            def run():
                for ws in Ws:
                    g.nvfp4_fp6_gateup_swiglu(xg, ws[0], ws[1], out=h, workspace=wsg, stream=s)
                    g.nvfp4_fp6_gemm(xd, ws[2], out=y, workspace=wsd, stream=s)
            run()
            s.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                run()
        ms = time_graph(graph, reps, 3, 1)  # replays run on the current stream
        nbytes = out["weight_bytes"] + layers * (N * Kg * 2 + N * Mg * 4 + N * Kd * 2 + N * Md * 4)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["stream"][f"N={N}"] = {"ms": ms, "gbs": gbs, "frac": gbs / peak_hbm if peak_hbm else None}
    N = 2048
    xg = inputs.activations(N, Kg, seed=5, device=dev)
    xd = inputs.activations(N, Kd, seed=6, device=dev)
    h = torch.empty(N, Mg, dtype=torch.float32, device=dev)
    y = torch.empty(N, Md, dtype=torch.float32, device=dev)
    wsg = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GATEUP_SWIGLU, N, Mg, Kg), dtype=torch.uint8, device=dev)
    wsd = torch.zeros(g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, N, Md, Kd), dtype=torch.uint8, device=dev)
    for name, fn, flops in (("gateup", lambda: g.nvfp4_fp6_gateup_swiglu(xg, Ws[0][0], Ws[0][1], out=h, workspace=wsg),
                             2 * 2.0 * N * Mg * Kg),
                            ("down", lambda: g.nvfp4_fp6_gemm(xd, Ws[0][2], out=y, workspace=wsd), 2.0 * N * Md * Kd)):
        ms = time_calls(fn, 10)
        tf = flops / (ms * 1e-3) / 1e12
        out["prefill"][f"{name} N={N}"] = {"ms": ms, "tflops": tf, "frac": tf / peak_tf if peak_tf else None}
    del Ws
    torch.cuda.empty_cache()
    return out


def prefill_profile(dev, spec):
    """Three prefill calls of one shape (a target for ncu; prints nothing)."""
    import gemm_nvfp4_gb300 as g
    from gemm_nvfp4_gb300 import inputs
    name, n = spec.split(":")
    N = int(n)
    shapes = inputs.LAYER_27B.shapes()
    if name == "gateup":
        M, K = shapes["gate"]
        Wg = g.nvfp4_quantize(inputs.weights(M, K, seed=inputs.matrix_seed("gate"), device=dev))
        Wu = g.nvfp4_quantize(inputs.weights(M, K, seed=inputs.matrix_seed("up"), device=dev))
        x = inputs.activations(N, K, seed=N, device=dev)
        for _ in range(3):
            g.nvfp4_gateup_swiglu(x, Wg, Wu)
    else:
        M, K = shapes["down"]
        W = g.nvfp4_quantize(inputs.weights(M, K, seed=inputs.matrix_seed("down"), device=dev))
        x = inputs.activations(N, K, seed=N, device=dev)
        for _ in range(3):
            g.nvfp4_gemm_prefill(x, W)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def host_threads():
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_sample(workload, rows_per_matrix=64):
    """A row sample of every matrix of one layer, quantised by the oracle:
    returns (jobs, algorithmic bytes of one pass over them)."""
    import oracle
    from gemm_nvfp4_gb300 import inputs
    shape_name, N, _, heavy, outliers = WORKLOADS[workload]
    shape = getattr(inputs, shape_name)
    jobs = []
    for name, (M, K) in shape.shapes().items():
        w = inputs.weights(rows_per_matrix, K, seed=inputs.matrix_seed(name), heavy_tail=heavy)
        x = inputs.activations(N, K, seed=inputs.matrix_seed(name) + 1, outlier_rows=outliers)
        jobs.append((oracle.quantize(w.numpy()), inputs.bf16_bits(x)))
    nbytes = sum(rows_per_matrix * (K // 2 + K // 16) + N * K * 2 + N * rows_per_matrix * 4
                 for _, K in shape.shapes().values())
    return jobs, nbytes


def oracle_pass(jobs, threads=1):
    """Seconds for one pass of the oracle's products over the sample.  With
    threads > 1 the rows of each matrix are split into that many contiguous
    ranges, each computed by the unchanged single-threaded oracle routine on
    its own thread (the C call releases the GIL)."""
    import concurrent.futures as cf

    import oracle
    M = jobs[0][0][0].shape[0]
    parts = [r for r in np.array_split(np.arange(M), threads) if len(r)]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        t0 = time.perf_counter()
        for (codes, scales, ts), xb in jobs:
            if len(parts) == 1:
                oracle.gemv(xb, codes, scales, ts)
            else:
                list(ex.map(lambda rows: oracle.gemv(xb, codes, scales, ts, rows=rows), parts))
        return time.perf_counter() - t0


def _timed_passes(jobs, nbytes, target_s, threads):
    total_dt, reps = 0.0, 0
    while total_dt < target_s:
        total_dt += oracle_pass(jobs, threads)
        reps += 1
    return reps * nbytes / total_dt / 1e9, reps, total_dt


def cpu_baseline(workload, target_s=6.0, rows=1024):
    """The oracle's products on a row sample of one layer, on all host cores
    (rows split across threads) and on one thread, each repeated until about
    target_s seconds have been spent."""
    threads = host_threads()
    jobs, nbytes = oracle_sample(workload, rows_per_matrix=rows)
    value, reps, dt = _timed_passes(jobs, nbytes, target_s, threads)
    v1, reps1, dt1 = _timed_passes(jobs, nbytes, target_s, 1)
    return {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} rows of each of the 5 matrices of one layer of {workload}, N as in the "
                      f"workload, the single-threaded C oracle on {threads} row ranges in parallel threads, "
                      f"{reps} passes, {dt:.1f} s",
            "single_thread": {"value": v1, "unit": "GB/s", "cores": 1,
                              "sample": f"the same rows on one thread, {reps1} passes, {dt1:.1f} s"}}


# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    shape_name, N, layers, _, _ = WORKLOADS[args.workload]
    threads = host_threads()
    rows = 24 * threads
    jobs, nb = oracle_sample(args.workload, rows_per_matrix=rows)
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_pass(jobs, threads)
        if i >= args.warmup:
            times.append(dt)
    dt = sum(times) / len(times)
    value = nb / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "tokens_N": N, "layers_sampled": 1,
                       "rows_per_matrix": rows},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{rows} rows of each matrix of one layer per step, split into "
                                       f"{threads} row ranges on parallel threads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def capture_graph(fn):
    """Capture fn(stream) once as a CUDA graph (after one eager call)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fn(s)
    torch.cuda.synchronize()
    return graph


def time_plan(plan, steps, warmup):
    import gemm_nvfp4_gb300 as g
    graph = capture_graph(lambda s: g.nvfp4_stream_run(plan, stream=s))
    ms = time_graph(graph, steps, warmup, 1)
    st_, code = g.nvfp4_device_status(plan.buffer, clear=False)
    assert st_ == g.NVFP4_OK, f"a stream wait gave up (code {code})"
    return ms


def stream_entry(nbytes, ms, N, peak, layers=None):
    gbs = nbytes / (ms * 1e-3) / 1e9
    d = {"ms": ms, "gbs": gbs, "frac": gbs / peak, "bytes": nbytes}
    if layers is not None:
        d["tokens_per_s_per_stream"] = N / (ms * 1e-3)
    return d


def more_streams(dev, st0, args, peak):
    """The other decode workloads (27B-class streams at N = 1/4/9/16, the
    deep-verify ones with heavy-tailed weights and outlier tokens), the single
    4096 x 4096 matrix over 32 rotating copies at N = 1, and the dependent
    chains, each as one product list per step."""
    import gemm_nvfp4_gb300 as g
    from gemm_nvfp4_gb300 import inputs
    streams, chains = {}, {}
    steps, warm = max(args.steps, 10), max(args.warmup, 3)
    # the default workload's chain
    plan = g.nvfp4_stream_plan(st0.chain_jobs(), st0.N)
    chains[st0.workload] = stream_entry(st0.chain_bytes(), time_plan(plan, steps, warm), st0.N, peak, True)
    del plan
    base = {}
    for wl in ("dense27b-n1", "dense27b-n4", "dense27b-n9", "dense27b-n16"):
        if wl == st0.workload:
            continue
        heavy = WORKLOADS[wl][3]
        st = LayerStream(wl, dev, layers_from=base.get(heavy))
        base.setdefault(heavy, st)
        plan = g.nvfp4_stream_plan(st.stream_jobs(), st.N)
        streams[wl] = stream_entry(st.step_bytes(), time_plan(plan, steps, warm), st.N, peak, True)
        del plan
        if wl in ("dense27b-n1", "dense27b-n4"):
            plan = g.nvfp4_stream_plan(st.chain_jobs(), st.N)
            chains[wl] = stream_entry(st.chain_bytes(), time_plan(plan, steps, warm), st.N, peak, True)
            del plan
        if st is not base.get(heavy):
            del st
    del base
    torch.cuda.empty_cache()
    # the single NVFP4 matrix (4096 x 4096, seed 0) over 32 rotating copies, N = 1
    M = K = 4096
    W = g.nvfp4_quantize(inputs.weights(M, K, seed=0, device=dev))
    jobs = []
    for c in range(32):
        Wc = g.NVFP4Weight(W.codes.clone(), W.scales.clone(), W.tensor_scale.clone())
        x = inputs.activations(1, K, seed=1 + c, device=dev)
        jobs.append(g.SkinnyJob(Wc, torch.empty(1, M, dtype=torch.float32, device=dev), x=x))
    plan = g.nvfp4_stream_plan(jobs, 1)
    nbytes = 32 * (M * K // 2 + M * K // 16 + K * 2 + M * 4)
    streams["single4096-n1"] = stream_entry(nbytes, time_plan(plan, steps, warm), 1, peak)
    streams["single4096-n1"]["copies"] = 32
    del plan, jobs, W
    torch.cuda.empty_cache()
    return streams, chains


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the NVFP4 path has no CPU fallback)")
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.prefill_profile:
        prefill_profile(dev, args.prefill_profile)
        return
    if args.profile_stream:
        import gemm_nvfp4_gb300 as g
        st = LayerStream(args.workload, dev, args.layers or 4)
        plan = g.nvfp4_stream_plan(st.stream_jobs(), st.N)
        for _ in range(3):
            g.nvfp4_stream_run(plan)
        torch.cuda.synchronize()
        assert g.nvfp4_device_status(plan.buffer, clear=False)[0] == g.NVFP4_OK
        return
    if args.ingest_only:
        print(json.dumps(ingest_gbs(dev)), flush=True)
        return
    if args.fp6_only:
        print(json.dumps(fp6_measure(dev)), flush=True)
        return
    import gemm_nvfp4_gb300 as g
    st = LayerStream(args.workload, dev, args.layers)
    hbm_peak, _, peak_kind = read_peaks()
    if args.only is None:
        # the step: every call of every layer as one product list, one launch
        plan = g.nvfp4_stream_plan(st.stream_jobs(), st.N)
        graph = capture_graph(lambda s: g.nvfp4_stream_run(plan, stream=s))
        launches_per_step = 1
    else:
        plan = None
        graph = st.capture(only=args.only)
        launches_per_step = st.launches_per_step(args.only)
    calls_graph = st.capture(only=args.only) if args.only is None else None

    with ClockSampler(torch.cuda.current_device()) as clk:
        ms = time_graph(graph, args.steps, args.warmup, world)
        calls_ms = time_graph(calls_graph, args.steps, args.warmup, world) if calls_graph is not None else None
    clocks = clk.summary()
    ms = max_over_ranks(ms, world)
    if plan is not None:
        assert g.nvfp4_device_status(plan.buffer, clear=False)[0] == g.NVFP4_OK, "a stream wait gave up"

    # end to end: pinned host inputs -> device, graph, device -> pinned host outputs
    xs, ys = st.host_io()
    h2d = sum(h.numel() * h.element_size() for _, h in xs)
    d2h = sum(h.numel() * h.element_size() for _, h in ys)
    stream = torch.cuda.current_stream()

    def e2e_step():
        for d, h in xs:
            d.copy_(h, non_blocking=True)
        graph.replay()
        for d, h in ys:
            h.copy_(d, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    step_bytes = st.step_bytes(args.only)
    value = world * step_bytes / (ms * 1e-3) / 1e9
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9
    # the dominant kernel is the whole step's single launch: its algorithmic
    # bytes per launch over its CUDA-event time on the replay stream
    achieved = step_bytes / (ms * 1e-3) / 1e9
    traffic = read_traffic(f"stream_kernel {args.workload}")
    calls = None
    if calls_ms is not None:
        cg = step_bytes / (calls_ms * 1e-3) / 1e9
        calls = {"what": "the same step as separate calls (prep + main kernel per call, PDL-chained, "
                         "one CUDA graph)", "ms": calls_ms, "gbs": cg, "frac": cg / hbm_peak,
                 "launches_per_step": st.launches_per_step()}
    streams = chains = None
    if not args.no_streams and args.only is None and world == 1:
        streams, chains = more_streams(dev, st, args, hbm_peak)

    prefill = prefill_tflops(dev) if not args.no_prefill else None
    ingest = ingest_gbs(dev) if not args.no_ingest else None
    fp6 = fp6_measure(dev) if not args.no_fp6 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "layer": st.shape.name, "tokens_N": st.N, "only": args.only,
                       "layers": st.n_layers, "weight_bytes_per_step": st.weight_bytes(),
                       "algorithmic_bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (rotating layers)", "graph": "one CUDA graph per step",
                       "tokens_per_s_per_stream": world * st.N / (ms * 1e-3),
                       "frac_of_8TBs": value / world / 8000.0},
            "roofline": {"bound": "hbm", "kernel": "stream_kernel (the step's product list, one launch)",
                         "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak if hbm_peak else None, "traffic": traffic,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s",
                         "timing": "CUDA events around graph replays of the launch on the replay stream"},
            "calls": calls,
            "streams": streams,
            "chain": chains,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "prefill": prefill,
            "ingest": ingest,
            "fp6": fp6,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
