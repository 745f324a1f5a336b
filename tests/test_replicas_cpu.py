"""Multi-process plumbing of bench.py on CPU (gloo, world size 2).

The path does not shard: under torchrun every rank runs its own replica of
the layer stream, and the ranks only meet at the barriers around the timed
region and in the max-over-ranks of the step time.  These tests run that host
logic in two processes without a GPU.
"""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    try:
        bench.barrier(w)
        # each replica's step time differs; the job's time is the slowest
        t = bench.max_over_ranks(1.5 + rank, w)
        bench.barrier(w)
        out.put((r, w, local, t))
    finally:
        dist.destroy_process_group()


def test_two_replicas_barrier_and_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    results = sorted(q.get(timeout=5) for _ in range(world))
    for p in procs:
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == world for r in results)
    assert [r[2] for r in results] == [0, 1]
    assert all(r[3] == pytest.approx(1.5 + world - 1) for r in results)


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (1, 0, 0)
    assert bench.max_over_ranks(3.25, w) == 3.25
    bench.barrier(w)  # no-op


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched as two torchrun ranks: rank 0
    alone times the oracle and prints one JSON line; the other rank exits 0
    without work."""
    import json
    import subprocess
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
