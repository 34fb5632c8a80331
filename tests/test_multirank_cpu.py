"""Multi-process paths on the CPU (gloo, world size 2).

The BitLinear forward shards by output features: each rank holds a block of
rows of the packed weights (the per-matrix gamma is global) and a replica of
the quantised activations, and computes its own block of y with no exchange.
These tests check, with the oracle and two gloo ranks, that the concatenated
blocks equal the unsplit product bit for bit, and they exercise the
rank handling of bench.py (max over ranks, rank-0-only output) without a GPU.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank: int, world: int, port: int):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _row_shard_worker(rank: int, world: int, port: int, result_q, fmt: str = "2bit"):
    sys.path.insert(0, ROOT)
    import oracle
    import workloads

    _init(rank, world, port)
    try:
        wl = workloads.WORKLOADS["tiny"]
        W, X = workloads.layer_inputs(wl, 0)
        N, K = W.shape
        # gamma is a property of the whole matrix: every rank packs with the global gamma
        pack = oracle.pack_weights_tq5 if fmt == "tq5" else oracle.pack_weights
        fwd = oracle.forward_tq5 if fmt == "tq5" else oracle.forward
        packed, gamma = pack(W.numpy())
        xq, s = oracle.quant_act(workloads.x_as_f32_numpy(X))
        # uneven split on purpose (N = 256 -> 100 + 156 rows)
        bounds = [0, 100, N]
        lo, hi = bounds[rank], bounds[rank + 1]
        y_part, acc_part = fwd(packed[lo:hi], gamma, xq, s, K)
        pieces = [None] * world
        dist.all_gather_object(pieces, (lo, y_part, acc_part))
        if rank == 0:
            pieces.sort(key=lambda p: p[0])
            y_cat = np.concatenate([p[1] for p in pieces], axis=1)
            acc_cat = np.concatenate([p[2] for p in pieces], axis=1)
            y_ref, acc_ref = fwd(packed, gamma, xq, s, K)
            result_q.put((bool(np.array_equal(acc_cat, acc_ref)),
                          bool(np.array_equal(y_cat.view(np.uint32), y_ref.view(np.uint32)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt", ["2bit", "tq5"])
def test_row_sharded_forward_equals_unsplit_gloo(fmt):
    """both weight formats shard by output rows: a row block of the packed
    array is the packing of that row block"""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_row_shard_worker, args=(r, 2, port, q, fmt)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    acc_ok, y_ok = q.get(timeout=5)
    assert acc_ok, "concatenated int32 accumulators differ from the unsplit product"
    assert y_ok, "concatenated y differs from the unsplit product"


def _max_worker(rank: int, world: int, port: int, result_q):
    sys.path.insert(0, ROOT)
    import bench

    _init(rank, world, port)
    try:
        got = bench.max_over_ranks(dist, 1.5 + 2.0 * rank)
        result_q.put((rank, got))
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_bench_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the CPU (gloo) launch of the reference arm")
def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0
