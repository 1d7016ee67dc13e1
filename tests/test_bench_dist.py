"""The benchmark's multi-rank host logic on CPU: world size 2 over gloo
(ranks are independent replicas; the only communication is the barrier and
the reductions of timings and unit counts)."""

from __future__ import annotations

import io
import os
import socket
import sys
import contextlib
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    args = types.SimpleNamespace(world=world, rank=rank, local=rank)
    # the description our arm prints for the same workload
    config = bench.decode_workload_config(
        types.SimpleNamespace(world=world, batch=None, sets=None), "local_decode")
    bench.barrier(args)
    t = bench.max_over_ranks(args, 10.0 + rank)       # slowest rank wins
    u = bench.sum_over_ranks(args, 100.0 * (rank + 1))  # units add up
    # the reference arm: rank 0 prints one line, the others print nothing
    rargs = types.SimpleNamespace(world=world, rank=rank, local=rank, workload="local_decode",
                                  steps=2, warmup=0, ref_budget=0.01, gpus=world, batch=None,
                                  sets=None)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(rargs)
    q.put((rank, t, u, buf.getvalue().strip(), config))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reductions_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (r0, t0, u0, out0, config), (r1, t1, u1, out1, _) = res
    assert t0 == t1 == 11.0
    assert u0 == u1 == 300.0
    assert out1 == ""
    import json
    line = json.loads(out0)
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    # both arms describe the workload identically
    assert line["config"] == config
    assert line["n_gpus"] == 2
    # the time per step is the time spent (the per-step budget is 0.01 s and
    # at least one unit runs), not the budget
    assert 0 < line["ms_per_step"] < 5000
    assert line["cpu_baseline"]["cores"] == os.cpu_count()
    assert line["cpu_baseline"]["blas_threads"] >= 1
