"""World-size-2 gloo test (CPU) of the benchmark's multi-rank logic: each rank
gets an independent replica of the workload (weak scaling, no data-path
collective) and the reported time is the maximum over ranks."""
from __future__ import annotations

import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench._dist_init()
    wl = bench.rank_workload("tiny", r, w)
    k, _ = __import__("bit_quantized_kv_gb300.workloads", fromlist=["x"]).sequence_kv(wl, 0, "cpu")
    bench._barrier(w)
    t = bench._max_over_ranks(10.0 + r, w)
    q.put((r, wl.seed, float(k.float().sum()), t, wl.B, wl.Hq))
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, k0, t0, b0, h0), (r1, s1, k1, t1, b1, h1) = res
    assert (r0, r1) == (0, 1)
    assert s0 != s1 and k0 != k1            # independent replicas
    assert (b0, h0) == (b1, h1)             # same per-rank shape (weak scaling)
    assert t0 == t1 == 11.0                 # max over ranks
