"""bench.py's multi-process plumbing on the CPU (gloo, world size 2): the
barrier and the max-over-ranks timing the replicas use, and the reference
arm doing its work on rank 0 only."""

import multiprocessing as mp
import os
import socket
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, _ = bench.dist_setup(world)
    slowest = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
    bench.barrier(dist)

    class Args:
        steps, warmup, gpus = 1, 3, world
    if r != 0:
        bench.run_reference(Args, r)   # returns at once: only rank 0 times the oracle
    out.put((r, w, slowest))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, 2, port, out)) for rank in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, 2, 20.0), (1, 2, 20.0)]
