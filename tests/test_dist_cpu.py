"""The multi-process path of bench.py on the CPU (gloo, world size 2): the
products have no exchange step, so N GPUs run N replicas; what the ranks
share is the barrier and the max-over-ranks time that the JSON line uses."""
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        slowest = bench.max_over_ranks(world, 10.0 + 5.0 * rank)
        # the reference arm: rank 0 alone runs and prints; the others do nothing
        args = types.SimpleNamespace(workload="ter_gemv", steps=1, warmup=0)
        ref = bench.run_reference(args, world, rank) if rank != 0 else "skipped"
        q.put((rank, slowest, ref))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 15.0 for g in got)   # both ranks report the slower rank's time
    assert got[1][2] is None                 # non-zero ranks print no reference line
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(1, 3.5) == 3.5
