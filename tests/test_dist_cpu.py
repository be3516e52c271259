"""The N > 1 host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The path needs no collective (each rank runs its own independent grids, i.e.
weak scaling over batch elements); bench.py only uses a barrier and a
max-over-ranks reduction of the timed duration, and the reference arm runs on
rank 0 alone.  These are exercised here without a GPU.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.0 + rank, world)  # rank r "took" 1 + r seconds
        # reference arm: only rank 0 produces a line
        class A:
            warmup = 0
            steps = 0
            workload = "tiny_shell"

        ref = bench.bench_reference(A, world, rank) if rank != 0 else "rank0"
        q.put((rank, t, ref))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_reference_rank_gating():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # max over ranks is the slowest rank's time on every rank
    assert res[0][1] == pytest.approx(2.0) and res[1][1] == pytest.approx(2.0)
    # non-zero ranks of the reference arm do no work and print nothing
    assert res[1][2] is None
