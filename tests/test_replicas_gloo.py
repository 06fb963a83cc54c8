"""The multi-GPU bench path is N independent replicas; its only cross-rank step is the
barrier and the max-over-ranks of the timed region.  Exercised here with two gloo ranks on
the CPU (no GPU, no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # Each replica reports its own timed region; the job's time is the slowest rank's.
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    q.put((rank, t))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
