"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2).

The prefill shards by replica only: every rank runs its own copy of the workload and nothing
is exchanged on the data path.  What crosses ranks is the timing: each rank's time is
max-reduced (the slowest replica sets the step time) and rank 0 reports the whole-job value
= world x work per replica / that time.  The reference arm runs on rank 0 alone.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        # rank r took (10 + r) ms and (1 + 2r) s of wall time
        ms, wall = bench.max_over_ranks([10.0 + rank, 1.0 + 2 * rank], "cpu")
        value = bench.weak_scaling_value(world, 5.0e12, ms)
        ref = bench.run_reference(None, rank) if rank != 0 else "rank0"
        out.put((rank, ms, wall, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, wall, value, ref in res:
        assert ms == 11.0 and wall == 3.0               # the maximum over both ranks
        assert value == pytest.approx(2 * 5.0e12 / 11.0e-3)
    assert res[1][4] is None                            # rank 1 does no reference work


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.5, 7.0], "cpu") == [3.5, 7.0]
    assert bench.weak_scaling_value(1, 8.0e12, 2.0) == pytest.approx(4.0e15)
