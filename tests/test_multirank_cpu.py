"""Multi-process host logic of bench.py at world size 2 on CPU (gloo).

The path shards by requests with no exchange step, so every rank runs an
independent replica; what crosses ranks is only the timing reduction (max over
ranks) and the weak-scaling aggregate.  Both run here as two gloo ranks.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        slowest = bench.reduce_max(0.010 + 0.005 * rank, w)      # seconds per step on this rank
        value = bench.aggregate_throughput(32, w, slowest)
        dist.barrier()
        results.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(results.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == pytest.approx(0.015)
        assert value == pytest.approx(2 * 32 / 0.015)    # all ranks' tokens / slowest time


def test_single_rank_is_the_identity():
    import bench

    assert bench.reduce_max(0.25, 1) == 0.25
    assert bench.aggregate_throughput(32, 1, 0.5) == 64
