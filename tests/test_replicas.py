"""The N > 1 bench path on CPU: world-size-2 gloo ranks run independent replicas,
barrier around the timed region, and take the maximum time over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    results[rank] = bench.reduce_max(local_ms, w)
    bench.barrier(w)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == 15.0


def test_single_process_needs_no_group():
    import bench

    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)  # no process group: a no-op


def test_job_value_sums_replicas_over_slowest_rank():
    # value = world * bytes / max_ms: two replicas of 1 GB in 1 ms (slowest) -> 2000 GB/s
    world, kvb, ms = 2, 1_000_000_000, 1.0
    assert world * kvb / (ms * 1e-3) / 1e9 == pytest.approx(2000.0)
