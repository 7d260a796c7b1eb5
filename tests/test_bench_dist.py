"""bench.py's multi-rank host logic on CPU: two gloo ranks, each a replica with
its own batch; barrier, max-over-ranks timing and whole-job aggregation."""
import os

import pytest
import torch.multiprocessing as mp

import bench


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    seconds = 1.0 + rank          # the slower rank decides the time
    t_max = bench.max_over_ranks(seconds, w)
    value = bench.aggregate(1e12, t_max, w)  # 1e12 units per rank
    q.put((rank, t_max, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, value in out:
        assert t_max == 2.0
        assert value == pytest.approx(2 * 1e12 / 2.0)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(10.0, 2.0, 1) == 5.0
