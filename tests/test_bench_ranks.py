"""The multi-rank host logic of bench.py on the CPU: two gloo ranks, a
barrier, the max of the ranks' elapsed times and the sum of their units
(value = all ranks' units / the slowest rank's time, weak scaling)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, lr = bench.rank_info()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    t, u = bench.reduce_max_sum(dist, elapsed_s=0.5 + rank, units=100.0 * (rank + 1))
    q.put((r, w, t, u))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_aggregate(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, t, u) in enumerate(res):
        assert rank == r and w == world
        assert t == pytest.approx(0.5 + world - 1)
        assert u == pytest.approx(sum(100.0 * (k + 1) for k in range(world)))


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max_sum(None, 1.25, 7.0) == (1.25, 7.0)
