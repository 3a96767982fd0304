"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, no GPU.

Each rank runs an independent replica (weak scaling); the whole-job rate is
all ranks' bytes over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ranks = bench.Ranks(backend="gloo")
    ranks.barrier()
    total, slowest, rate = bench.aggregate(100.0 * (rank + 1), 2.0 + rank, ranks)
    q.put((rank, ranks.world, total, slowest, rate))
    ranks.close()


@pytest.mark.parametrize("world", [2])
def test_aggregate_over_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, total, slowest, rate in out:
        assert w == world
        assert total == 300.0          # 100 + 200 bytes
        assert slowest == 3.0          # max(2, 3) seconds
        assert rate == 100.0


def test_single_rank_needs_no_process_group():
    import bench
    r = bench.Ranks()
    assert r.world == 1 and r.pg is None
    assert bench.aggregate(10.0, 2.0, r) == (10.0, 2.0, 5.0)
