"""The N>1 bench path on CPU: two gloo ranks agree on the slowest rank's time
and on the whole-job rate (weak scaling: every rank runs its own batch, no
collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ranks = bench.Ranks(backend="gloo")
    try:
        ranks.barrier()
        seconds = 1.0 + rank              # rank 1 is the slow one
        slowest = ranks.max(seconds)
        rate = bench.aggregate(1000 * 10, ranks.world, slowest)
        q.put((rank, ranks.world, slowest, rate))
    finally:
        ranks.close()


def test_two_gloo_ranks_report_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, w, slowest, rate in got:
        assert w == world
        assert slowest == pytest.approx(2.0)
        assert rate == pytest.approx(1000 * 10 * world / 2.0)


def test_single_process_needs_no_process_group():
    import bench
    r = bench.Ranks()
    assert r.world == int(os.environ.get("WORLD_SIZE", "1")) and not r.pg or r.world > 1
    assert r.max(3.5) == 3.5
    assert bench.aggregate(75600 * 10, 1, 2.0) == pytest.approx(378000.0)
