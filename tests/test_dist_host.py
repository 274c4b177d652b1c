"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): replicas
exchange only timing maxima, never data; the max over ranks is elementwise."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    d = bench.Dist(world)
    try:
        d.barrier()
        # each rank reports its own timings; every rank gets the max
        mine = [1.0 + rank, 10.0 - rank, 3.0 * (rank + 1)]
        got = d.max(mine)
        q.put((rank, got, d.world, d.rank))
    finally:
        d.close()


@pytest.mark.timeout(120)
def test_dist_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=100) for _ in range(world)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, got, w, r in results:
        assert w == world and r == rank
        assert got == [2.0, 10.0, 6.0]


def test_dist_single_rank_is_identity(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist(1)
    assert d.world == 1 and d.pg is None
    assert d.max([1.5, 2.5]) == [1.5, 2.5]
    d.barrier()
    d.close()
