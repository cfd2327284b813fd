"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1) run independent replicas and agree
on the barrier and on the max-over-ranks step time; no data-path collective exists."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    d = bench.Dist(backend="gloo")
    d.barrier()
    got = d.max(1.5 + rank)          # each rank's own step time
    d.barrier()
    q.put((rank, d.rank, d.world, got))
    d.close()


def test_two_gloo_ranks_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 0, 2, 2.5), (1, 1, 2, 2.5)]


def test_single_rank_is_identity():
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.max(3.25) == 3.25
    d.barrier()
