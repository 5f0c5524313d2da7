"""The N > 1 host logic of bench.py on two gloo ranks (CPU): replicas draw
distinct uniforms, the timing is the maximum over ranks and the throughput
counts every rank's cycles."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    secs = 1.0 + rank          # rank 1 is the slow one
    t = bench.max_over_ranks(secs)
    value, tmax = bench.aggregate(10, [t], ws)
    bench.barrier()
    q.put((r, ws, local, t, value, bench.rank_seed(2, r)))
    dist.destroy_process_group()


def test_two_rank_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[3] == pytest.approx(2.0) for r in res)   # max over ranks
    assert all(r[4] == pytest.approx(2 * 10 / 2.0) for r in res)
    assert res[0][5] != res[1][5]                          # distinct seeds
