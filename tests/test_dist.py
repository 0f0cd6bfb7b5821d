"""Multi-rank host logic of bench.py (replicas; max over ranks) on 2 gloo ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 1.0 + rank  # rank 1 is the slowest
    m = bench.max_over_ranks(elapsed, world)
    value, ms = bench.aggregate(m, tokens_per_rank_step=1000, steps=4, world=world)
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, m, value, ms))


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, value, ms in res:
        assert m == 2.0  # max over ranks
        assert value == 1000 * 4 * 2 / 2.0  # all ranks' tokens / slowest rank's time
        assert ms == 500.0
