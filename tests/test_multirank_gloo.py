"""Multi-rank host logic on CPU (gloo, world_size 2): rows shard across
replicas with no data-path collective; the bench's whole-job numbers take the
slowest rank's time and the sum of all ranks' rows."""

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
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, n = bench.aggregate_over_ranks(1.0 + rank, 100 * (rank + 1))
        q.put((rank, t, n, bench.dist_env()))
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, n, env in res:
        assert t == 2.0 and n == 300
        assert env == (rank, rank, 2)


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate_over_ranks(0.5, 64) == (0.5, 64)
