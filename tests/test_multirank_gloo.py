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


def _bench(args, env=None):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    e = {k: v for k, v in os.environ.items()
         if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    e.update(env or {})
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], env=e,
                         capture_output=True, text=True, timeout=240)
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    return res.returncode, lines, res.stderr


def test_bench_gpus_two_starts_two_replica_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (gloo
    here, the stub arm standing in for the timed GPU region) and prints one
    line whose totals cover both ranks."""
    rc, lines, err = _bench(["--gpus", "2", "--stub", "--steps", "5", "--warmup", "3"])
    assert rc == 0, err
    assert len(lines) == 1, lines
    line = lines[0]
    assert line["stub"] is True and line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["rows_total"] == 2 * 64 * 5
    # the slowest rank (rank 1 sleeps 40 ms) sets the whole-job time
    assert line["max_rank_seconds"] >= 0.04
    assert abs(line["value"] - line["rows_total"] / line["max_rank_seconds"]) < 1e-6 * line["value"]


def test_bench_refuses_gpus_that_disagree_with_world_size():
    rc, lines, _ = _bench(["--gpus", "2", "--stub", "--steps", "1", "--warmup", "3"],
                          env={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc != 0 and not lines
