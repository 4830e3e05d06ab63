"""bench.py's multi-rank bookkeeping on CPU: world size 2 over gloo.  Each
rank reports its own elapsed time; every rank must see the maximum, and the
whole-job value is all ranks' units over that maximum (replicas, weak
scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    env = bench.dist_env()
    local = 1.0 + rank              # rank 1 is the slow one
    bench.barrier()
    mx = bench.max_over_ranks(local, device="cpu")
    value = bench.whole_job_value(units_per_rank=10.0, world=world, max_seconds=mx)
    q.put((rank, env, mx, value))
    dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, mx, value in results:
        assert env == (rank, 2, rank)
        assert mx == 2.0                 # max over ranks, seen by every rank
        assert value == pytest.approx(10.0 * 2 / 2.0)


def test_single_process_defaults():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_value(4.0, 1, 2.0) == 2.0
