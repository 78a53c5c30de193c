"""The benchmark's multi-GPU arithmetic (replicas only) on two CPU ranks over gloo: every rank
sees the slowest rank's time, and the whole-job value counts every rank's bytes."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
    dist.barrier()
    q.put((rank, ms, bench.whole_job_gbs(1e9, world, ms)))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in res:
        assert ms == 15.0                       # the slower rank's time, on every rank
        assert gbs == pytest.approx(2 * 1e9 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.whole_job_gbs(2e9, 1, 1.0) == pytest.approx(2000.0)
