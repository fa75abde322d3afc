"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks report different times,
both see the slowest, and the whole-job throughput counts every rank's shard."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, dist, "cpu")
        out[rank] = (t, bench.job_gparams_per_s(1_000_000, 10, t, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0
    assert res[0][1] == pytest.approx(2 * 1_000_000 * 10 / 2.0 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_gparams_per_s(2_000_000_000, 1, 2.0, 1) == 1.0
