"""The multi-GPU form of the bench is replicas only (no exchange on the data
path): each rank runs the whole request on its GPU, the job time is the
slowest rank's, and the rate is the units of all ranks over that time.  The
cross-rank step runs here on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [4.0 + rank, 30.0 - 3.0 * rank]          # rank 0 slower at decode, 1 at prefill
        t_pre, t_dec = bench.max_over_ranks(mine, world, dist, "cpu")
        dist.barrier()
        q.put((rank, t_pre, t_dec, bench.job_rates(t_pre, t_dec, world, 4000, 500)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_pre, t_dec, (pre, dec) in out:
        assert (t_pre, t_dec) == (5.0, 30.0)             # elementwise max over ranks
        assert pre == pytest.approx(2 * 4000 / 5e-3)
        assert dec == pytest.approx(2 * 500 / 30e-3)


def test_single_rank_unchanged():
    assert bench.max_over_ranks([1.5, 2.5], 1, None, "cpu") == [1.5, 2.5]
    assert bench.job_rates(2.0, 10.0, 1, 4000, 500) == pytest.approx((2e6, 5e4))
