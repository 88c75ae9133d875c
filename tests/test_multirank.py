"""The N > 1 bench path on CPU with gloo: every rank runs its own replica, the
reported time is the slowest rank's, the rate counts all ranks' units, and the
reference arm runs on rank 0 only."""

import contextlib
import io
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 + rank)
        rate = bench.whole_job_rate(917504, 100, world, mx)
        ws, rk, lr = bench.dist_setup()

        class A:
            steps, warmup = 5, 3
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(A)
        q.put((rank, mx, rate, ws, rk, lr, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate, ws, rk, lr, printed in out:
        assert mx == 11.0                                    # the slowest rank
        assert rate == pytest.approx(917504 * 100 * 2 / 11.0)
        assert (ws, rk, lr) == (2, rank, rank)
        if rank != 0:
            assert printed == ""                             # reference arm: rank 0 only


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(10, 4, 1, 2.0) == 20.0
