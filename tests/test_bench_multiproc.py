"""The benchmark's multi-rank timing plumbing on CPU: two `gloo` ranks.

Replicas only: each rank runs its own sequences, and the job's number is the
units of all ranks over the slowest rank's time (max all-reduce).  The
reference arm runs on rank 0 only.  CPU only.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 25.0][rank]
        dist.barrier()
        ms = bench.max_over_ranks(local_ms, world)
        out[rank] = (ms, bench.job_rate(100, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_units():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 25.0
    assert rate == pytest.approx(2 * 100 / 0.025)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(64, 1, 1000.0) == 64.0


def test_reference_arm_is_silent_on_other_ranks(capsys):
    class A:
        steps, warmup = 1, 0
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""
