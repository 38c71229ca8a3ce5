"""bench.py's multi-rank host logic on two gloo ranks (CPU): the job time is
the slowest rank's, and the whole-job GB/s counts every rank's bytes."""

import os
import socket

import pytest
import torch.distributed as td
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(local_ms)
        gbs = bench.whole_job_gbps(10 ** 9, world, ms)
        out[rank] = (ms, gbs)
    finally:
        td.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, gbs = res[0]
    assert ms == 5.0
    assert gbs == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.whole_job_gbps(6_700_500_000, 1, 1000.0) == pytest.approx(6.7005)
