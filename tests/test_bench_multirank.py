"""bench.py host logic on the CPU: on two gloo ranks the job time is the
slowest rank's and the whole-job GB/s counts every rank's bytes; the traffic
figure comes from an ncu summary only while its kernel source is unchanged."""

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


def test_profile_traffic_follows_the_source_the_summary_names(tmp_path, monkeypatch):
    """A committed ncu summary feeds the bench line's traffic only while the
    kernel source it names still has the recorded sha256; the captured bytes
    are scaled by the ratio of algorithmic bytes."""
    import hashlib

    import bench
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "decode_partition_x.md").write_text(
        f"source_sha256: {sha}   (k.cu at capture time)\n"
        "captured_traffic_bytes: 1010\ncaptured_algorithmic_bytes: 1000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("x", 2000.0) == 2020
    assert bench.profile_traffic("missing", 2000.0) is None
    src.write_text("kernel v2\n")                        # the kernel changed since the capture
    assert bench.profile_traffic("x", 2000.0) is None
