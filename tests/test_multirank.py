"""The N > 1 path of the benchmark on CPU (gloo, world size 2): every rank
runs the same per-GPU expert shard, the timed region is the slowest rank's,
and the reported value is the whole job's throughput.  No GPU is used."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.slowest_rank_ms(times[rank], dist, "cpu")
        out[rank] = (ms, bench.job_throughput(1e12, ms, world))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_the_job_total():
    world, times = 2, [3.0, 5.0]
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, times, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 5.0
    assert value == pytest.approx(world * 1e12 / 5e-3 / 1e12)


def test_single_process_keeps_its_own_time():
    assert bench.slowest_rank_ms(4.0, None, "cpu") == 4.0
    assert bench.job_throughput(2e12, 1.0, 1) == pytest.approx(2000.0)
