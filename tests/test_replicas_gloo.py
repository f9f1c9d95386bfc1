"""Multi-process path of bench.py on CPU: replicas only, so the one
collective is the max over ranks of the timed region.  Two gloo ranks with
different times must both see the slowest one, and the whole-job rate counts
every rank's units over that time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank           # rank 1 is the slower replica
        got = bench.replica_max_ms(ms, world, "cpu")
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_job_rate_counts_every_rank():
    import bench
    # 100 units per rank, 2 ranks, slowest rank 15 ms
    assert bench.job_rate(100, 2, 15.0) == pytest.approx(100 * 2 / 0.015)
    assert bench.replica_max_ms(12.5, 1, "cpu") == 12.5


def test_committed_traffic_record_matches_the_kernel_sources():
    """roofline.traffic comes from a committed ncu capture keyed to a hash of
    the sources the decode GEMV is built from; a source changed since the
    capture makes bench.py report null.  The committed record must match."""
    import bench
    assert bench.load_traffic(bench.DOMINANT) is not None
