"""The benchmark's multi-rank aggregation on CPU: two gloo ranks, each with
its own time, report the units of both ranks over the slower rank's time."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, units, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        rate, ms = bench.job_rate(times[rank], units, dist, "cpu")
        out[rank] = (rate, ms)
    finally:
        dist.destroy_process_group()


def test_job_rate_is_all_units_over_slowest_rank():
    mp = pytest.importorskip("torch.multiprocessing")
    world, units = 2, 16384
    times = [40.0, 55.0]  # ms per rank
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, units, out), nprocs=world, join=True)
        res = dict(out)
    want_ms = max(times)
    for rank in range(world):
        rate, ms = res[rank]
        assert ms == want_ms
        assert rate == pytest.approx(units * world / (want_ms / 1000.0))


def test_job_rate_single_rank():
    import bench
    rate, ms = bench.job_rate(50.0, 1000)
    assert ms == 50.0 and rate == pytest.approx(20000.0)
