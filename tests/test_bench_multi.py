"""Host logic of bench.py's multi-GPU path, on CPU with world size 2 (gloo):
the job's time is the slowest rank's, and the value divides it over the
units of every rank (weak scaling; the decode path has no data-path
collective)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_timing(times[rank], world, torch.device("cpu"))
        q.put((rank, ms, bench.job_value(ms, 4, 2048, world)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [180.0, 196.0]
    procs = [ctx.Process(target=_rank, args=(r, 2, PORT, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [196.0, 196.0]
    assert res[0][2] == pytest.approx(196.0 / 4 * 1e3 / (2048 * 2))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_timing(12.5, 1, None) == 12.5
    assert bench.job_value(49.0, 1, 2048, 1) == pytest.approx(49.0e3 / 2048)


PORT = _free_port()
