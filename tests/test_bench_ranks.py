"""The multi-rank bookkeeping of bench.py on CPU ranks (gloo, world size 2).

bench.py runs one replica of the decode step per GPU (the work shards by tile
rows, and a replica needs no exchange); the job's time is the slowest rank's
and its throughput counts every rank's bytes.  These tests run that
bookkeeping on two CPU processes.
"""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        ms = b.max_over_ranks(times[rank], world)
        dist.barrier()
        out[rank] = (ms, b.job_throughput(world, 275_251_200, 100, ms / 1e3))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_all_ranks_count():
    world, port = 2, _free_port()
    times = [4.0, 5.5]                              # ms per 100 steps on rank 0, rank 1
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 5.5
    expect = 2 * 275_251_200 * 100 / 5.5e-3 / 1e9
    assert res[0][1] == pytest.approx(expect) and res[1][1] == pytest.approx(expect)


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(3.25, 1) == 3.25
    assert b.job_throughput(1, 1e9, 10, 2.0) == pytest.approx(5.0)
