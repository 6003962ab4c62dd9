"""The multi-rank bench path on CPU: two gloo ranks (replicas).

Decode attention shards by sequence with no data-path collective, so
``bench.py --gpus N`` runs N replicas, each on its own batch; the only
cross-rank step is the timing: the slowest rank's time, and whole-job
throughput = the units all ranks processed / that time.  These tests run that
host logic (``bench.rank_info`` and ``bench.aggregate``) as two processes over
gloo on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, units, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.rank_info()
        elapsed, value = bench.aggregate(times[rank], units, w, dist)
        out.put((r, w, lr, elapsed, value))
    finally:
        dist.destroy_process_group()


def _run(times, units):
    world = len(times)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, units, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_replicas_take_the_slowest_rank():
    times = [0.010, 0.025]                     # rank 1 is slower
    units = 600e6                              # KV bytes one rank reads
    res = _run(times, units)
    assert [r[:3] for r in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, elapsed, value in res:        # every rank agrees
        assert elapsed == pytest.approx(0.025)
        assert value == pytest.approx(2 * units / 0.025)


def test_single_rank_needs_no_process_group():
    import importlib
    sys.path.insert(0, ROOT)
    bench = importlib.import_module("bench")
    elapsed, value = bench.aggregate(0.5, 10.0, 1)
    assert elapsed == 0.5 and value == pytest.approx(20.0)
