"""The N > 1 path of bench.py on CPU: world-size-2 `gloo` process groups.

The bench runs one independent replica of the layer per GPU (no collective
touches the data path); across ranks it only takes the slowest rank's time
(MAX all-reduce) and reports the whole-job rate.  These tests run that
aggregation on two CPU ranks with different local times, and check that the
reference arm does no work on ranks other than 0.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out_q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(torch, dist, local_ms[rank], world, torch.device("cpu"))
        rate = bench.whole_job_rate(world, 16384, 10, m)
        out_q.put((rank, m, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    world, port = 2, _free_port()
    local_ms = [7.5, 9.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, m, rate in res:
        assert m == max(local_ms)   # every rank sees the slowest rank's time
        assert rate == pytest.approx(world * 16384 * 10 / (max(local_ms) / 1e3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, None, 3.0, 1, torch.device("cpu")) == 3.0
    assert bench.whole_job_rate(1, 100, 4, 2.0) == pytest.approx(200000.0)


def test_reference_arm_only_on_rank_0(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    # rank 1 returns before touching the workload (the args are never read)
    assert bench.run_reference(None) is None
