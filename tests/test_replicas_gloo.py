"""Multi-GPU runs of bench.py are independent replicas (the path shards with no
collective): each rank times its own copy of the step, the step time is the slowest
rank's, and the throughput is the sum over ranks. This checks that host logic with a
two-rank gloo process group on the CPU."""

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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.9, 1.3][rank]
    ms = bench.max_over_ranks(local_ms, torch.device("cpu"))
    value = bench.replica_throughput(1_000_000, ms, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, value))


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [1.3, 1.3]
    expect = 2 * 1_000_000 / 1.3e-3 / 1e9
    assert all(abs(o[2] - expect) < 1e-9 for o in out)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import torch

    import bench

    assert bench.max_over_ranks(2.5, torch.device("cpu")) == 2.5
    assert bench.replica_throughput(10**9, 1000.0, 1) == pytest.approx(1.0)
