"""The multi-GPU path of the benchmark is independent replicas (the boundary
engine has no exchange step): each rank times its own events and rank 0
reports the events of all ranks over the slowest rank's time.  Checked here
with two gloo ranks on CPU; the reference arm prints on rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank 0 took 100 ms for its 8 events, rank 1 took 250 ms
        value, ms_max = bench.replica_value(100.0 if rank == 0 else 250.0, 8)
        q.put((rank, value, ms_max))
    finally:
        dist.destroy_process_group()


def test_replicas_aggregate_over_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, ms_max in got:
        assert ms_max == pytest.approx(250.0)
        assert value == pytest.approx(2 * 8 / 0.25)   # 16 events over the slowest rank's 0.25 s


def test_single_process_is_one_replica():
    sys.path.insert(0, ROOT)
    import bench
    value, ms_max = bench.replica_value(200.0, 10)
    assert ms_max == pytest.approx(200.0) and value == pytest.approx(50.0)


def test_reference_arm_prints_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, ref_units = 1, 0, 1
    assert bench.run_reference(A, 2, 1) is None
