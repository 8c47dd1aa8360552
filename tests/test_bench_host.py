"""Host logic of the benchmark's multi-process path, on CPU with gloo ranks:
the timed region is the slowest rank's, and the reported value counts every
rank's bytes over it; the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 10.0 - rank]  # rank-dependent timings
        got = bench.reduce_max(local)
        value = bench.whole_job_gbs(world, 2e9, 5, got[0])
        ref_line = bench.run_reference(type("A", (), {"m": None, "warmup": 0, "steps": 0})(),
                                       bench.WORKLOADS["single_token"]) if rank > 0 else "skip"
        q.put((rank, got, value, ref_line))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_with_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, ref_line in results:
        assert got == [2.0, 10.0]                      # max over ranks, element-wise
        assert value == pytest.approx(2 * 2e9 * 5 / 2.0 / 1e9)
        if rank > 0:
            assert ref_line is None                    # reference arm: rank 0 only


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_gbs(1, 150e6, 10, 1e-3) == pytest.approx(1500.0)
    assert bench.layer_bytes(5120, 17408, 1) == 3 * 5120 * 17408 * 0.5625 + 4 * 5120
