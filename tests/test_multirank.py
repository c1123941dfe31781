"""bench.py's multi-GPU path is replicas with host-side aggregation only: a
barrier, then the max of the ranks' times and the sum of their work.  This
checks that aggregation with two gloo ranks on the CPU, and that the
reference arm lets every rank but 0 exit at once."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world)
    bench.barrier(dist)
    elapsed = [3.0, 5.0][rank]
    work = [10.0, 32.0][rank]
    out[rank] = (bench.max_over_ranks(dist, elapsed), bench.sum_over_ranks(dist, work))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_work():
    import torch.multiprocessing as mp
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert out[0] == (5.0, 42.0) and out[1] == (5.0, 42.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "build_case", lambda name: called.append(name))
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "1"]) == 0
    assert called == []


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1) is None
    assert bench.max_over_ranks(None, 2.5) == 2.5 and bench.sum_over_ranks(None, 4.0) == 4.0
