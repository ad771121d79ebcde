"""The benchmark's multi-rank host logic with two gloo ranks on the CPU: the
job time is the slowest rank's, the value counts every rank's tokens, each
replica draws its own batch, and the reference arm runs on rank 0 only."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [12.5, 20.25][rank]          # rank 1 is the slow one
    t = bench.max_over_ranks(elapsed, world, "cpu")
    v = bench.job_tokens_per_s(128, world, 10, t)
    results[rank] = (t, v, bench.replica_seed(7, rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 20.25
    assert res[0][1] == res[1][1] == pytest.approx(128 * 2 * 10 / 20.25e-3)
    assert {res[0][2], res[1][2]} == {7, 8}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0     # returns before touching any data or device


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(128, 1, 100, 200.0) == pytest.approx(64000.0)
