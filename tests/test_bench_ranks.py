"""Multi-rank logic of bench.py on CPU: two gloo ranks, no GPU.

The bench times the same work on every rank, takes the slowest rank's time
and reports the tokens of all ranks over it (weak scaling, replicas of
independent heads); the step count is the smallest any rank picked; the
reference arm prints from rank 0 only.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        elapsed = bench.reduce_over_ranks(10.0 * (r + 1), dist.ReduceOp.MAX, "cpu", w)
        steps = int(bench.reduce_over_ranks(100 + 7 * r, dist.ReduceOp.MIN, "cpu", w))
        value = bench.job_throughput(1000, w, steps, elapsed)
        out[r] = (elapsed, steps, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        elapsed, steps, value = res[r]
        assert elapsed == 20.0          # the slowest rank's time
        assert steps == 100             # the smallest step count
        assert value == pytest.approx(1000 * world * 100 / 0.020)  # all ranks' tokens


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(3.5, None, "cpu", 1) == 3.5
    assert bench.job_throughput(512, 1, 10, 5.0) == pytest.approx(512 * 10 / 0.005)


def test_reference_arm_prints_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps = 1
        warmup = 0
        gpus = 2

    bench.run_reference(Args(), bench.workloads.WORKLOADS["c1"])
    assert capsys.readouterr().out == ""
