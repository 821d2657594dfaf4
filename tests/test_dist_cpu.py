"""The benchmark's multi-rank host logic, on CPU with gloo and two ranks: the
timing is the max over ranks, the value counts every rank's replica, and
only rank 0 does the reference arm's work."""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], dist, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0, 0.5]


def test_single_process_and_whole_job_value():
    assert bench.max_over_ranks([3.0, 4.0], None, "cpu") == [3.0, 4.0]
    f = 4.4e12
    assert bench.whole_job_tflops(1, f, 2.0) == pytest.approx(f / 2e-3 / 1e12)
    assert bench.whole_job_tflops(8, f, 2.0) == pytest.approx(8 * f / 2e-3 / 1e12)


def test_reference_arm_does_nothing_on_other_ranks(capsys):
    class Args:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
