"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

Each rank runs its own replica of the workload (sequences and heads are
independent, so there is no data-path collective); the only collective is the
max-reduction of the per-rank timings, and the job throughput counts every
rank's work against that slowest time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank               # rank 1 is the slow one
        worst = bench.reduce_max(my_ms)
        value = bench.job_throughput(world, 8192, worst)
        w, r, lr = bench.dist_setup()
        results[rank] = (worst, value, w, r, lr)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert set(res) == {0, 1}
    for rank, (worst, value, w, r, lr) in res.items():
        assert worst == 15.0                     # both ranks see the slowest rank's time
        assert value == pytest.approx(2 * 8192 / 15e-3)
        assert (w, r, lr) == (2, rank, rank)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 0
    bench.run_reference(A())                     # returns without work or output
    assert capsys.readouterr().out == ""
