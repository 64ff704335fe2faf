"""The N > 1 bench path on CPU: two gloo ranks on 127.0.0.1 check the
cross-rank reduction of the timed region (max over ranks) and the whole-job
value, and that the reference arm does no work on ranks other than 0."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    m = bench.max_over_ranks(ms, world)
    v = bench.job_value(4, 1000, world, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, v in got:
        assert m == 15.0
        assert v == pytest.approx(2 * 4 * 1000 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(10, 100, 1, 1000.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(bench, "build_workload", lambda *a, **k: pytest.fail("rank 1 did work"))

    class A:
        steps, warmup, gpus, workload = 2, 1, 2, "stack"
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
