"""The bench's host logic on CPU: two gloo ranks on 127.0.0.1 check the
cross-rank reduction of the timed region (max over ranks) and the whole-job
value, and that bench.py's own spawner starts one process per rank; the
reference arm does no work on ranks other than 0, on rank 0 prints one
contract line, and extrapolates a set's oracle time from every shape."""
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


def test_reference_arm_prints_the_contract_line(capsys):
    """Rank 0 of the reference arm times the float64 oracle on host cores and
    prints one JSON line carrying the keys of the bench contract."""
    import json

    class A:
        steps, warmup, gpus, workload = 2, 1, 1, "single"
    assert bench.run_reference(A()) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 1)
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["ms_per_step"] > 0 and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("single") and d["config"]["rows"] == 256
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "matrices of 256x512" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_clock_summary_parses_nvidia_smi_rows(tmp_path):
    """The clocks object is read from nvidia-smi's csv rows (noheader, nounits):
    median SM clock under load, the maximum, and every throttle reason seen."""
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    cs.proc = object()                       # stands for the sampler process
    rows = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1440, 2070, 1398.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1425, 2070, [N/A], 0x4, Not Active, Not Active, Not Active, Active",
            "garbage line"]
    open(cs.path, "w").write("\n".join(rows) + "\n")
    d = cs.summary()
    assert d["sm_mhz"] == 1440.0 and d["sm_max_mhz"] == 2070.0 and d["samples"] == 3
    assert d["reasons"] == ["sw_power_cap"] and d["power_w_max"] == 1398.0

    open(cs.path, "w").write("0, 1300, 2070, [N/A], 0x40, Not Active, Active, Not Active, Not Active\n")
    d = cs.summary()
    assert d["reasons"] == ["hw_thermal_slowdown"] and d["power_w_max"] is None


def test_traffic_is_reported_only_for_the_profiled_kernel_source(tmp_path):
    """roofline.traffic comes from a committed ncu summary only while the
    kernel source it was taken on is unchanged; otherwise it is null."""
    import json
    p = tmp_path / "traffic.json"
    entry = {"kernels": {"ns_gram_poly": {"dram_bytes_per_launch_full_workload": 123.0}}}
    p.write_text(json.dumps(dict(entry, source_hash=bench.kernel_source_hash())))
    assert bench.read_traffic("ns_gram_poly", summary=str(p)) == 123.0
    assert bench.read_traffic("ns_update", summary=str(p)) is None
    p.write_text(json.dumps(dict(entry, source_hash="0" * 16)))
    assert bench.read_traffic("ns_gram_poly", summary=str(p)) is None
    assert bench.read_traffic("ns_gram_poly", summary=str(tmp_path / "absent.json")) is None


def test_chain_memory_model_of_the_split_head_set():
    """The split_head set (32 heads of 4096 x 128, bf16 W, ten iterations)
    against an unfused chain's memory traffic: per head and iteration the
    128 x 4096 iterate is read by the Gram and by the update and written
    once; the last update reads and writes the head's W."""
    heads, n, m, iters = 32, 128, 4096, 10
    per_iter = heads * 3 * n * m * 2
    w_rmw = 2 * (4096 * 4096) * 2
    mm = bench.chain_memory_model(heads * n * m, iters, 2, 0.5e-3, 6795.1, 101e6)
    assert mm["alg_bytes_per_launch"] == iters * per_iter + w_rmw == 1_073_741_824
    assert abs(mm["gbs"] - 1_073_741_824 / 0.5e-3 / 1e9) < 1e-9
    assert abs(mm["frac_of_measured_copy"] - mm["gbs"] / 6795.1) < 1e-12
    assert mm["dram_bytes_per_launch"] == 101e6 and mm["iterations"] == 10


def test_kernel_hash_ignores_comments_only():
    """The traffic summaries are keyed to the kernel code: comments and blank
    lines do not change the hash, code does."""
    code = "int f(int x) {\n  return x + 1;  // one\n}\n"
    commented = "/* doc\n   more */\nint f(int x) {\n\n  return x + 1;  // another note\n}\n"
    changed = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_only(code) == bench.code_only(commented)
    assert bench.code_only(code) != bench.code_only(changed)


def _stub_step(args):
    """Stands for one rank's bench run: joins the gloo group the spawner's
    environment describes, reduces its timed region, rank 0 prints one line."""
    import json
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    assert int(os.environ["LOCAL_RANK"]) == rank and os.environ["MASTER_ADDR"] == "127.0.0.1"
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + rank, world)
    if rank == 0:
        print(json.dumps({"n_gpus": world, "ms": ms,
                          "value": bench.job_value(args.steps, 100, world, ms)}), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    return 0


def test_spawner_launches_one_process_per_rank(capfd):
    import argparse
    import json
    args = argparse.Namespace(steps=4, gpus=2)
    assert bench.spawn_ranks(2, _stub_step, args, timeout_s=120) == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["ms"] == 11.0
    assert d["value"] == pytest.approx(2 * 4 * 100 / 0.011)


def test_plain_launch_with_several_gpus_goes_through_the_spawner(monkeypatch):
    seen = {}
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "spawn_ranks", lambda n, target, args: seen.update(n=n) or 0)
    monkeypatch.setattr(bench, "run", lambda args: pytest.fail("ran in the launching process"))
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "3", "--steps", "2"])
    assert bench.main() == 0 and seen == {"n": 3}
    # under torchrun (WORLD_SIZE set) the process is already one rank
    monkeypatch.setenv("WORLD_SIZE", "3")
    monkeypatch.setattr(bench, "run", lambda args: 0)
    monkeypatch.setattr(bench, "spawn_ranks", lambda *a: pytest.fail("spawned under torchrun"))
    assert bench.main() == 0


def test_step_plan_covers_every_group():
    plan = bench.step_plan(4, 6, cheapest=1)
    assert plan == [[0], [1], [2], [3], [1], [1]]
    plan = bench.step_plan(4, 3, cheapest=1)       # fewer steps than groups
    assert sorted(g for step in plan for g in step) == [0, 1, 2, 3] and len(plan) == 3


def test_extrapolation_weights_shapes_by_count():
    counts = {(4, 8): 10, (16, 16): 2}
    secs = {(4, 8): [1.0, 3.0], (16, 16): [5.0]}
    v, total = bench.extrapolate(counts, secs)
    assert total == pytest.approx(10 * 2.0 + 2 * 5.0)
    assert v == pytest.approx((10 * 32 + 2 * 256) / total)


def test_reference_arm_on_a_set_prints_the_extrapolated_line(monkeypatch, capsys):
    """The set path of the reference arm on a tiny stand-in set (two shapes),
    so that it runs on CPU in seconds: one JSON line, every shape sampled."""
    import argparse
    import json

    import torch

    def tiny(name, rank, dev, layers=1, experts=1):
        g = torch.Generator().manual_seed(0)
        mk = lambda r, c: ((torch.randn(1, r, c, generator=g) * 0.02).to(torch.bfloat16),
                           (torch.randn(1, r, c, generator=g) * 1e-3).to(torch.bfloat16),
                           torch.zeros(1, r, c))
        return {"a": mk(16, 32), "b": mk(16, 32), "c": mk(48, 16)}
    monkeypatch.setattr(bench, "draw_set", tiny)
    args = argparse.Namespace(steps=3, warmup=1, gpus=1, workload="dense", layers=32,
                              experts=256)
    assert bench.run_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 3
    assert d["config"]["workload"].startswith("dense: 32 layers")
    assert "16x32" in d["cpu_baseline"]["sample"] and "48x16" in d["cpu_baseline"]["sample"]
    assert "extrapolated" in d["cpu_baseline"]["sample"]
