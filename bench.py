#!/usr/bin/env python3
"""Benchmark of the batched Muon step on GB300.

A step is one full ``muon_step_batched`` call (momentum + look-ahead + norm,
10-iteration hybrid Newton–Schulz, scale + decoupled weight decay) over one
batch of synthetic input.  The default workload is the largest one, the
32-layer dense-transformer matrix set (hidden 4096, FFN 14336; per layer
q, o 4096x4096, k, v 1024x4096, gate, up 14336x4096, down 4096x14336; bf16 W
and G, fp32 momentum, 6.98 B params), grouped by shape into batched
Newton–Schulz chains, with Gaussian grads (sigma 1e-3) plus rank-8 spikes;
spectral scale, mu 0.95, lr 2.7e-4, wd 0.1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense|moe|stack|single|heads|adamw]

--workload adamw times the AdamW partition instead (muon_adamw_step over the
dense 32-layer model's embedding, output head and norm scales: 1.05 B params).

N > 1 runs one process per GPU: under torchrun (RANK / WORLD_SIZE set), or,
launched plainly with --gpus N, through bench.py's own spawner.  Each rank
updates its own copy of the workload (matrices are independent units: weak
scaling, no collective on the data path).  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "Muon-step params/s; Newton–Schulz TFLOP/s vs GB300 bf16 dense peak"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# default timed steps: the dense and MoE steps take 0.4-0.6 s each
DEFAULT_STEPS = {"dense": 60, "moe": 100}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 60 dense, 100 moe, 300 otherwise: about a minute or less)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["stack", "single", "heads", "dense", "moe", "adamw"],
                    default="dense")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="stack / single / heads / adamw: seconds of oracle work in cpu_baseline")
    ap.add_argument("--cpu-per-group", type=int, default=2,
                    help="dense / moe: matrices per shape group the oracle is timed on "
                         "(0: no cpu_baseline, for profiling runs)")
    ap.add_argument("--prof-steps", type=int, default=50)
    ap.add_argument("--layers", type=int, default=32,
                    help="dense: layers of the matrix set (fewer: a small case, e.g. for ncu)")
    ap.add_argument("--experts", type=int, default=256,
                    help="moe: experts of the set (fewer: a small case, e.g. for ncu)")
    ap.add_argument("--merge", type=int, choices=[0, 1], default=0,
                    help="dense / moe: groups of one wide shape share a Newton–Schulz chain")
    ap.add_argument("--prec", choices=["bf16", "x3"], default="bf16",
                    help="Newton–Schulz precision: bf16 (default) or split-bf16 (MUON_NS_BF16X3)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.workload, 300)
    return args


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# workloads (host-generated, seeded)
# ---------------------------------------------------------------------------
def build_workload(name: str, rank: int):
    import workloads
    if name == "stack":
        st = workloads.stacked(seed=1 + 1000 * rank)
        grads = [st.grad(t) for t in range(st.steps)]
        return dict(kind="stack", W=st.W, M=st.M, grads=grads,
                    desc=dict(workload="stack: 64 x bf16 1024x1024, fp32 momentum, 5-step grad cycle",
                              matrices=64, rows=1024, cols=1024, w_dtype="bf16", g_dtype="bf16",
                              m_dtype="fp32", schedule="8x(3.4445,-4.775,2.0315)+2x(2,-1.5,0.5)",
                              scale="spectral", seed=1))
    if name == "single":
        s = workloads.single_matrix(seed=rank)
        return dict(kind="single", W=s.W[None], M=s.M[None], grads=[s.G[None]],
                    desc=dict(workload="single: fp32 256x512 with rank-4 spike", matrices=1,
                              rows=256, cols=512, w_dtype="fp32", g_dtype="fp32", m_dtype="fp32",
                              scale="spectral", seed=0))
    h = workloads.split_heads(seed=2 + 1000 * rank)
    return dict(kind="heads", W=h.W, M=h.M, grads=[h.G], n_heads=h.n_heads, head_dim=h.head_dim,
                desc=dict(workload="heads: QKV 4096 x (32 x 128) bf16 split per head",
                          matrices=32, rows=4096, cols=128, w_dtype="bf16", g_dtype="bf16",
                          m_dtype="fp32", scale="spectral", seed=2))


def set_desc(name: str, layers: int = 32, experts: int = 256) -> dict:
    if name == "dense":
        return dict(workload=f"dense: {layers} layers x {{q,o 4096^2; k,v 1024x4096; gate,up "
                             f"14336x4096; down 4096x14336}}", matrices=layers * 7,
                    w_dtype="bf16", g_dtype="bf16", m_dtype="fp32", scale="spectral", seed=3,
                    grads="Gaussian 1e-3 + rank-8 spike")
    return dict(workload=f"moe: {experts} experts x {{up 2048x7168, down 7168x2048}}",
                matrices=2 * experts, w_dtype="bf16", g_dtype="bf16", m_dtype="fp32",
                scale="spectral", seed=4, grads="1e-3 * Student-t(3)")


def draw_set(name: str, rank: int, dev, layers: int = 32, experts: int = 256):
    """A multi-GB set drawn on the device: {member name: (W [B,r,c], G, M)}."""
    import workloads
    if name == "dense":
        return workloads.dense_layers(seed=3 + 1000 * rank, layers=layers, device=dev)
    return workloads.moe_experts(seed=4 + 1000 * rank, experts=experts, device=dev)


def device_sets(name: str, rank: int, dev, layers: int = 32, experts: int = 256):
    """Multi-GB sets drawn on the device: {shape name: (W [B,r,c], G, M)}."""
    return draw_set(name, rank, dev, layers, experts), set_desc(name, layers, experts)


def set_groups(m, sets):
    """One group per shape (muon_group_by_shape), every matrix of the set."""
    mats, descs = [], []
    for nm, (W, G, M) in sets.items():
        for b in range(W.shape[0]):
            mats.append((nm, b))
            descs.append((W.shape[1], W.shape[2], W.shape[2], m.MUON_BF16, m.MUON_BF16, 0))
    gid, ng = m.muon_group_by_shape(descs, 0)
    groups = []
    for g in range(ng):
        mem = [mats[i] for i in range(len(mats)) if gid[i] == g]
        groups.append(m.Group([sets[nm][0][b] for nm, b in mem], [sets[nm][1][b] for nm, b in mem],
                              [sets[nm][2][b] for nm, b in mem]))
    return groups


def make_groups(m, wl, Wd, Md, Gd):
    if wl["kind"] == "heads":
        return [[m.Group.split_head(Wd, g, Md, wl["n_heads"], wl["head_dim"])] for g in Gd]
    return [[m.Group.stacked(Wd, g, Md)] for g in Gd]


def n_params(wl):
    return int(wl["W"].numel())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"muon_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = [n for k, n in enumerate(names) if any(r[5 + k].lower() == "active" for r in rows)]
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": float(rows[0][2]),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                                   default=None),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample
# ---------------------------------------------------------------------------
def oracle_sample(wl, seconds: float, min_units: int = 1):
    import numpy as np
    import oracle
    W = wl["W"]
    G = wl["grads"][0]
    M = wl["M"]
    hp = oracle.MuonHyper()
    if wl["kind"] == "heads":
        hd = wl["head_dim"]
        mats = [(W[:, h * hd:(h + 1) * hd], G[:, h * hd:(h + 1) * hd], M[:, h * hd:(h + 1) * hd])
                for h in range(wl["n_heads"])]
        hp.fan_out_axis = 1
    else:
        mats = [(W[b], G[b], M[b]) for b in range(W.shape[0])]
    done, params, t0 = 0, 0, time.perf_counter()
    while done < min_units or (time.perf_counter() - t0 < seconds and done < len(mats)):
        w, g, mm = mats[done % len(mats)]
        oracle.muon_step(w.float().numpy().astype(np.float64), g.float().numpy().astype(np.float64),
                         mm.numpy().astype(np.float64), hp)
        done += 1
        params += w.numel()
    dt = time.perf_counter() - t0
    return params / dt, done, dt


def shape_groups(sets) -> dict:
    """{(rows, cols): [(name, index), ...]}: the matrices of a device-drawn set
    by shape (the groups muon_group_by_shape forms), in order of first
    appearance."""
    out = {}
    for nm, (W, _, _) in sets.items():
        key = (int(W.shape[1]), int(W.shape[2]))
        out.setdefault(key, []).extend((nm, b) for b in range(W.shape[0]))
    return out


def oracle_matrix_seconds(sets, nm: str, b: int) -> float:
    """Wall time of one float64 oracle Muon step on matrix b of set member nm
    (the host copies are made before the clock starts)."""
    import numpy as np
    import oracle
    W, G, M = sets[nm]
    w, g, mm = (x[b].float().cpu().numpy().astype(np.float64) for x in (W, G, M))
    t0 = time.perf_counter()
    oracle.muon_step(w, g, mm, oracle.MuonHyper())
    return time.perf_counter() - t0


def extrapolate(counts: dict, seconds: dict) -> tuple:
    """Whole-set oracle time from per-shape samples: sum over shapes of the
    shape's matrix count x its mean sampled time per matrix.
    counts {(r, c): matrices}, seconds {(r, c): [sampled seconds, ...]}.
    Returns (params/s, extrapolated seconds per step)."""
    params = sum(r * c * n for (r, c), n in counts.items())
    total = sum(n * (sum(seconds[k]) / len(seconds[k])) for k, n in counts.items())
    return params / total, total


def oracle_sample_sets(sets, per_group: int):
    """Oracle on `per_group` matrices of every shape group of a device-drawn
    set, extrapolated to the whole set by the groups' matrix counts (the cost
    per parameter grows with the Gram size, so every shape is timed)."""
    groups = shape_groups(sets)
    secs = {k: [oracle_matrix_seconds(sets, nm, b) for nm, b in mem[:max(1, per_group)]]
            for k, mem in groups.items()}
    value, total = extrapolate({k: len(v) for k, v in groups.items()}, secs)
    timed = sum(sum(v) for v in secs.values())
    sample = (", ".join(f"{len(secs[k])} of {len(groups[k])} {k[0]}x{k[1]}" for k in groups) +
              f" (one Muon step each, float64 NumPy, {timed:.1f} s); whole-set time "
              f"extrapolated by each shape's matrix count: {total:.0f} s per step")
    return value, sample


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest `value` over all ranks (a no-op for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(steps: int, params_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job params/s: every rank updates params_per_rank per step."""
    return world * steps * params_per_rank / (ms_max / 1e3)


def reference_line(args, value: float, dt: float, desc: dict, sample: str) -> dict:
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": desc,
            "cpu_baseline": {"value": value, "unit": "params/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def step_plan(n_groups: int, steps: int, cheapest: int) -> list:
    """Shape groups the oracle runs in each timed step of the reference arm:
    every group at least once over the run (one matrix each), the remaining
    steps on the cheapest group; with fewer steps than groups a step takes
    several."""
    if steps >= n_groups:
        return [[i] if i < n_groups else [cheapest] for i in range(steps)]
    return [list(range(i, n_groups, steps)) for i in range(steps)]


def run_reference_sets(args):
    """Reference arm on a device-drawn set: each step times the oracle on whole
    matrices of one layer's (expert's) draw of the set, per step_plan; the
    params/s is the whole set's, extrapolated from the per-shape times by each
    shape's matrix count."""
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    small = draw_set(args.workload, 0, dev, layers=1, experts=1)
    groups = shape_groups(small)
    keys = list(groups)
    scale = args.layers if args.workload == "dense" else args.experts
    counts = {k: len(groups[k]) * scale for k in keys}
    cost = lambda k: min(k) ** 2 * max(k)
    cheapest = min(range(len(keys)), key=lambda i: cost(keys[i]))
    for _ in range(args.warmup):
        nm, b = groups[keys[cheapest]][0]
        oracle_matrix_seconds(small, nm, b)
    secs = {k: [] for k in keys}
    nxt = {k: 0 for k in keys}
    t0 = time.perf_counter()
    for grp in step_plan(len(keys), args.steps, cheapest):
        for gi in grp:
            k = keys[gi]
            nm, b = groups[k][nxt[k] % len(groups[k])]
            nxt[k] += 1
            secs[k].append(oracle_matrix_seconds(small, nm, b))
    dt = time.perf_counter() - t0
    value, total = extrapolate(counts, secs)
    sample = ("per step one matrix (float64 NumPy oracle Muon step), every shape group at least "
              "once, the other steps on the cheapest: " +
              ", ".join(f"{len(secs[k])} x {k[0]}x{k[1]}" for k in keys) +
              f"; whole-set time extrapolated by each shape's matrix count: {total:.0f} s")
    print(json.dumps(reference_line(args, value, dt, set_desc(args.workload, args.layers,
                                                                args.experts), sample)),
          flush=True)
    return 0


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    if args.workload in ("dense", "moe"):
        return run_reference_sets(args)
    wl = build_workload(args.workload, 0)
    per_step = 120.0 / max(1, args.steps + args.warmup)   # whole run ~2 min (>= 1 matrix/step)
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0)
    t0 = time.perf_counter()
    params = units = 0
    for _ in range(args.steps):
        v, n, dt = oracle_sample(wl, min(per_step, 10.0))
        params += v * dt
        units += n
    dt = time.perf_counter() - t0
    value = params / dt
    rows, cols = wl["desc"]["rows"], wl["desc"]["cols"]
    sample = f"{units} matrices of {rows}x{cols} over {args.steps} steps (float64 NumPy oracle)"
    print(json.dumps(reference_line(args, value, dt, wl["desc"], sample)), flush=True)
    return 0


def code_only(text: str) -> str:
    """C++/CUDA source without comments and blank lines (the files hashed hold
    no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(files=("ns_gemm.cu", "ptx.cuh")):
    """sha256 (first 16 hex) of the kernel sources' code, comments aside: the
    committed DRAM-traffic summaries hold the hash of the code they were
    captured on."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "newton_schulz_02_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def read_traffic(kernel: str, summary="ns_gemm_traffic_stack.json", files=("ns_gemm.cu", "ptx.cuh")):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", summary)
    if not summary or not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash(files):
        return None
    e = d.get("kernels", {}).get(kernel)
    if not e:
        return None
    return e.get("dram_bytes_per_launch_full_workload")


def pick_peak(peaks: dict, timed_s: float) -> tuple:
    """Tensor peak for the roofline: the sustained measurement (a seconds-long
    loop under the power cap) for kernels timed inside a timed region of a
    second or more, the burst one for a short region."""
    if timed_s >= 1.0:
        return peaks["bf16_tflops_sustained"], "sustained"
    return peaks["bf16_tflops"], "burst"


def chain_memory_model(elems: float, iters: int, w_bytes: int, avg_s: float, hbm_gbs: float,
                       dram_bytes) -> dict:
    """The on-chip chain against the memory bound of an unfused Newton-Schulz
    chain over the same matrices: every iteration reads the bf16 iterate
    twice (Gram and update) and writes it once, 6 B per element, and the
    last update reads and writes W.  `dram_bytes` is what ncu measured per
    launch (or None)."""
    model = elems * (6 * iters + 2 * w_bytes)
    gbs = model / avg_s / 1e9
    return {"model": "unfused chain: bf16 X read twice and written once per iteration, "
                     "W read and written once",
            "elements_per_launch": elems, "iterations": iters,
            "alg_bytes_per_launch": model, "gbs": gbs, "frac_of_measured_copy": gbs / hbm_gbs,
            "dram_bytes_per_launch": dram_bytes}


def pinned_like(tensors):
    """Pinned host copies (uninitialised) of `tensors`, carved out of one
    pinned buffer."""
    import torch
    sizes = [t.numel() * t.element_size() for t in tensors]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    buf = torch.empty(max(1, o), dtype=torch.uint8, pin_memory=True)
    return [buf[a:a + n].view(t.dtype).view(t.shape) for a, n, t in zip(offs, sizes, tensors)]


def e2e_leg(m, stream, groups_of, grads, W_list, hp, ws, sched, n_e, world, dev, barrier):
    """End to end through host buffers, pipelined the way a training loop fed
    from host memory runs: step i's gradients (pinned host -> one of two
    device slots, on a copy stream) upload while step i - 1 computes, and step
    i's W leaves for pinned host memory from a device snapshot (one of two, so
    that a slow download never holds up the next snapshot) taken right after
    the step, while step i + 1 computes.  Every step's uploads and downloads
    lie inside the timed region (the first upload waits for its start, its end
    waits for the last download); each step's status word is saved on the
    device and all are checked at the end.  The first upload (pipeline fill)
    and the last download (drain) are timed as well: they are paid once per
    run, so their share falls with the number of steps.
    grads: per step of the input cycle, the list of gradient tensors;
    groups_of(list of gradient tensors) -> the step's muon groups."""
    import torch
    Gh = []
    for gl in grads:
        hs = pinned_like(gl)
        for h, g in zip(hs, gl):
            h.copy_(g)
        Gh.append(hs)
    slots = [[torch.empty_like(g) for g in grads[0]] for _ in range(2)]
    egs = [groups_of(sl) for sl in slots]
    Wsnap = [[torch.empty_like(w) for w in W_list] for _ in range(2)]
    Wh = pinned_like(W_list)
    status_word = ws[:4].view(torch.int32)
    flags_d = torch.zeros(n_e, dtype=torch.int32, device=dev)
    flags_h = torch.empty(n_e, dtype=torch.int32).pin_memory()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_g = [torch.cuda.Event() for _ in range(n_e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e)]
    for i in range(2):
        for d, h in zip(slots[i], Gh[i % len(Gh)]):
            d.copy_(h, non_blocking=True)
        m.muon_step_batched(egs[i], hp, ws, sched)
    torch.cuda.synchronize()
    barrier()
    timing = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    e0, fill_end, drain_start, drain_end, e1 = timing
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        e0.record(stream)
        for i in range(n_e):
            slot = i % 2
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(e0 if i < 2 else ev_done[i - 2])  # slot free again
                for d, h in zip(slots[slot], Gh[i % len(Gh)]):
                    d.copy_(h, non_blocking=True)
                ev_g[i].record(s_h2d)
                if i == 0:
                    fill_end.record(s_h2d)
            stream.wait_event(ev_g[i])
            m.muon_step_batched(egs[slot], hp, ws, sched)
            flags_d[i:i + 1].copy_(status_word)
            if i > 1:
                stream.wait_event(ev_out[i - 2])  # this snapshot buffer has left for the host
            for d, w in zip(Wsnap[slot], W_list):
                d.copy_(w)
            ev_done[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[i])
                if i == n_e - 1:
                    drain_start.record(s_d2h)
                for h, d in zip(Wh, Wsnap[slot]):
                    h.copy_(d, non_blocking=True)
                ev_out[i].record(s_d2h)
        s_d2h.wait_event(ev_out[n_e - 1])
        drain_end.record(s_d2h)
        stream.wait_event(ev_out[n_e - 1])
        flags_h.copy_(flags_d, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if int(flags_h.abs().sum()) != 0:
        raise RuntimeError("device status set during the end-to-end steps")
    P = sum(w.numel() for w in W_list)
    return {"value": job_value(n_e, P, world, e_ms), "unit": "params/s",
            "h2d_bytes_per_step": int(sum(g.numel() * g.element_size() for g in slots[0])),
            "d2h_bytes_per_step": int(sum(w.numel() * w.element_size() for w in Wh) + 4),
            "steps": n_e, "ms_per_step": e_ms / n_e, "wall_s": round(wall, 4),
            "fill_ms": round(e0.elapsed_time(fill_end), 3),
            "drain_ms": round(drain_start.elapsed_time(drain_end), 3),
            "clocks": clk.summary(),
            "path": "pinned host G -> device (copy stream, overlapping the previous step), "
                    "muon_step_batched, W snapshot on the device (two buffers) -> pinned "
                    "host (copy stream, overlapping the next step); each step's status "
                    "word saved on the device and checked after the last step"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import newton_schulz_02_gb300 as m

    world, rank, local = dist_setup(args)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m.load_library()
    peaks, peak_src = load_peaks()

    sets = None
    if args.workload in ("dense", "moe"):
        sets, desc = device_sets(args.workload, rank, dev, args.layers, args.experts)
        groups = [set_groups(m, sets)]
        P = int(sum(W.numel() for W, _, _ in sets.values()))
        wl = {"kind": args.workload, "sets": sets, "desc": desc}
        names = list(sets)

        def groups_of(gl):
            return set_groups(m, {nm: (sets[nm][0], g, sets[nm][2]) for nm, g in zip(names, gl)})
        step_grads = [[sets[nm][1] for nm in names]]
        W_list = [sets[nm][0] for nm in names]
    else:
        wl = build_workload(args.workload, rank)
        Wd = wl["W"].to(dev)
        Md = wl["M"].to(dev)
        Gd = [g.to(dev) for g in wl["grads"]]
        groups = make_groups(m, wl, Wd, Md, Gd)
        P = n_params(wl)

        def groups_of(gl):
            return make_groups(m, wl, Wd, Md, gl)[0]
        step_grads = [[g] for g in Gd]
        W_list = [Wd]
    hp = m.hparams()
    sched = None
    merge = args.merge == 1 and args.workload in ("dense", "moe")
    if args.prec == "x3" or merge:
        sched = m.muon_ns_hybrid_schedule()
        if args.prec == "x3":
            sched.prec = m.MUON_NS_BF16X3
        sched.merge_groups = 1 if merge else 0
    ws = m.workspace(m.muon_step_workspace_size(groups[0], sched), device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(args.warmup):
        m.muon_step_batched(groups[i % len(groups)], hp, ws, sched)
    code, flags = m.muon_get_status(ws)
    if code != m.MUON_OK or flags:
        raise RuntimeError(f"device status {code} flags {flags:#x} after warm-up")

    # Timed region: K steps back to back, no per-kernel events (those would sit
    # between dependent kernels and stop them overlapping); launches counted.
    m.muon_profile_reset()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            m.muon_step_batched(groups[i % len(groups)], hp, ws, sched)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = start.elapsed_time(stop)
    clocks = clk.summary()
    launches = int(sum(v["launches"] for v in m.muon_profile_query().values()))
    code, flags = m.muon_get_status(ws)
    if code != m.MUON_OK or flags:
        raise RuntimeError(f"device status {code} flags {flags:#x} after timed steps")
    # Per-kernel pass: the same steps again with a CUDA event pair recorded on
    # the launching stream around every kernel (roofline and kernel table).
    prof_steps = max(1, min(args.steps, args.prof_steps, 5 if sets is not None else args.prof_steps))
    m.muon_profile_reset()
    m.muon_profile_enable(True)
    torch.cuda.synchronize()
    for i in range(prof_steps):
        m.muon_step_batched(groups[i % len(groups)], hp, ws, sched)
    torch.cuda.synchronize()
    m.muon_profile_enable(False)
    prof = m.muon_profile_query()
    ms = max_over_ranks(ms, world, dev)
    value = job_value(args.steps, P, world, ms)

    # ---- per-kernel roofline (event-timed on the launching stream) --------
    gemm = {k: prof[k] for k in ("ns_gram", "ns_poly", "ns_gram_poly", "ns_update", "ns_chain")
            if k in prof and prof[k]["launches"]}
    ns_ms = sum(v["total_ms"] for v in gemm.values())
    ns_flops = sum(v["alg_flops"] for v in gemm.values())
    ns_tflops = ns_flops / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else None
    timed = {k: v for k, v in prof.items() if v["launches"] and v["total_ms"] > 0}
    dom = max(timed, key=lambda k: timed[k]["total_ms"])
    d = timed[dom]
    avg_s = d["total_ms"] / d["launches"] / 1e3
    timing = f"event pair per launch, {prof_steps} profiled steps after the timed region"
    # the committed DRAM counters were taken in the default configuration
    # (bf16 precision, one chain per group): other configurations report none
    traffic_file = (f"ns_gemm_traffic_{args.workload}.json"
                    if args.prec == "bf16" and not merge else "")
    if dom.startswith("ns_"):
        per_launch = d["alg_flops"] / d["launches"]
        achieved = per_launch / avg_s / 1e12
        peak, peak_kind = pick_peak(peaks, ms / 1e3)
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "timing": timing,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "frac_burst_peak": achieved / peaks["bf16_tflops"],
                "frac_sustained_peak": achieved / peaks["bf16_tflops_sustained"],
                "alg_flops_per_launch": per_launch, "avg_launch_ms": avg_s * 1e3,
                "traffic": read_traffic(dom, traffic_file),
                "peak_source": f"{peak_src} bf16 {peak_kind} (timed region {ms / 1e3:.2f} s)"}
    else:
        per_launch = d["alg_bytes"] / d["launches"]
        achieved = per_launch / avg_s / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "timing": timing, "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": None, "alg_bytes_per_launch": per_launch,
                "avg_launch_ms": avg_s * 1e3, "peak_source": f"{peak_src} copy"}
    if dom == "ns_chain":
        sc = sched if sched is not None else m.muon_ns_hybrid_schedule()
        iters = sum(sc.stages[i].steps for i in range(sc.n_stages))
        w_bytes = (sets[names[0]][0] if sets is not None else wl["W"]).element_size()
        roof["memory_model"] = chain_memory_model(P * prof_steps / d["launches"], iters, w_bytes,
                                                  avg_s, peaks["hbm_gbs"], roof["traffic"])
    kernels = {}
    for k, v in timed.items():
        e = {"launches": v["launches"], "total_ms": round(v["total_ms"], 4),
             "share": round(v["total_ms"] / sum(x["total_ms"] for x in timed.values()), 4)}
        if v["alg_flops"]:
            e["tflops"] = round(v["alg_flops"] / (v["total_ms"] / 1e3) / 1e12, 2)
        if v["alg_bytes"]:
            e["gbs"] = round(v["alg_bytes"] / (v["total_ms"] / 1e3) / 1e9, 1)
            e["hbm_frac_of_measured"] = round(e["gbs"] / peaks["hbm_gbs"], 3)
        kernels[k] = e
    # ---- the elementwise pass before Newton–Schulz (momentum, look-ahead,
    # norm partials) against HBM, at the minimal byte count: G + M read and
    # written + X written once (12 B per bf16-G parameter); the library's own
    # count adds the iterate's 2-byte residual plane
    elementwise = None
    if "prepare" in timed:
        pe = timed["prepare"]
        g_bytes = 4 if args.workload == "single" else 2
        min_bytes = (g_bytes + 8 + 2) * P * prof_steps
        gbs = min_bytes / (pe["total_ms"] / 1e3) / 1e9
        elementwise = {"kernel": "prepare", "bound": "hbm", "bytes_per_param": g_bytes + 10,
                       "gbs": gbs, "frac_of_measured_copy": gbs / peaks["hbm_gbs"],
                       "frac_of_8tbs": gbs / 8000.0,
                       "library_count": {"bytes_per_param": g_bytes + 12,
                                         "gbs": kernels["prepare"]["gbs"],
                                         "frac_of_measured_copy":
                                             kernels["prepare"]["hbm_frac_of_measured"]}}

    # ---- end to end: host buffers, copies inside the timed region ------------
    e2e = None
    if args.e2e_steps > 0:
        n_e = args.e2e_steps if sets is None else max(3, min(args.e2e_steps, 20))
        e2e = e2e_leg(m, stream, groups_of, step_grads, W_list, hp, ws, sched, n_e, world, dev,
                      barrier)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not (sets is not None and args.cpu_per_group <= 0):
        if sets is not None:
            cpu_v, sample = oracle_sample_sets(sets, args.cpu_per_group)
        else:
            cpu_v, cpu_n, cpu_dt = oracle_sample(wl, args.cpu_seconds)
            sample = (f"{cpu_n} matrices of {wl['desc']['rows']}x{wl['desc']['cols']}, one Muon "
                      f"step each, float64 NumPy, {cpu_dt:.1f} s")
        cpu = {"value": cpu_v, "unit": "params/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample}
    desc = dict(wl["desc"])
    desc["ns_precision"] = {"bf16": "bf16 (MUON_NS_BF16)",
                            "x3": "split-bf16 (MUON_NS_BF16X3, three products per GEMM)"}[args.prec]
    if sets is not None:
        desc["merge_groups"] = bool(merge)
    desc.update(parallelism=f"replicas x{world} (independent matrices, no collective)",
                l2={"stack": "inputs larger than L2: per step 128 MiB G + 128 MiB W + 256 MiB M "
                             "+ 768 MiB workspace",
                    "dense": f"inputs larger than L2 (about {P * 8 / 1e9:.0f} GB of W, G, M)",
                    "moe": f"inputs larger than L2 (about {P * 8 / 1e9:.0f} GB of W, G, M)"}.get(
                    wl["kind"], "small workload (L2-resident between steps)"))
    out = {"metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded, drawn on the device)" if sets is not None
                   else "synthetic (seeded, drawn on the host)", "config": desc,
           "ns_tflops": ns_tflops,
           "ns_frac_of_bf16_peak": ns_tflops / peaks["bf16_tflops"] if ns_tflops else None,
           "roofline": roof, "elementwise": elementwise, "kernels": kernels,
           "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
           "peaks": dict(peaks, source=peak_src)}
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# AdamW partition (muon_adamw_step)
# ---------------------------------------------------------------------------
ADAMW_METRIC = "AdamW-step params/s (AdamW partition of the dense 32-layer model)"
ADAMW_DESC = dict(workload="adamw: dense 32-layer model's AdamW partition: embedding and head "
                           "128256x4096, 65 norm scales of 4096", params=2 * 128256 * 4096 + 65 * 4096,
                  w_dtype="bf16", g_dtype="bf16", moments="fp32", beta1=0.9, beta2=0.95,
                  eps=1e-20, weight_decay=0.1, seed=5,
                  l2="inputs larger than L2 (12.6 GB of W, G, m, v)")


def adamw_oracle_sample(W, G, M, V, seconds: float):
    """Oracle AdamW on consecutive 2^20-element slices of the embedding until
    `seconds` have passed (host copies outside the timing)."""
    import numpy as np
    from oracle import adamw_ref
    n = 1 << 20
    flat = [x.view(-1) for x in (W, G, M, V)]
    done = params = 0
    spent = 0.0
    while done < 1 or spent < seconds:
        lo = (done * n) % (flat[0].numel() - n)
        w, g, mm, vv = (x[lo:lo + n].float().cpu().numpy().astype(np.float64) for x in flat)
        t0 = time.perf_counter()
        adamw_ref.adamw_step(w, g, mm, vv, adamw_ref.AdamWHyper(t=3))
        spent += time.perf_counter() - t0
        done += 1
        params += n
    return params / spent, done, spent


def run_adamw(args):
    import torch
    import torch.distributed as dist

    import newton_schulz_02_gb300 as m
    import workloads

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        if rank != 0:
            return 0
        torch.manual_seed(5)
        n = 1 << 24
        W = (torch.randn(n) * 0.02).to(torch.bfloat16)
        G = (torch.randn(n) * 1e-3).to(torch.bfloat16)
        M, V = torch.zeros(n), torch.zeros(n)
        per = 120.0 / max(1, args.steps + args.warmup)
        t0 = time.perf_counter()
        params = units = 0
        for _ in range(args.steps):
            v, k, dt = adamw_oracle_sample(W, G, M, V, min(per, 10.0))
            params += v * dt
            units += k
        dt = time.perf_counter() - t0
        value = params / max(dt, 1e-9)
        sample = f"{units} slices of 2^20 elements over {args.steps} steps (float64 NumPy oracle)"
        print(json.dumps({"impl": "reference", "metric": ADAMW_METRIC, "value": value,
                          "unit": "params/s", "n_gpus": args.gpus, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic", "config": ADAMW_DESC,
                          "cpu_baseline": {"value": value, "unit": "params/s",
                                           "cores": cpu_cores(), "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m.load_library()
    peaks, peak_src = load_peaks()
    part = workloads.dense_adamw_partition(seed=5 + 1000 * rank, device=dev)
    W, G, M, V = part["W"], part["G"], part["m"], part["v"]
    groups = m.adamw_groups(W, G, M, V, wd_mask=part["wd_mask"])
    P = int(sum(w.numel() for w in W))
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    t = 1
    for _ in range(args.warmup):
        m.muon_adamw_step(groups, m.adamw_hparams(t=t), flags)
        t += 1
    torch.cuda.synchronize()
    m.muon_profile_reset()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            m.muon_adamw_step(groups, m.adamw_hparams(t=t), flags)
            t += 1
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = start.elapsed_time(stop)
    launches = int(sum(v["launches"] for v in m.muon_profile_query().values()))
    if int(flags.item()) != 0:
        raise RuntimeError(f"device flags {int(flags.item()):#x}")
    prof_steps = max(1, min(args.steps, args.prof_steps))
    m.muon_profile_reset()
    m.muon_profile_enable(True)
    for _ in range(prof_steps):
        m.muon_adamw_step(groups, m.adamw_hparams(t=t), flags)
        t += 1
    torch.cuda.synchronize()
    m.muon_profile_enable(False)
    d = m.muon_profile_query()["adamw"]
    ms = max_over_ranks(ms, world, dev)
    value = job_value(args.steps, P, world, ms)
    avg_s = d["total_ms"] / d["launches"] / 1e3
    per_launch = d["alg_bytes"] / d["launches"]
    achieved = per_launch / avg_s / 1e9
    roof = {"kernel": "adamw", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "traffic": read_traffic("adamw", "adamw_traffic.json", ("adamw.cu",)),
            "alg_bytes_per_launch": per_launch, "avg_launch_ms": avg_s * 1e3,
            "timing": f"event pair per launch, {prof_steps} profiled steps after the timed region",
            "peak_source": f"{peak_src} copy"}

    e2e = None
    if args.e2e_steps > 0:
        # pinned host gradients in, updated W out, every step; pipelined as in
        # the Muon leg: uploads into two device gradient slots on one copy
        # stream, W snapshots on the device, downloads on another copy stream
        steps = max(1, min(args.e2e_steps, 5))
        Gh = [g.cpu().pin_memory() for g in G]
        Wh = [torch.empty(w.shape, dtype=w.dtype).pin_memory() for w in W]
        Gslots = [G, [torch.empty_like(g) for g in G]]
        Wsnap = [torch.empty_like(w) for w in W]
        sgroups = [m.adamw_groups(W, gs, M, V, wd_mask=part["wd_mask"]) for gs in Gslots]
        s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev_g = [torch.cuda.Event() for _ in range(steps)]
        ev_done = [torch.cuda.Event() for _ in range(steps)]
        ev_out = [torch.cuda.Event() for _ in range(steps)]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            slot = i % 2
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(e0 if i < 2 else ev_done[i - 2])
                for g, gh in zip(Gslots[slot], Gh):
                    g.copy_(gh, non_blocking=True)
                ev_g[i].record(s_h2d)
            stream.wait_event(ev_g[i])
            m.muon_adamw_step(sgroups[slot], m.adamw_hparams(t=t), flags)
            t += 1
            if i > 0:
                stream.wait_event(ev_out[i - 1])
            for ws_, w in zip(Wsnap, W):
                ws_.copy_(w)
            ev_done[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[i])
                for wh, ws_ in zip(Wh, Wsnap):
                    wh.copy_(ws_, non_blocking=True)
                ev_out[i].record(s_d2h)
        stream.wait_event(ev_out[steps - 1])
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        if int(flags.item()) != 0:
            raise RuntimeError(f"device flags {int(flags.item()):#x}")
        e2e = {"value": job_value(steps, P, world, e_ms), "unit": "params/s",
               "h2d_bytes_per_step": int(sum(g.numel() * g.element_size() for g in G)),
               "d2h_bytes_per_step": int(sum(w.numel() * w.element_size() for w in W)),
               "steps": steps, "path": "pinned host G -> device (copy stream, overlapping the "
                                        "previous step), muon_adamw_step, W snapshot on the "
                                        "device -> pinned host (copy stream, overlapping the "
                                        "next step)"}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    cpu_v, cpu_n, cpu_dt = adamw_oracle_sample(W[0], G[0], M[0], V[0], args.cpu_seconds)
    desc = dict(ADAMW_DESC, parallelism=f"replicas x{world} (independent tensors, no collective)")
    out = {"metric": ADAMW_METRIC, "value": value, "unit": "params/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded Gaussian weights and grads)", "config": desc,
           "roofline": roof,
           "kernels": {"adamw": {"launches": d["launches"], "total_ms": round(d["total_ms"], 4),
                                 "share": 1.0, "gbs": round(achieved, 1),
                                 "hbm_frac_of_measured": round(achieved / peaks["hbm_gbs"], 3)}},
           "cpu_baseline": {"value": cpu_v, "unit": "params/s", "cores": cpu_cores(),
                            "kind": "oracle",
                            "sample": f"{cpu_n} slices of 2^20 embedding elements, one AdamW "
                                      f"step each, float64 NumPy, {cpu_dt:.1f} s"},
           "e2e": e2e, "gpu_launches": launches, "clocks": clk.summary(),
           "peaks": dict(peaks, source=peak_src)}
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, target, args):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    sys.exit(target(args) or 0)


def spawn_ranks(n: int, target, args, timeout_s: float = 3600.0) -> int:
    """Run target(args) as n processes, one per rank (GPU), with the
    environment a torchrun launch gives them (RANK, LOCAL_RANK, WORLD_SIZE,
    MASTER_ADDR 127.0.0.1, a free MASTER_PORT).  Returns the first non-zero
    exit code, else 0."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, n, port, target, args)) for r in range(n)]
    for p in procs:
        p.start()
    rc = 0
    for p in procs:
        p.join(timeout_s)
        if p.exitcode is None:
            p.kill()
            p.join()
        code = p.exitcode if p.exitcode is not None else 1
        if code != 0 and rc == 0:
            rc = code
    return rc


def run(args) -> int:
    if args.workload == "adamw":
        return run_adamw(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


def main():
    args = parse()
    sys.path.insert(0, ROOT)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # launched plainly: one process per GPU from here (torchrun sets WORLD_SIZE)
        return spawn_ranks(args.gpus, run, args)
    return run(args)


if __name__ == "__main__":
    sys.exit(main())
