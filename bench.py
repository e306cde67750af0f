"""Benchmark of the W4A16 fused matrix multiply on GB300.

Default workload: the Llama-2-7B decode linears, symmetric group 128:
(K, N) in {4096x12288 QKV, 4096x4096 O, 4096x22016 gate+up, 11008x4096 down},
M in {1, 2, 4, 8, 16, 32}.  One step = the 24 matrix multiplies of that grid,
each reading its weights from HBM: every call of a step reads its own copy
of the layer's repacked weights (624 MB in all, more than two L2s), so no call
finds its weights in L2.  The step is captured once as a CUDA graph and
replayed.

Output: one JSON line (rank 0).  value = algorithmic bytes of the whole step
(codes + scales + X + Y) / step time, in GB/s, summed over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the CPU oracle (the plain fp64 definition) on a bounded
sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (ALL_CONFIGS, SPARSE_CONFIGS, Problem, make_activations,  # noqa: E402
                       make_sparse_weights, make_weights, seed_for)

METRIC = "W4A16 GEMM µs, HBM GB/s & TFLOP/s (% roofline) vs M; speedup over FP16 GEMM"
WORKLOAD_NAMES = {
    "7b-decode": "llama2-7b-decode-linears (K,N) in {4096x12288, 4096x4096, 4096x22016, 11008x4096}, "
                 "M in {1,2,4,8,16,32}, group 128, z=8",
    "single": "single GEMM M=16 K=4096 N=4096 group 128 z=8",
    "70b-decode": "llama2-70b batched decode (K,N) in {8192x10240, 8192x8192, 8192x57344, 28672x8192}, "
                  "M in {1,4,16,32,64,128}, group 128, z=8",
    "prefill": "prefill M in {1024,4096,8192} x (K,N) in {8192x8192, 8192x28672}, group 128, z=8",
    "sparse-7b-decode": "llama2-7b-decode-linears (K,N) in {4096x12288, 4096x4096, 4096x22016, 11008x4096} "
                        "with 2:4-sparse weights (sparse path), M in {1,2,4,8,16,32}, group 128, z=8",
    "asym-odd": "asymmetric zeros, group 128 and per-column, (K,N) in {2048x2048, 2048x5632, 5120x15360, "
                "13824x5120}, M in {1,16,48}",
}
L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a16_mixed_precision_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def kernel_names(problems) -> str:
    """The fused kernels a workload launches: the warp-level path for M <= 16,
    the tcgen05 path above (the library's default split); 2:4 weights: the
    sparse instantiation of the warp-level kernel at every M <= 32."""
    if any(p.sparse for p in problems):
        return "w4a16_small_m_kernel (2:4-sparse instantiation, mma.sp)"
    small = any(p.M <= 16 for p in problems)
    big = any(p.M > 16 for p in problems)
    return " + ".join(n for n, on in (("w4a16_small_m_kernel", small), ("w4a16_gemm_kernel", big)) if on)


def recorded_traffic(workload: str):
    """dram bytes per launch from a committed ncu capture, if the kernel sources
    have not changed since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_src") != kernel_source_digest():
        return None
    return e.get("dram_bytes_per_launch")


# ---- workload description (shared by both arms) ------------------------------------

def weight_bytes(K: int, N: int, g: int, asym: bool, sparse: bool) -> int:
    codes = K * N // 4 + K * N // 8 if sparse else K * N // 2
    return codes + (K // g) * N * 2 + ((K // g) * N // 2 if asym else 0)


def rotation(problems):
    """Weight rotation of a workload: per layer (K, N, group, asym), how many
    calls of a step use it, the number P of graph phases (steps between two
    reads of one weight copy) and the number of copies per layer, so that P
    steps stream more than two L2s and each per-problem table rotates through
    more than two L2s."""
    sparse = any(p.sparse for p in problems)
    layers = sorted({(p.K, p.N, p.group, p.asym) for p in problems})
    uses = {lk: sum(1 for p in problems if (p.K, p.N, p.group, p.asym) == lk) for lk in layers}
    step_wbytes = sum(weight_bytes(*lk, sparse) * uses[lk] for lk in layers)
    P = max(1, -(-2 * L2_BYTES // step_wbytes))
    copies = {lk: max(uses[lk] * P, -(-2 * L2_BYTES // weight_bytes(*lk, sparse)) + 1) for lk in layers}
    return layers, uses, P, copies


def workload_config(workload: str, problems) -> dict:
    """The `config` object of the JSON line: the same for the GPU arm and the
    reference arm (it depends on the workload only)."""
    sparse = any(p.sparse for p in problems)
    layers, uses, P, copies = rotation(problems)
    weight_copies_bytes = sum(weight_bytes(*lk, sparse) * copies[lk] for lk in layers)
    return {"workload": WORKLOAD_NAMES.get(workload, workload),
            "problems_per_step": len(problems), "graph_phases": P,
            "l2": f"inputs larger than L2: rotating weight copies ({weight_copies_bytes / 1e6:.0f} MB "
                  f"in all), each read once per {P} step(s), so no call finds its weights in L2",
            "timing": "step captured as a CUDA graph (one per rotation phase), replayed K times; "
                      "CUDA events on the replay stream",
            "step_bytes": sum(p.algorithmic_bytes() for p in problems),
            "step_flops": sum(p.flops() for p in problems)}


# ---- clocks --------------------------------------------------------------------

class ClockSampler:
    FIELDS = ["uuid", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            if self.uuid and self.uuid not in parts[0].lower():
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        used = inside if inside else [s for (_, s) in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in used if num(s[1]) is not None]
        smax = [num(s[2]) for s in used if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in used for i in range(4) if s[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(inside)}


# ---- distributed ------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def _dist_device():
    """Device of the tensors exchanged by the process group (CPU for gloo)."""
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def dist_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=_dist_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(step_bytes: int, ms_local: float, steps: int, world: int):
    """Whole-job throughput of `world` replicas that each ran `steps` steps of
    `step_bytes`: the slowest rank's time decides.  Returns (ms per step, GB/s)."""
    ms_per_step = dist_max(ms_local, world) / steps
    return ms_per_step, step_bytes * world / (ms_per_step * 1e-3) / 1e9


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- CPU oracle baseline ------------------------------------------------------------

def host_cores() -> int:
    """Cores this process may run on (its affinity mask, which a cgroup or
    taskset narrows), used both as the oracle's thread count and as the
    reported core count."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


class OracleSampler:
    """Times the CPU oracle (as it stands) on column samples of the workload.

    A sample of problem p = all M rows x `cols` random columns; its share of
    the algorithmic bytes is p.algorithmic_bytes() * cols / N."""

    def __init__(self, threads: int):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.threads = threads
        self.cache = {}
        self.sec_per_mk = None

    def inputs(self, p):
        if p.key not in self.cache:
            if p.sparse:
                Qp, S, Zp = make_sparse_weights(p.K, p.N, p.group, p.asym, seed_for(p.key))
                kc, ki, _ = self.oracle.sparse_compress(Qp, Zp, p.K, p.N, p.group)
                Qp = (kc, ki)
            else:
                Qp, S, Zp = make_weights(p.K, p.N, p.group, p.asym, seed_for(p.key))
            X = make_activations(p.M, p.K, seed_for(p.key) + 1)
            self.cache = {p.key: (X, Qp, S, Zp)}   # keep one problem's inputs at a time
        return self.cache[p.key]

    def product(self, p, X, Qp, S, Zp, idx, threads):
        """The oracle's product for this problem: the 2:4 form sums the kept terms only."""
        if p.sparse:
            return self.oracle.w4a16_sparse(X, Qp[0], Qp[1], S, Zp, p.group, p.N, idx=idx, threads=threads)
        return self.oracle.w4a16(X, Qp, S, Zp, p.group, p.N, idx=idx, threads=threads)

    def calibrate(self, p):
        X, Qp, S, Zp = self.inputs(p)
        t = time.perf_counter()
        self.product(p, X, Qp, S, Zp, np.arange(p.M) * p.N, 1)
        self.sec_per_mk = max((time.perf_counter() - t) / (p.M * p.K), 1e-10)

    def run(self, p, budget_s: float):
        """Returns (bytes credited, seconds, columns)."""
        if self.sec_per_mk is None:
            self.calibrate(p)
        X, Qp, S, Zp = self.inputs(p)
        cols = int(budget_s * self.threads / (self.sec_per_mk * p.M * p.K))
        cols = max(1, min(p.N, cols))
        rng = np.random.default_rng(seed_for(p.key))
        sel = np.sort(rng.choice(p.N, cols, replace=False))
        idx = (np.arange(p.M)[:, None] * p.N + sel[None, :]).ravel()
        t = time.perf_counter()
        self.product(p, X, Qp, S, Zp, idx, self.threads)
        dt = time.perf_counter() - t
        return p.algorithmic_bytes() * cols / p.N, dt, cols


def oracle_baseline(problems, budget_s: float, threads: int):
    """(GB/s, seconds, sample description) over every problem of the workload."""
    smp = OracleSampler(threads)
    tot_b = tot_s = 0.0
    cols = []
    for p in problems:
        b, s, c = smp.run(p, budget_s / len(problems))
        tot_b += b
        tot_s += s
        cols.append(c)
    desc = (f"all {len(problems)} problems of the workload, each: all M rows x {min(cols)}-{max(cols)} "
            f"random columns (of N); bytes credited = algorithmic bytes x sampled columns / N")
    return tot_b / tot_s / 1e9, tot_s, desc


def run_reference(args, problems, rank, world):
    if rank != 0:
        return
    threads = host_cores()
    smp = OracleSampler(threads)
    steps = args.steps + args.warmup
    budget = max(0.02, min(10.0, 90.0 / max(steps, 1)))
    # one step = one problem of the workload (cycling), a column sample sized to the budget;
    # steps walk the problems in order so consecutive steps reuse inputs
    order = sorted(range(len(problems)), key=lambda i: problems[i].key)
    tot_b = tot_s = 0.0
    cols = []
    for i in range(steps):
        p = problems[order[(i * len(problems)) // steps if steps >= len(problems) else i % len(problems)]]
        b, s, c = smp.run(p, budget)
        if i >= args.warmup:
            tot_b += b
            tot_s += s
            cols.append(c)
    value = tot_b / tot_s / 1e9
    desc = (f"each step: one problem of the workload (steps walk all {len(problems)}), all M rows x "
            f"{min(cols)}-{max(cols)} random columns; bytes credited = algorithmic bytes x columns / N")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / max(args.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(args.workload, problems),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- GPU arm -------------------------------------------------------------------------

def run_gpu(args, problems, rank, world, local):
    import torch

    import w4a16_mixed_precision_gb300 as w4
    from w4a16_mixed_precision_gb300 import build as cuda_build

    cuda_build.build()
    sparse = problems[0].sparse
    assert all(p.sparse == sparse for p in problems)
    call = w4.sparse_gemm_into if sparse else w4.gemm_into
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    # ---- weights: rotating copies so that no call finds its weights in L2 ----
    layers, uses, P, _ = rotation(problems)
    packed, dense_pw, _ = make_weight_copies(problems, dev, with_dense=sparse and not args.no_table)
    max_m = max(p.M for p in problems)
    ws = {lk: w4.Workspace(max_m, lk[0], lk[1], lk[2]) for lk in layers}
    xs = [torch.from_numpy(make_activations(p.M, p.K, seed_for(p.key))).to(dev) for p in problems]
    ys = [torch.empty((p.M, p.N), dtype=torch.float16, device=dev) for p in problems]
    plans = []  # per phase: (problem index, weight copy) in step order
    for c in range(P):
        seen = {lk: 0 for lk in layers}
        plan = []
        for i, p in enumerate(problems):
            lk = (p.K, p.N, p.group, p.asym)
            plan.append((i, c * uses[lk] + seen[lk]))
            seen[lk] += 1
        plans.append(plan)

    def step(plan):
        for i, c in plan:
            p = problems[i]
            lk = (p.K, p.N, p.group, p.asym)
            call(xs[i], packed[lk][c], ws[lk], ys[i])

    # eager warm-up (one-time host set-up happens outside the graphs)
    for plan in plans:
        step(plan)
    torch.cuda.synchronize()
    for lk in layers:
        assert w4.device_status(ws[lk]) == 0

    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for plan in plans:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(plan)
            graphs.append(g)
    torch.cuda.synchronize()

    step_bytes = sum(p.algorithmic_bytes() for p in problems)
    step_flops = sum(p.flops() for p in problems)

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    # clock soak: keep the GPU busy ~1 s before the timed region
    with torch.cuda.stream(stream):
        t_end = time.time() + (0.0 if args.no_soak else 1.0)
        while time.time() < t_end:
            for i in range(20):
                graphs[i % P].replay()
            stream.synchronize()
        for i in range(args.warmup):
            graphs[i % P].replay()
    torch.cuda.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            graphs[i % P].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    dist_barrier(world)
    torch.cuda.synchronize()
    time.sleep(0.25)
    sampler.stop()
    ms_per_step, value = aggregate_throughput(step_bytes, ev0.elapsed_time(ev1), args.steps, world)
    for lk in layers:
        assert w4.device_status(ws[lk]) == 0, "a kernel reported an expired wait"

    launches = len(problems)
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    clocks = sampler.summary(t_wall0 - 1.2, t_wall1)

    # ---- per-run table (outside the timed region): our kernel vs cuBLAS fp16 ----
    runs = []
    if not args.no_table:
        runs = per_run_table(problems, packed, ws, xs, ys, dev, peaks, call, dense_pw if sparse else None)

    # ---- end to end through the public API with host buffers ----
    e2e = None if args.no_e2e else end_to_end(problems, packed, ws, plans, dev, args, step_bytes, call)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(args.workload, problems),
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(args.workload),
                     "peak_source": peaks["source"],
                     "kernel": kernel_names(problems) + " (every launch of the step)",
                     "bytes_per_launch": step_bytes / launches,
                     "avg_launch_us": ms_per_step * 1e3 / launches},
        "clocks": clocks,
        "e2e": e2e,
        "runs": runs,
    }
    if not args.no_per_config and not args.shape and world == 1:
        # release this workload's weights first: the other workloads need room
        del graphs, packed, dense_pw, xs, ys, ws
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["per_config"] = per_config_tables(args.workload, dev, peaks)
    if args.workload == "prefill":
        # the timed region replays the step for seconds under the power cap:
        # the sustained (seconds-long) dense rate is the denominator
        tf = step_flops / (ms_per_step * 1e-3) / 1e12
        pk = peaks["bf16_tflops_sustained"]
        line["roofline"] = {"bound": "tensor", "achieved": tf, "peak": pk,
                            "unit": "TFLOP/s", "frac": tf / pk, "traffic": None,
                            "peak_source": peaks["source"] + " bf16 sustained (fp16 dense rate is the same); "
                                           f"burst {peaks['bf16_tflops']:.0f} TFLOP/s -> "
                                           f"{tf / peaks['bf16_tflops']:.3f}",
                            "kernel": kernel_names(problems)}
    if rank == 0 and not args.no_cpu_baseline:
        threads = host_cores()
        v, s, desc = oracle_baseline(problems, args.cpu_budget, threads)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": s}
    if rank == 0:
        print(json.dumps(line), flush=True)


def make_weight_copies(problems, dev, with_dense=False):
    """Repacked weights of every layer of a workload, as rotating copies (the
    counts of `rotation`); with_dense: also the dense layout of 2:4 weights,
    for the per-problem comparison.  Returns (packed, dense, bytes of copies)."""
    import dataclasses

    import torch

    import w4a16_mixed_precision_gb300 as w4
    sparse = any(p.sparse for p in problems)
    layers, uses, P, ncopies = rotation(problems)
    packed, dense_pw = {}, {}
    for (K, N, g, a) in layers:
        gen = make_sparse_weights if sparse else make_weights
        Qp, S, Zp = gen(K, N, g, a, seed=seed_for(f"w:{K}:{N}:{g}:{int(a)}"))
        tq, ts = torch.from_numpy(Qp).to(dev), torch.from_numpy(S).to(dev)
        tz = torch.from_numpy(Zp).to(dev) if a else None
        pw = w4.sparse_repack(tq, ts, tz, g) if sparse else w4.repack(tq, ts, tz, g)
        packed[(K, N, g, a)] = [pw] + [dataclasses.replace(pw, buf=pw.buf.clone())
                                      for _ in range(ncopies[(K, N, g, a)] - 1)]
        if with_dense:
            d = w4.repack(tq, ts, tz, g)
            dense_pw[(K, N, g, a)] = [d] + [dataclasses.replace(d, buf=d.buf.clone())
                                           for _ in range(max(1, -(-2 * L2_BYTES // (K * N // 2))))]
        del tq, ts, tz
    total = sum(weight_bytes(*lk, sparse) * len(packed[lk]) for lk in layers)
    return packed, dense_pw, total


def per_config_tables(main_workload: str, dev, peaks) -> dict:
    """The other benchmark workloads, per problem (µs, GB/s, TFLOP/s, roofline
    fraction, cuBLAS fp16 speedup) and summed: measured the same way as the
    per-run table of the main workload, outside its timed region."""
    import torch

    import w4a16_mixed_precision_gb300 as w4
    out = {}
    for name in ("single", "70b-decode", "prefill", "asym-odd"):
        if name == main_workload:
            continue
        problems = ALL_CONFIGS[name]
        packed, _, _ = make_weight_copies(problems, dev)
        max_m = max(p.M for p in problems)
        ws = {lk: w4.Workspace(max_m, lk[0], lk[1], lk[2]) for lk in packed}
        xs = [torch.from_numpy(make_activations(p.M, p.K, seed_for(p.key))).to(dev) for p in problems]
        ys = [torch.empty((p.M, p.N), dtype=torch.float16, device=dev) for p in problems]
        rows = per_run_table(problems, packed, ws, xs, ys, dev, peaks, w4.gemm_into)
        for lk in ws:
            assert w4.device_status(ws[lk]) == 0, "a kernel reported an expired wait"
        tot_us = sum(r["us"] for r in rows)
        tot_b = sum(p.algorithmic_bytes() for p in problems)
        tot_f = sum(p.flops() for p in problems)
        gbs = tot_b / (tot_us * 1e-6) / 1e9
        tfl = tot_f / (tot_us * 1e-6) / 1e12
        geo = float(np.exp(np.mean(np.log([r["speedup_vs_fp16"] for r in rows]))))
        entry = {"workload": WORKLOAD_NAMES[name], "problems": len(problems),
                 "sum_us": round(tot_us, 2), "GBps": round(gbs, 1), "TFLOPs": round(tfl, 2),
                 "cublas_fp16_speedup_geomean": round(geo, 3), "runs": rows}
        if name == "prefill":
            entry["bound"] = "tensor"
            entry["frac"] = round(tfl / peaks["bf16_tflops_sustained"], 4)
            entry["peak"] = peaks["bf16_tflops_sustained"]
            entry["peak_note"] = (f"{peaks['source']} bf16 sustained (the fp16 dense rate is the same); "
                                  f"{tfl / peaks['bf16_tflops']:.3f} of the burst peak")
        else:
            entry["bound"] = "hbm"
            entry["frac"] = round(gbs / peaks["hbm_gbs"], 4)
            entry["peak"] = peaks["hbm_gbs"]
        out[name] = entry
        del packed, ws, xs, ys
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def per_run_table(problems, packed, ws, xs, ys, dev, peaks, call, dense_packed=None):
    """Per problem: our call vs cuBLAS fp16 (and, for 2:4 weights, vs the dense
    kernel on the same weights in the dense layout), each timed as a CUDA graph
    of repeated launches over rotating weight copies."""
    import torch

    import w4a16_mixed_precision_gb300 as w4
    out = []
    fp16_w = {}
    for p in problems:
        lk = (p.K, p.N, p.group, p.asym)
        if lk not in fp16_w:
            g = torch.Generator(device=dev)
            g.manual_seed(p.K * 31 + p.N)
            # enough fp16 copies that a rotation streams more than two L2s
            n = max(2, min(len(packed[lk]), -(-2 * L2_BYTES // (p.K * p.N * 2)) + 1))
            fp16_w[lk] = [torch.randn((p.K, p.N), dtype=torch.float16, device=dev, generator=g)
                          for _ in range(n)]
    stream = torch.cuda.Stream()
    for i, p in enumerate(problems):
        lk = (p.K, p.N, p.group, p.asym)
        R = len(packed[lk])
        Rf = len(fp16_w[lk])
        reps = 60 if p.M * p.N * 2 < (64 << 20) else 6   # bounds the graphs' output memory
        # both sides captured as CUDA graphs of `reps` launches over rotating
        # copies, so host launch cost does not enter the per-call time
        with torch.cuda.stream(stream):
            for _ in range(3):
                call(xs[i], packed[lk][0], ws[lk], ys[i])
                torch.matmul(xs[i], fp16_w[lk][0])
            stream.synchronize()
            g_ours, g_ref = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_ours, stream=stream):
                for r in range(reps):
                    call(xs[i], packed[lk][r % R], ws[lk], ys[i])
            with torch.cuda.graph(g_ref, stream=stream):
                for r in range(reps):
                    torch.matmul(xs[i], fp16_w[lk][r % Rf])
            graphs = [g_ours, g_ref]
            if dense_packed is not None:
                dc = dense_packed[lk]
                g_dense = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_dense, stream=stream):
                    for r in range(reps):
                        w4.gemm_into(xs[i], dc[r % len(dc)], ws[lk], ys[i])
                graphs.append(g_dense)
            times = []
            for g in graphs:
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                stream.synchronize()
                times.append(e0.elapsed_time(e1) * 1e3 / reps)
        us, cu = times[0], times[1]
        gbs = p.algorithmic_bytes() / (us * 1e-6) / 1e9
        tfl = p.flops() / (us * 1e-6) / 1e12
        row = {"M": p.M, "K": p.K, "N": p.N, "group": p.group, "zeros": p.asym, "us": round(us, 3),
               "GBps": round(gbs, 1), "TFLOPs": round(tfl, 2),
               "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
               "tensor_frac": round(tfl / peaks["bf16_tflops"], 4),
               "cublas_fp16_us": round(cu, 3), "speedup_vs_fp16": round(cu / us, 3)}
        if dense_packed is not None:
            row["dense_kernel_us"] = round(times[2], 3)
            row["speedup_vs_dense"] = round(times[2] / us, 3)
        out.append(row)
    return out


def end_to_end(problems, packed, ws, plans, dev, args, step_bytes, call):
    """The step through the public API with host buffers: every step copies all
    of its activations in from pinned host memory, makes the 24 marlin_gemm
    calls (gemm_into), copies every Y back to pinned host memory and
    synchronises.

    Reported value: the step captured once as a CUDA graph and replayed per
    step, as a decode loop replays its step.  The first call's X is copied on
    the compute stream; the other activations are copied in one transfer on a
    side stream, which the second call waits for; each Y is copied back on the
    side stream as soon as its call has finished, so the transfers overlap the
    calls.  `eager`: the step issued call by call from Python on one stream
    (one H2D copy, the calls, one D2H copy)."""
    import torch

    xs_n = [p.M * p.K for p in problems]
    ys_n = [p.M * p.N for p in problems]

    def offsets(ns):  # 16-byte aligned element offsets
        out, o = [], 0
        for n in ns:
            out.append(o)
            o += (n + 7) // 8 * 8
        return out, o

    xo, xt = offsets(xs_n)
    yo, yt = offsets(ys_n)
    hx = torch.empty(xt, dtype=torch.float16).pin_memory()
    hy = torch.empty(yt, dtype=torch.float16).pin_memory()
    for p, o, n in zip(problems, xo, xs_n):
        hx[o:o + n].copy_(torch.from_numpy(make_activations(p.M, p.K, seed_for(p.key)).reshape(-1)))
    dxb = torch.empty(xt, dtype=torch.float16, device=dev)
    dyb = torch.empty(yt, dtype=torch.float16, device=dev)
    dx = [dxb[o:o + n].view(p.M, p.K) for p, o, n in zip(problems, xo, xs_n)]
    dy = [dyb[o:o + n].view(p.M, p.N) for p, o, n in zip(problems, yo, ys_n)]
    steps = max(3, min(args.steps, 200))

    def issue(plan):
        dxb.copy_(hx, non_blocking=True)
        for i, c in plan:
            p = problems[i]
            lk = (p.K, p.N, p.group, p.asym)
            call(dx[i], packed[lk][c], ws[lk], dy[i])
        hy.copy_(dyb, non_blocking=True)

    stream = torch.cuda.Stream()
    side = torch.cuda.Stream()
    fork, x_rest = torch.cuda.Event(), torch.cuda.Event()
    done = [torch.cuda.Event() for _ in problems]

    def issue_overlapped(plan):
        first = plan[0][0]
        fork.record(stream)
        side.wait_event(fork)
        dx[first].view(-1).copy_(hx[xo[first]:xo[first] + xs_n[first]], non_blocking=True)
        rest = [i for i, _ in plan[1:]]
        if rest:
            lo = min(xo[i] for i in rest)
            hi = max(xo[i] + xs_n[i] for i in rest)
            with torch.cuda.stream(side):
                dxb[lo:hi].copy_(hx[lo:hi], non_blocking=True)
                x_rest.record(side)
        for j, (i, c) in enumerate(plan):
            p = problems[i]
            lk = (p.K, p.N, p.group, p.asym)
            if j == 1:
                stream.wait_event(x_rest)
            call(dx[i], packed[lk][c], ws[lk], dy[i])
            done[j].record(stream)
            side.wait_event(done[j])
            with torch.cuda.stream(side):
                hy[yo[i]:yo[i] + ys_n[i]].copy_(dy[i].view(-1), non_blocking=True)
        stream.wait_stream(side)

    with torch.cuda.stream(stream):
        # eager: call by call
        for k in range(3):
            issue(plans[k % len(plans)])
            stream.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            issue(plans[k % len(plans)])
            stream.synchronize()
        dt_eager = (time.perf_counter() - t0) / steps
        # graph: one capture per rotation phase, replayed per step
        graphs = []
        for plan in plans:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                issue_overlapped(plan)
            graphs.append(g)
        for k in range(3):
            graphs[k % len(graphs)].replay()
            stream.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            graphs[k % len(graphs)].replay()
            stream.synchronize()
        dt = (time.perf_counter() - t0) / steps
        # the host copies of the last step's outputs must be the device's outputs
        dyh, dxh = dyb.cpu(), dxb.cpu()
        checked = all(torch.equal(hy[o:o + n], dyh[o:o + n]) for o, n in zip(yo, ys_n)) and \
            all(torch.equal(hx[o:o + n], dxh[o:o + n]) for o, n in zip(xo, xs_n))
    return {"value": step_bytes / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": xt * 2, "copies_checked": checked,
            "d2h_bytes_per_step": yt * 2, "ms_per_step": dt * 1e3, "steps": steps,
            "path": f"per step: one CUDA-graph replay holding the H2D copies of all activations from pinned "
                    f"host memory (the first call's X on the compute stream, the rest in one copy on a side "
                    f"stream), the {len(problems)} library calls ({call.__name__}) and a D2H copy of each "
                    "output on the side stream as soon as its call has finished, then a stream "
                    "synchronisation; host wall clock around each whole step",
            "eager": {"value": step_bytes / dt_eager / 1e9, "ms_per_step": dt_eager * 1e3,
                      "path": "the same step issued call by call through the Python binding"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="7b-decode", choices=sorted(ALL_CONFIGS) + sorted(SPARSE_CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-table", action="store_true", help="skip the per-run table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak (profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-problem tables of the other benchmark workloads")
    ap.add_argument("--shape", default=None,
                    help="one problem M,K,N[,group[,asym]] instead of a workload (profiling a single kernel)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    problems = {**ALL_CONFIGS, **SPARSE_CONFIGS}[args.workload]
    if args.shape:
        v = [int(t) for t in args.shape.split(",")]
        M, K, N = v[0], v[1], v[2]
        sparse = args.workload in SPARSE_CONFIGS
        problems = [Problem("shape", M, K, N, v[3] if len(v) > 3 else 128, bool(v[4]) if len(v) > 4 else False,
                            sparse)]
        args.workload = f"shape {M}x{K}x{N}" + (" 2:4-sparse" if sparse else "")
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, problems, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_setup(args.gpus)
    run_gpu(args, problems, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
