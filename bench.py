#!/usr/bin/env python3
"""Benchmark of one batched Muon optimizer step on a GB300.

Workload (default): the Llama-3-8B-shaped set, 32 layers x {q 4096x4096,
k 1024x4096, v 1024x4096, o 4096x4096, gate 14336x4096, up 14336x4096,
down 4096x14336} = 224 bf16 matrices, gradients N(0,1)*1e-3 with 1 % of the
entries x100, zero momentum, 5 Newton-Schulz steps, lr 0.02, beta 0.95,
wd 0.01.  The step is the whole hot path: momentum + pack + norms, the Gram
products, the Newton-Schulz polynomial products and the final product fused
with the update.  Inputs (42 GB) are resident in HBM and larger than L2.

Prints one JSON line (rank 0).  At N = 1 the line also carries ``configs``:
the other sets (single 256x1024 fp32 matrix, small transformer, 2 000 mixed
small matrices, large-layer stress) timed the same way after the headline set,
each beside the oracle on the host cores.  ``--impl reference`` times the fp64
CPU oracle instead: each step one seeded matrix of one shape bucket, the set's
rate extrapolated by bucket counts.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dmuon", "reference"], default="dmuon")
    ap.add_argument("--config", default="c3", help="workload: c1..c5 (c3 is the measured one)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adamw", action="store_true", help="skip the AdamW comparison step")
    ap.add_argument("--routes", choices=["auto", "tuned"], default="auto",
                    help="tuned: time each bucket's routes (Gram, direct) and tile rules (packed, single) "
                         "first (autotune cache), plan with the fastest")
    ap.add_argument("--owners", type=int, default=8,
                    help="owner-model leg: ranks D the set is split over (0 = skip)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--extra-configs", default="c1,c2,c4,c5",
                    help="after the headline set, time these sets too (N=1 only; '' = none)")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--budget-gb", type=float, default=0.0,
                    help="workspace budget per wave in GiB (0 = the configuration's own)")
    return ap.parse_args()


def measured_traffic():
    """DRAM bytes per gemm_tc launch from the committed ncu summary, while the kernel is unchanged."""
    import hashlib
    csrc = os.path.join(ROOT, "matrix_orthogonalising_optimizer_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "epilogue.cuh", "internal.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    try:
        text = open(os.path.join(ROOT, "profiles", "launches_llama8b_set.md")).read()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines()
                  if line.startswith(("traffic_bytes_per_launch:", "kernel_sources_sha256_16:")))
    if fields.get("kernel_sources_sha256_16", "").strip() != h.hexdigest()[:16]:
        return None
    return float(fields["traffic_bytes_per_launch"])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id):
        self.device_id = device_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.device_id is not None:
            cmd += ["-i", str(self.device_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, val in zip(names, p[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle


def oracle_flops(m, n, T=5):
    """Multiply-add flops of the oracle's direct Newton-Schulz (full products)."""
    return T * (4.0 * m * m * n + 2.0 * m ** 3)


def oracle_sample(cfg, index):
    """Time the fp64 oracle on matrix ``index`` of ``cfg`` (CPU inputs, same recipe)."""
    import numpy as np

    import oracle
    import workloads
    w, g, m = workloads.make_matrix(cfg, index, "cpu")
    args = (w.double().numpy(), g.double().numpy(), m.double().numpy())
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    t0 = time.perf_counter()
    oracle.muon_step(*args, lr=f32(cfg.lr), beta=f32(cfg.beta), wd=f32(cfg.wd), ns_steps=cfg.ns_steps,
                     dtype=cfg.dtype)
    return time.perf_counter() - t0


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [x.get("num_threads") for x in threadpool_info() if x.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count()


def _buckets(cfg):
    """Oracle cost classes of a set: (m, n) -> member indices (tall matrices
    transposed, as the oracle and the planner both do), smallest first."""
    b = {}
    for i, (r, c) in enumerate(cfg.shapes):
        b.setdefault((min(r, c), max(r, c)), []).append(i)
    return dict(sorted(b.items(), key=lambda kv: (kv[0][0] * kv[0][1], kv[0])))


def cpu_baseline(cfg, full_limit_tflop=2.0):
    """Oracle matrices/s for the whole set on the host's cores.

    Sets whose oracle work is under ``full_limit_tflop`` (c1, c2) are timed in
    full.  Larger sets time one seeded matrix of every (m, n) bucket (its first
    member) and extrapolate the set's time by each bucket's count; the result
    is labelled "extrapolated" and the per-bucket oracle GFLOP/s are listed."""
    buckets = _buckets(cfg)
    T = cfg.ns_steps
    total_flop = sum(oracle_flops(m, n, T) * len(ix) for (m, n), ix in buckets.items())
    full = total_flop / 1e12 <= full_limit_tflop
    per_bucket, t_set, t_timed = [], 0.0, 0.0
    for (m, n), ix in buckets.items():
        timed = ix if full else ix[:1]
        t = sum(oracle_sample(cfg, i) for i in timed)
        t_timed += t
        t_one = t / len(timed)
        t_set += t_one * len(ix)
        per_bucket.append({"m": m, "n": n, "count": len(ix), "timed": len(timed), "s_per_matrix": t_one,
                           "oracle_gflops": oracle_flops(m, n, T) / t_one / 1e9})
    what = ("the whole set, every matrix timed" if full else
            "one seeded matrix per bucket (" + ", ".join(f"{b['m']}x{b['n']}" for b in per_bucket) +
            "), set time extrapolated by each bucket's count")
    return {"value": len(cfg.shapes) / t_set, "unit": "matrices/s", "cores": cpu_threads(), "kind": "oracle",
            "extrapolated": not full, "per_bucket": per_bucket,
            "sample": f"{what}; fp64 direct Newton-Schulz, {t_timed:.1f} s of oracle time, "
                      f"{t_set:.1f} s per step of the whole set"}


def cpu_baseline_estimate(cfg, rate_gflops, source):
    """Oracle matrices/s of a set too large to sample in a bench run (one of
    its matrices takes minutes): its flop count at a measured oracle rate."""
    T = cfg.ns_steps
    total_flop = sum(oracle_flops(min(r, c), max(r, c), T) for r, c in cfg.shapes)
    t_set = total_flop / (rate_gflops * 1e9)
    return {"value": len(cfg.shapes) / t_set, "unit": "matrices/s", "cores": cpu_threads(), "kind": "oracle",
            "extrapolated": True, "estimated": True,
            "sample": f"not timed (one matrix of this set takes minutes): the set's oracle flop count at "
                      f"{rate_gflops:.0f} GFLOP/s, the oracle rate measured on {source}"}


# ---------------------------------------------------------------- distributed


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The slowest rank's time: every rank gets the maximum of x (timing only, not data)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(n_matrices, world, ms_per_step):
    """Whole-job matrices/s: every rank steps its own replica of the set (weak scaling)."""
    return world * n_matrices / (ms_per_step / 1000.0)


# ---------------------------------------------------------------- arms


def run_reference(args, cfg, world, rank):
    """The fp64 CPU oracle as the reference arm (rank 0 only).

    Each step times the oracle on one seeded matrix of one (m, n) bucket of the
    set, the buckets taken in turn (warm-up steps use the smallest), so every
    step is a bounded sample and ``ms_per_step`` is its real wall time.  The
    set's matrices/s is extrapolated from the per-bucket times by each
    bucket's count (buckets no timed step reached: by the oracle's flop rate
    on the others)."""
    if rank != 0:
        return
    buckets = list(_buckets(cfg).items())
    T = cfg.ns_steps
    for _ in range(args.warmup):
        oracle_sample(cfg, buckets[0][1][0])
    times = {}
    walls = []
    for k in range(args.steps):
        (m, n), ix = buckets[k % len(buckets)]
        t0 = time.perf_counter()
        dt = oracle_sample(cfg, ix[0])
        walls.append(time.perf_counter() - t0)
        times.setdefault((m, n), []).append(dt)
    rate = (sum(oracle_flops(m, n, T) * len(v) for (m, n), v in times.items()) /
            sum(sum(v) for v in times.values()))
    t_set = 0.0
    for (m, n), ix in buckets:
        t_one = statistics.median(times[(m, n)]) if (m, n) in times else oracle_flops(m, n, T) / rate
        t_set += t_one * len(ix)
    v = len(cfg.shapes) / t_set
    ms_step = 1000.0 * statistics.mean(walls)
    sample = (f"each step one seeded matrix of one (m, n) bucket, the {len(buckets)} buckets in turn "
              f"({', '.join(f'{m}x{n}' for (m, n), _ in buckets)}); set time extrapolated by each bucket's "
              f"count: {t_set:.1f} s per step of the whole set")
    print(json.dumps({
        "impl": "reference", "metric": "Muon optimizer-step matrices/s", "value": v, "unit": "matrices/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, "auto", 1),
        "cpu_baseline": {"value": v, "unit": "matrices/s", "cores": cpu_threads(), "kind": "oracle",
                         "extrapolated": True, "sample": sample},
        "set_seconds_extrapolated": t_set,
        "e2e": {"value": v, "unit": "matrices/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def config_dict(cfg, routes, world):
    import workloads
    return {"workload": workloads_name(cfg), "matrices": len(cfg.shapes), "ns_steps": cfg.ns_steps,
            "elements": workloads.total_elements(cfg), "lr": cfg.lr, "beta": cfg.beta, "wd": cfg.wd,
            "l2": "inputs larger than L2 (resident in HBM)",
            "parallelism": "replicas" if world > 1 else "single GPU", "routes": routes}


def workloads_name(cfg):
    return f"{cfg.name}: {cfg.title}"


def run_dmuon(args, cfg, world, rank, local):
    import torch

    import workloads
    from matrix_orthogonalising_optimizer_gb300 import Muon, _lib

    _lib.load(build_if_missing=True)
    dt = 0 if cfg.dtype == "bf16" else 1
    budget = int((args.budget_gb or cfg.budget_gb) * (1 << 30))
    shapes = [(r, c, dt) for r, c in cfg.shapes]
    if args.routes == "tuned":
        from matrix_orthogonalising_optimizer_gb300.autotune import autotune_buckets
        choices, _ = autotune_buckets([(r, c, cfg.dtype) for r, c in cfg.shapes], precision=cfg.precision,
                                      ns_steps=cfg.ns_steps)
        shapes = [s + ch for s, ch in zip(shapes, choices)]
    muon = Muon(shapes, precision=cfg.precision, workspace_budget=budget).bind()
    ws, gs, ms = workloads.make_set(cfg, "cuda")
    torch.cuda.synchronize()
    lr, beta, wd, T = cfg.lr, cfg.beta, cfg.wd, cfg.ns_steps
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 0)):
        muon.step(ws, gs, ms, lr, beta, wd, T, stream)
    torch.cuda.synchronize()
    if muon.device_status(stream) != 0:
        raise RuntimeError("device status set during warm-up")

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    sampler.start()
    time.sleep(0.3)
    muon.set_timing(True)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        muon.step(ws, gs, ms, lr, beta, wd, T, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_step = e0.elapsed_time(e1) / args.steps
    timing = muon.timing()
    muon.set_timing(False)
    if muon.device_status(stream) != 0:
        raise RuntimeError("device status set during the timed steps")
    ms_step = max_over_ranks(ms_step, world)

    n_mat = len(cfg.shapes)
    value = replica_value(n_mat, world, ms_step)
    flops_total, flops_tc = muon.flops(T)
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tc_ms = timing["tc"][0] / args.steps
    achieved = flops_tc / (tc_ms / 1000.0) / 1e12 if tc_ms > 0 else 0.0
    launches = sum(timing[k][1] for k in ("momentum", "norm", "tc", "simt"))
    stages = {k: round(v[0] / args.steps, 4) for k, v in timing.items()}
    launches_per_step = {k: v[1] // args.steps for k, v in timing.items()}

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(muon, cfg, ws, gs, ms, args.e2e_steps, stream, world)

    owners = None
    if args.owners > 0 and world == 1:
        owners = measure_owner_model(cfg, ws, gs, ms, stream, args.owners, ms_step)

    adamw = None
    if not args.no_adamw:
        adamw = measure_adamw(cfg, ws, gs, stream, args.steps, args.warmup, world, peaks, src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg)

    configs = None
    if world == 1 and args.extra_configs:
        import gc
        del ws, gs, ms, muon
        gc.collect()
        torch.cuda.empty_cache()
        configs = {}
        rate = None
        if cpu and cpu.get("per_bucket"):
            big = max(cpu["per_bucket"], key=lambda b: b["m"] * b["n"])
            rate = (big["oracle_gflops"], f"the {big['m']}x{big['n']} bucket of {args.config}")
        for name in [c for c in args.extra_configs.split(",") if c and c != args.config]:
            est = rate if name == "c5" else None
            configs[name] = measure_config(name, args.extra_steps if name != "c5" else 3, 3 if name != "c5" else 2,
                                           peaks, src, cpu=not args.no_cpu_baseline and (name != "c5" or rate),
                                           oracle_rate=est)

    if rank == 0:
        line = {
            "metric": "Muon optimizer-step matrices/s", "value": value, "unit": "matrices/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg.precision == "bf16" else "fp32",
            "data": "synthetic",
            "config": config_dict(cfg, args.routes, world),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "traffic": measured_traffic() if args.config == "c3" else None,
                         "kernel": "gemm_tc_kernel (all tcgen05 GEMM launches of a step)",
                         "peak_source": f"bf16_tflops_sustained of {src} peaks"},
            "gemm_algorithmic_tflop_per_step": flops_tc / 1e12,
            "step_tflops": flops_total / (ms_step / 1000.0) / 1e12,
            "step_frac_of_peak": flops_total / (ms_step / 1000.0) / 1e12 / peak,
            "stages_ms_per_step": stages, "launches_per_step": launches_per_step,
            "gpu_launches": int(launches), "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "adamw": adamw, "owner_model": owners, "configs": configs,
            "muon_over_adamw_step_time": ms_step / adamw["ms_per_step"] if adamw and "ms_per_step" in adamw
            else None,
        }
        print(json.dumps(line), flush=True)


L2_BYTES = 129 * 10 ** 6


def measure_config(name, steps, warmup, peaks, src, cpu, oracle_rate=None):
    """One more workload, timed like the headline one: ms/step, matrices/s, the
    tcgen05 GEMM fraction of peak and the stage split, and beside it the oracle
    on the host (``cpu``).  Sets whose inputs fit in L2 have L2 flushed
    (a 512 MB write) before every timed step, each step timed alone."""
    import gc

    import torch

    import workloads
    from matrix_orthogonalising_optimizer_gb300 import Muon
    cfg = workloads.get(name)
    dt = 0 if cfg.dtype == "bf16" else 1
    esz = 2 if cfg.dtype == "bf16" else 4
    budget = int(cfg.budget_gb * (1 << 30))
    muon = Muon([(r, c, dt) for r, c in cfg.shapes], precision=cfg.precision, workspace_budget=budget)
    inputs = 3 * workloads.total_elements(cfg) * esz
    free, _ = torch.cuda.mem_get_info()
    if inputs + muon.workspace_bytes() + (4 << 30) > free:
        return {"workload": workloads_name(cfg),
                "skipped": f"needs {(inputs + muon.workspace_bytes()) / 1e9:.0f} GB, {free / 1e9:.0f} GB free"}
    muon.bind()
    ws, gs, ms = workloads.make_set(cfg, "cuda")
    lr, beta, wd, T = cfg.lr, cfg.beta, cfg.wd, cfg.ns_steps
    stream = torch.cuda.current_stream()
    flush = inputs < 2 * L2_BYTES
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device="cuda") if flush else None
    for _ in range(warmup):
        muon.step(ws, gs, ms, lr, beta, wd, T, stream)
    torch.cuda.synchronize()

    def timed_steps():
        per_step = []
        if flush:
            for _ in range(steps):
                scrub.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                muon.step(ws, gs, ms, lr, beta, wd, T, stream)
                e1.record(stream)
                per_step.append((e0, e1))
            torch.cuda.synchronize()
            return sum(a.elapsed_time(b) for a, b in per_step) / steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            muon.step(ws, gs, ms, lr, beta, wd, T, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    # the step time without the stage timers (whose events between launches
    # keep each launch from starting while the previous one finishes), then
    # the same steps again with them for the stage split and the GEMM rate
    ms_step = timed_steps()
    muon.set_timing(True)
    ms_with_timers = timed_steps()
    timing = muon.timing()
    muon.set_timing(False)
    status = muon.device_status(stream)
    flops_total, flops_tc = muon.flops(T)
    del ws, gs, ms, muon, scrub
    gc.collect()
    torch.cuda.empty_cache()
    if status != 0:
        raise RuntimeError(f"device status set in the {name} measurement")
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tc_ms = timing["tc"][0] / steps
    out = {"workload": workloads_name(cfg), "matrices": len(cfg.shapes), "steps": steps, "warmup": warmup,
           "ms_per_step": ms_step, "matrices_per_s": len(cfg.shapes) / (ms_step / 1000.0),
           "ms_per_step_with_stage_timers": ms_with_timers,
           "dtype": "bf16" if cfg.precision == "bf16" else "fp32",
           "l2": "L2 flushed (512 MB write) before every timed step" if flush
           else "inputs larger than L2 (resident in HBM)",
           "stages_ms_per_step": {k: round(v[0] / steps, 4) for k, v in timing.items()},
           "launches_per_step": {k: v[1] // steps for k, v in timing.items()},
           "step_tflops": flops_total / (ms_step / 1000.0) / 1e12}
    if flops_tc > 0 and tc_ms > 0:
        achieved = flops_tc / (tc_ms / 1000.0) / 1e12
        out["gemm"] = {"algorithmic_tflop_per_step": flops_tc / 1e12, "achieved_tflops": achieved,
                       "frac_of_sustained_peak": achieved / peak, "peak_source": f"bf16_tflops_sustained of {src} peaks"}
    if cpu:
        out["cpu_baseline"] = (cpu_baseline(cfg) if oracle_rate is None
                               else cpu_baseline_estimate(cfg, *oracle_rate))
    return out


def _time_subset(cfg, idx, ws, gs, ms, stream, warmup=2, steps=3):
    """ms per step of the Muon step restricted to the matrices `idx` (own plan and workspace)."""
    import torch

    from matrix_orthogonalising_optimizer_gb300 import Muon
    dt = 0 if cfg.dtype == "bf16" else 1
    sub = Muon([(cfg.shapes[i][0], cfg.shapes[i][1], dt) for i in idx], precision=cfg.precision).bind()
    w, g, m = [ws[i] for i in idx], [gs[i] for i in idx], [ms[i] for i in idx]
    for _ in range(warmup):
        sub.step(w, g, m, cfg.lr, cfg.beta, cfg.wd, cfg.ns_steps, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        sub.step(w, g, m, cfg.lr, cfg.beta, cfg.wd, cfg.ns_steps, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    status = sub.device_status(stream)
    del sub
    torch.cuda.empty_cache()
    if status != 0:
        raise RuntimeError("device status set in the owner-model leg")
    return e0.elapsed_time(e1) / steps


def measure_owner_model(cfg, ws, gs, ms, stream, ranks, redundant_ms):
    """The pages' owner-centric execution at one GPU (DMuon summary, sections 2.1 and 2.3).

    Without owners every rank runs the whole set's update (the replicated
    step timed above).  With owners each matrix is updated once, by the rank
    that owns it; owners are assigned from measured costs (each bucket's step
    timed alone, divided by its count), and the step of each rank's share is
    timed here one rank after another.  Reports the slowest rank against the
    replicated step."""
    from matrix_orthogonalising_optimizer_gb300 import Muon, assign_owners
    dt = 0 if cfg.dtype == "bf16" else 1
    plan = Muon([(r, c, dt) for r, c in cfg.shapes], precision=cfg.precision)
    cost = [0.0] * len(cfg.shapes)
    per_bucket = []
    for b in plan.buckets():
        t = _time_subset(cfg, b["members"], ws, gs, ms, stream)
        per_bucket.append({"m": b["m"], "n": b["n"], "count": len(b["members"]), "ms": t})
        for i in b["members"]:
            cost[i] = t / len(b["members"])
    owner, predicted = assign_owners(cost, ranks, "greedy")
    flops_owner, flops_pred = assign_owners(plan.matrix_flops(cfg.ns_steps), ranks, "greedy")
    rank_ms = [_time_subset(cfg, [i for i in range(len(owner)) if owner[i] == r], ws, gs, ms, stream)
               if r in owner else 0.0 for r in range(ranks)]
    slowest = max(rank_ms)
    return {"ranks": ranks, "cost_model": "measured: each bucket's step alone / its count",
            "bucket_ms": per_bucket, "predicted_makespan_ms": predicted, "rank_ms": rank_ms,
            "slowest_rank_ms": slowest, "replicated_ms": redundant_ms,
            "speedup_over_replicated": redundant_ms / slowest if slowest > 0 else None,
            "owners_same_as_flop_model": owner == flops_owner}


def measure_adamw(cfg, ws, gs, stream, steps, warmup, world, peaks, src):
    """The element-wise optimizer the pages compare against, on the same tensors: one
    multi-tensor AdamW step (states in the parameters' dtype) timed like the Muon step.
    Context for the Muon step time, not a second headline."""
    import torch

    from matrix_orthogonalising_optimizer_gb300 import adamw_step
    need = 2 * sum(w.numel() * w.element_size() for w in ws)
    free, _ = torch.cuda.mem_get_info()
    if free < need + (4 << 30):
        return {"skipped": f"states need {need / 2**30:.1f} GiB, {free / 2**30:.1f} GiB free"}
    m = [torch.zeros_like(w) for w in ws]
    v = [torch.zeros_like(w) for w in ws]
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=cfg.wd)
    t = 0
    for _ in range(max(warmup, 1)):
        t += 1
        adamw_step(ws, gs, m, v, step=t, stream=stream, **kw)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        t += 1
        adamw_step(ws, gs, m, v, step=t, stream=stream, **kw)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    elems = sum(w.numel() for w in ws)
    per_elem = 7 * ws[0].element_size()  # read W, g, m, v; write W, m, v
    gbs = elems * per_elem / (ms_step / 1000.0) / 1e9
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    del m, v
    torch.cuda.empty_cache()
    return {"ms_per_step": ms_step, "matrices_per_s": replica_value(len(ws), world, ms_step),
            "bytes_per_step": elems * per_elem, "achieved_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm,
            "peak_source": f"hbm_gbs of {src} peaks", "states_dtype": str(ws[0].dtype).replace("torch.", ""),
            "hyper": kw}


def measure_e2e(muon, cfg, ws, gs, ms, steps, stream, world, overlap=None, host_out=None):
    """Same metric through the public API with host buffers: every step copies the
    gradients host->device from pinned memory and reads the updated parameters back.

    The copies run on their own streams and overlap the compute: step i+1's gradients
    go into a second device buffer while step i computes, and step i's parameters are
    read back while step i+1 runs its momentum and Newton-Schulz phases; step i+1 waits
    for that read only before its first parameter write (dmuon_step_ex's params_ready
    event).  The timed region spans the first upload to the last read-back.  Without
    room for a second copy of the gradients on the device the copies run in line."""
    import torch
    host_g = [g.cpu().pin_memory() for g in gs]
    host_w = [torch.empty(w.shape, dtype=w.dtype, pin_memory=True) for w in ws]
    h2d = sum(g.numel() * g.element_size() for g in gs)
    d2h = sum(w.numel() * w.element_size() for w in ws)
    lr, beta, wd, T = cfg.lr, cfg.beta, cfg.wd, cfg.ns_steps
    free, _ = torch.cuda.mem_get_info()
    if overlap is None:
        overlap = free > h2d + (4 << 30)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if not overlap:
        e0.record(stream)
        for _ in range(steps):
            for d, h in zip(gs, host_g):
                d.copy_(h, non_blocking=True)
            muon.step(ws, gs, ms, lr, beta, wd, T, stream)
            for h, d in zip(host_w, ws):
                h.copy_(d, non_blocking=True)
        e1.record(stream)
    else:
        gbuf = [gs, [torch.empty_like(g) for g in gs]]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        uploaded, computed, read = [], [], []

        def upload(i):
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[i - 2])  # its buffer was read by step i-2
                for d, h in zip(gbuf[i % 2], host_g):
                    d.copy_(h, non_blocking=True)
                uploaded.append(ev())
                uploaded[-1].record(s_in)

        e0.record(stream)
        s_in.wait_event(e0)
        upload(0)
        for i in range(steps):
            stream.wait_event(uploaded[i])
            muon.step(ws, gbuf[i % 2], ms, lr, beta, wd, T, stream, params_ready=read[i - 1] if i else None)
            computed.append(ev())
            computed[-1].record(stream)
            if i + 1 < steps:
                upload(i + 1)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                for h, w in zip(host_w, ws):
                    h.copy_(w, non_blocking=True)
                read.append(ev())
                read[-1].record(s_out)
        stream.wait_event(read[-1])
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    if host_out is not None:
        host_out.extend(host_w)
    return {"value": replica_value(len(cfg.shapes), world, ms_step), "unit": "matrices/s",
            "ms_per_step": ms_step, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "overlapped with compute (double-buffered gradients; parameters read back during the next step's earlier phases)"
            if overlap else "in line"}


def main():
    args = parse_args()
    import workloads
    cfg = workloads.get(args.config)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, cfg, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup(args)
    run_dmuon(args, cfg, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
