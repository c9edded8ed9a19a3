"""Per-bucket route autotune with a cache (plan time, on the GPU that will run the steps).

The DMuon pages choose work from measured costs rather than FLOP counts
(technical summary, section 2.3) and tune their kernels per shape (section
2.4).  Here the choice tuned is each bucket's Newton-Schulz form.  The AUTO
rule picks Gram space where the bf16 Gram recurrence is accurate enough (n >=
3m, or small m with split-bf16 m x m products); the direct form is accurate
for every shape with m >= 128, so where AUTO picks Gram both forms are
candidates there, Gram alone below, and elsewhere direct is the only one.  Each candidate is timed as a step over a
sample of matrices of the bucket's shape (seeded synthetic data, CUDA events
on the stream), and the faster is kept.

Results are cached per (m, n, dtype, precision, ns_steps) in a dict that can
be saved as JSON, so a set is timed once per machine.  The routes come back
per shape, ready to pass as the fourth element of each shape to ``Muon`` /
``dmuon_plan``.  The timing runs the library's own step; nothing here is on
the step's path.
"""
from __future__ import annotations

import json
import os

from . import _lib
from ._lib import BF16, FP32

__all__ = ["candidates", "cache_key", "autotune_routes"]

_DT_NAMES = {BF16: "bf16", FP32: "fp32"}


# Below this short side the bf16 direct iteration's error reaches the 3e-2
# bar on O (emulated: 0.025-0.037 for m = 64, at most 0.025 from m = 128 on),
# so a measured choice never sends such a bucket there.
DIRECT_MIN_M = 128


def candidates(m: int, n: int, precision: str = "bf16", small_m: int = 0) -> list:
    """Routes a bucket of canonical shape (m, n) may take: the AUTO rule's choice and,
    where that is Gram and m >= DIRECT_MIN_M, also direct (the header's AUTO rule,
    restated)."""
    if small_m == 0:
        small_m = 256
    if precision == "fp32":
        return ["gram", "direct"]
    auto_gram = n >= 3 * m or (small_m > 0 and m <= small_m)
    if not auto_gram:
        return ["direct"]
    return ["gram", "direct"] if m >= DIRECT_MIN_M else ["gram"]


def cache_key(m: int, n: int, dtype: str, precision: str, ns_steps: int) -> str:
    return f"{m}x{n}:{dtype}:{precision}:T{ns_steps}"


def _dtype_name(dt) -> str:
    return dt if isinstance(dt, str) else _DT_NAMES[int(dt)]


def _time_route(m, n, dtype, precision, route, ns_steps, sample, steps, seed):
    import torch

    from . import Muon
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = [(torch.randn(m, n, device="cuda", generator=g) * 0.02).to(tdt) for _ in range(sample)]
    gr = [(torch.randn(m, n, device="cuda", generator=g) * 1e-3).to(tdt) for _ in range(sample)]
    mo = [torch.zeros(m, n, device="cuda", dtype=tdt) for _ in range(sample)]
    opt = Muon([(m, n, dtype, route)] * sample, precision=precision).bind()
    stream = torch.cuda.current_stream()
    for _ in range(2):
        opt.step(w, gr, mo, 0.02, 0.95, 0.01, ns_steps, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        opt.step(w, gr, mo, 0.02, 0.95, 0.01, ns_steps, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if opt.device_status(stream) != 0:
        raise _lib.DmuonError(_lib.ERR_DEVICE_TIMEOUT, "autotune step")
    ms = e0.elapsed_time(e1) / steps / sample
    del opt, w, gr, mo
    torch.cuda.empty_cache()
    return ms


def autotune_routes(shapes, precision: str = "bf16", ns_steps: int = 5, small_m: int = 0, cache=None,
                    cache_path: str | None = None, sample: int = 8, steps: int = 3, timer=None):
    """Route per shape ("gram" / "direct") and the cache table.

    shapes: (rows, cols[, dtype]) as for ``Muon``.  cache: a dict from an
    earlier call (updated in place); cache_path: a JSON file read first and
    written back.  Each untimed (m, n, dtype) with two candidates is timed
    with ``sample`` matrices (at most the bucket's own count) over ``steps``
    steps; ``timer`` replaces the GPU timing (tests).  One candidate: no
    timing, the entry records the route alone.
    """
    if cache is None:
        cache = {}
    if cache_path and os.path.exists(cache_path):
        with open(cache_path) as f:
            cache.update(json.load(f))
    timer = timer or _time_route
    counts = {}
    keys = []
    for s in shapes:
        rows, cols = int(s[0]), int(s[1])
        dtype = _dtype_name(s[2] if len(s) > 2 else "bf16")
        m, n = min(rows, cols), max(rows, cols)
        keys.append((m, n, dtype))
        counts[(m, n, dtype)] = counts.get((m, n, dtype), 0) + 1
    for (m, n, dtype), count in counts.items():
        key = cache_key(m, n, dtype, precision, ns_steps)
        if key in cache:
            continue
        cand = candidates(m, n, precision, small_m)
        entry = {"candidates": cand, "ms_per_matrix": {}}
        if len(cand) > 1:
            k = max(1, min(sample, count))
            for i, route in enumerate(cand):
                entry["ms_per_matrix"][route] = timer(m, n, dtype, precision, route, ns_steps, k, steps, 1000 + i)
            entry["route"] = min(cand, key=lambda r: entry["ms_per_matrix"][r])
        else:
            entry["route"] = cand[0]
        cache[key] = entry
    if cache_path:
        with open(cache_path, "w") as f:
            json.dump(cache, f, indent=1, sort_keys=True)
    routes = [cache[cache_key(m, n, dt, precision, ns_steps)]["route"] for m, n, dt in keys]
    return routes, cache
