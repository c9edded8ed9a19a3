"""Per-bucket route and tile autotune with a cache (plan time, on the GPU that will run the steps).

The DMuon pages choose work from measured costs rather than FLOP counts
(technical summary, section 2.3) and tune their kernels' tiles per shape
(section 2.4).  Here the choices tuned are each bucket's Newton-Schulz form
and, for bf16 buckets with m <= 128, its tile rule: several matrices packed
block-diagonally into one 256 x 256 pair tile, or one matrix per tile.  The AUTO
rule picks Gram space where the bf16 Gram recurrence is accurate enough (n >=
3m, or small m with split-bf16 m x m products); the direct form is accurate
for every shape with m >= 128, so where AUTO picks Gram both forms are
candidates there, Gram alone below, and elsewhere direct is the only one.
Each (route, tile) candidate is timed as a step over a sample of matrices of
the bucket's shape (seeded synthetic data, CUDA events on the stream), and
the fastest is kept.

Results are cached per (m, n, dtype, precision, ns_steps) in a dict that can
be saved as JSON, so a set is timed once per machine.  The routes come back
per shape, ready to pass as the fourth and fifth elements of each shape to
``Muon`` / ``dmuon_plan``.  The timing runs the library's own step; nothing here is on
the step's path.
"""
from __future__ import annotations

import json
import os

from . import _lib
from ._lib import BF16, FP32

__all__ = ["candidates", "tile_candidates", "cache_key", "autotune_buckets"]

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


def tile_candidates(m: int, precision: str = "bf16") -> list:
    """Tile rules a bucket may take: packing applies to the tensor-core
    products of bf16 buckets with m <= 128; elsewhere the plan's (AUTO) rule,
    which resolves to one matrix per tile."""
    return ["packed", "single"] if precision == "bf16" and m <= 128 else ["auto"]


def cache_key(m: int, n: int, dtype: str, precision: str, ns_steps: int) -> str:
    return f"{m}x{n}:{dtype}:{precision}:T{ns_steps}"


def _dtype_name(dt) -> str:
    return dt if isinstance(dt, str) else _DT_NAMES[int(dt)]


def _time_choice(m, n, dtype, precision, route, tile, ns_steps, sample, steps, seed):
    import torch

    from . import Muon
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = [(torch.randn(m, n, device="cuda", generator=g) * 0.02).to(tdt) for _ in range(sample)]
    gr = [(torch.randn(m, n, device="cuda", generator=g) * 1e-3).to(tdt) for _ in range(sample)]
    mo = [torch.zeros(m, n, device="cuda", dtype=tdt) for _ in range(sample)]
    opt = Muon([(m, n, dtype, route, tile)] * sample, precision=precision).bind()
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


def autotune_buckets(shapes, precision: str = "bf16", ns_steps: int = 5, small_m: int = 0, cache=None,
                     cache_path: str | None = None, sample: int = 8, steps: int = 3, timer=None):
    """(route, tile) per shape and the cache table.

    shapes: (rows, cols[, dtype]) as for ``Muon``.  cache: a dict from an
    earlier call (updated in place); cache_path: a JSON file read first and
    written back.  Each untimed (m, n, dtype) with several candidates is
    timed with ``sample`` matrices (at most the bucket's own count) over
    ``steps`` steps; ``timer`` replaces the GPU timing (tests).  One
    candidate: no timing, the entry records it alone.
    """
    if cache is None:
        cache = {}
    if cache_path and os.path.exists(cache_path):
        with open(cache_path) as f:
            cache.update(json.load(f))
    timer = timer or _time_choice
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
        cand = [f"{r}/{t}" for r in candidates(m, n, precision, small_m) for t in tile_candidates(m, precision)]
        entry = {"candidates": cand, "ms_per_matrix": {}}
        if len(cand) > 1:
            k = max(1, min(sample, count))
            for i, c in enumerate(cand):
                route, tile = c.split("/")
                entry["ms_per_matrix"][c] = timer(m, n, dtype, precision, route, tile, ns_steps, k, steps, 1000 + i)
            best = min(cand, key=lambda c: entry["ms_per_matrix"][c])
        else:
            best = cand[0]
        entry["route"], entry["tile"] = best.split("/")
        cache[key] = entry
    if cache_path:
        with open(cache_path, "w") as f:
            json.dump(cache, f, indent=1, sort_keys=True)
    out = []
    for m, n, dt in keys:
        e = cache[cache_key(m, n, dt, precision, ns_steps)]
        out.append((e["route"], e["tile"]))
    return out, cache
