"""Per-bucket route autotune: candidate rule and cache (CPU), measured choice and parity (GPU)."""
import json
import random

import numpy as np
import pytest
import torch

from matrix_orthogonalising_optimizer_gb300 import Muon
from matrix_orthogonalising_optimizer_gb300.autotune import autotune_routes, cache_key, candidates
from oracle import plan as oplan
from tests.helpers import TOL, oracle_O, rel_fro, run_step

import oracle


def test_candidates_follow_the_planner_rule():
    # the AUTO route (the oracle planner's restatement) is always a candidate,
    # Gram only where AUTO picks it, and direct except where AUTO picks Gram
    # for a bf16 bucket of m < 128 (direct bf16 iteration too inaccurate there)
    rng = random.Random(0)
    for _ in range(300):
        r, c = rng.randint(1, 5000), rng.randint(1, 5000)
        m, n = min(r, c), max(r, c)
        for prec, pcode in (("bf16", oplan.PREC_BF16), ("fp32", oplan.PREC_FP32)):
            for small in (0, -1, 100):
                b, _ = oplan.plan_buckets([(r, c, 0)], precision=pcode, small_m=small)
                auto = "gram" if b[0]["route"] == oplan.BUCKET_GRAM else "direct"
                cand = candidates(m, n, prec, small)
                assert auto in cand
                assert ("gram" in cand) == (auto == "gram")
                assert ("direct" in cand) == (auto == "direct" or prec == "fp32" or m >= 128)


def test_cache_and_choice_with_a_fake_timer(tmp_path):
    calls = []

    def timer(m, n, dtype, precision, route, T, sample, steps, seed):
        calls.append((m, n, dtype, route, sample))
        return {"gram": 2.0, "direct": 1.0}[route] if n == 3000 else {"gram": 1.0, "direct": 3.0}[route]

    shapes = [(1000, 3000, "bf16")] * 3 + [(4000, 1000)] * 20 + [(500, 600)] * 2
    path = str(tmp_path / "routes.json")
    routes, table = autotune_routes(shapes, cache_path=path, sample=8, timer=timer)
    assert routes == ["direct"] * 3 + ["gram"] * 20 + ["direct"] * 2
    # two candidates timed per Gram-eligible shape, samples capped by the bucket's count
    assert sorted(calls) == sorted([(1000, 3000, "bf16", "gram", 3), (1000, 3000, "bf16", "direct", 3),
                                    (1000, 4000, "bf16", "gram", 8), (1000, 4000, "bf16", "direct", 8)])
    assert table[cache_key(500, 600, "bf16", "bf16", 5)] == {"candidates": ["direct"], "ms_per_matrix": {},
                                                             "route": "direct"}
    # a second call reads the cache file and times nothing
    calls.clear()
    again, _ = autotune_routes(shapes, cache_path=path, timer=timer)
    assert again == routes and not calls
    assert json.load(open(path)) == table
    # the routes go straight into the plan: one bucket per (shape, route)
    plan = Muon([s[:2] + ("bf16", r) for s, r in zip(shapes, routes)])
    got = {(b["m"], b["n"]): b["route"] for b in plan.buckets()}
    assert got == {(1000, 3000): oplan.BUCKET_DIRECT, (1000, 4000): oplan.BUCKET_GRAM,
                   (500, 600): oplan.BUCKET_DIRECT}


@pytest.mark.gpu
def test_measured_routes_give_the_oracle_result():
    shapes = [(320, 1400)] * 3 + [(1400, 320)] * 2 + [(64, 512)] * 4 + [(300, 300)] * 2
    routes, table = autotune_routes([s + ("bf16",) for s in shapes], sample=4, steps=2)
    for (r, c), route in zip(shapes, routes):
        m, n = min(r, c), max(r, c)
        entry = table[cache_key(m, n, "bf16", "bf16", 5)]
        assert route in candidates(m, n)
        if len(entry["candidates"]) == 2:
            t = entry["ms_per_matrix"]
            assert set(t) == {"gram", "direct"} and all(v > 0 for v in t.values())
            assert route == min(t, key=t.get)
    from tests.test_gpu_parity import BETA, make_inputs
    inputs = make_inputs(shapes, "bf16", 31)
    muon = Muon([(r, c, 0, rt) for (r, c), rt in zip(shapes, routes)]).bind()
    w, _, _ = run_step(shapes, inputs, "bf16", lr=1.0, beta=BETA, wd=0.0, zero_w=True, muon=muon)
    want = oracle_O(inputs, beta=BETA)
    for (r, c), wi, o in zip(shapes, w, want):
        got = -wi.double().numpy() / oracle.shape_scale(r, c)
        assert rel_fro(got, o) <= TOL["bf16"]
