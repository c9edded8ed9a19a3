"""Per-bucket route and tile autotune: candidate rules and cache (CPU), measured choice and parity (GPU)."""
import json
import random

import numpy as np
import pytest
import torch

from matrix_orthogonalising_optimizer_gb300 import Muon
from matrix_orthogonalising_optimizer_gb300.autotune import autotune_buckets, cache_key, candidates, tile_candidates
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


def test_tile_candidates():
    assert tile_candidates(64) == ["packed", "single"] and tile_candidates(128) == ["packed", "single"]
    assert tile_candidates(129) == ["auto"] and tile_candidates(64, "fp32") == ["auto"]


def test_cache_and_choice_with_a_fake_timer(tmp_path):
    calls = []

    def timer(m, n, dtype, precision, route, tile, T, sample, steps, seed):
        calls.append((m, n, dtype, route, tile, sample))
        if m == 100:  # below 128 rows only Gram: packed against single
            return {("gram", "packed"): 1.0, ("gram", "single"): 2.0}[(route, tile)]
        return {"gram": 2.0, "direct": 1.0}[route] if n == 3000 else {"gram": 1.0, "direct": 3.0}[route]

    shapes = [(1000, 3000, "bf16")] * 3 + [(4000, 1000)] * 20 + [(500, 600)] * 2 + [(100, 300)] * 5
    path = str(tmp_path / "routes.json")
    choices, table = autotune_buckets(shapes, cache_path=path, sample=8, timer=timer)
    assert choices == [("direct", "auto")] * 3 + [("gram", "auto")] * 20 + [("direct", "auto")] * 2 + \
        [("gram", "packed")] * 5
    # every candidate timed once per shape, samples capped by the bucket's count
    assert sorted(calls) == sorted([(1000, 3000, "bf16", "gram", "auto", 3), (1000, 3000, "bf16", "direct", "auto", 3),
                                    (1000, 4000, "bf16", "gram", "auto", 8), (1000, 4000, "bf16", "direct", "auto", 8)] +
                                   [(100, 300, "bf16", "gram", t, 5) for t in ("packed", "single")])
    assert table[cache_key(500, 600, "bf16", "bf16", 5)] == {"candidates": ["direct/auto"], "ms_per_matrix": {},
                                                             "route": "direct", "tile": "auto"}
    # a second call reads the cache file and times nothing
    calls.clear()
    again, _ = autotune_buckets(shapes, cache_path=path, timer=timer)
    assert again == choices and not calls
    assert json.load(open(path)) == table
    # the choices go straight into the plan: one bucket per (shape, route, tile)
    plan = Muon([s[:2] + ("bf16",) + ch for s, ch in zip(shapes, choices)])
    got = {(b["m"], b["n"]): (b["route"], b["tile"]) for b in plan.buckets()}
    assert got == {(1000, 3000): (oplan.BUCKET_DIRECT, oplan.TILE_SINGLE),
                   (1000, 4000): (oplan.BUCKET_GRAM, oplan.TILE_SINGLE),
                   (500, 600): (oplan.BUCKET_DIRECT, oplan.TILE_SINGLE),
                   (100, 300): (oplan.BUCKET_GRAM, oplan.TILE_PACKED)}


@pytest.mark.gpu
def test_measured_choices_give_the_oracle_result():
    # 100-row and 64-row Gram buckets time packed against single tiles (and,
    # for m >= 128, Gram against direct); the tuned plan matches the oracle
    shapes = [(320, 1400)] * 3 + [(1400, 320)] * 2 + [(64, 512)] * 4 + [(300, 300)] * 2 + [(100, 700)] * 3
    choices, table = autotune_buckets([s + ("bf16",) for s in shapes], sample=4, steps=2)
    for (r, c), (route, tile) in zip(shapes, choices):
        m, n = min(r, c), max(r, c)
        entry = table[cache_key(m, n, "bf16", "bf16", 5)]
        assert route in candidates(m, n) and tile in tile_candidates(m)
        if len(entry["candidates"]) > 1:
            t = entry["ms_per_matrix"]
            assert set(t) == set(entry["candidates"]) and all(v > 0 for v in t.values())
            assert f"{route}/{tile}" == min(t, key=t.get)
    assert len(table[cache_key(64, 512, "bf16", "bf16", 5)]["candidates"]) == 2      # Gram, packed or single
    assert len(table[cache_key(320, 1400, "bf16", "bf16", 5)]["candidates"]) == 2    # Gram or direct
    from tests.test_gpu_parity import BETA, make_inputs
    inputs = make_inputs(shapes, "bf16", 31)
    muon = Muon([(r, c, 0) + ch for (r, c), ch in zip(shapes, choices)]).bind()
    w, _, _ = run_step(shapes, inputs, "bf16", lr=1.0, beta=BETA, wd=0.0, zero_w=True, muon=muon)
    want = oracle_O(inputs, beta=BETA)
    for (r, c), wi, o in zip(shapes, w, want):
        got = -wi.double().numpy() / oracle.shape_scale(r, c)
        assert rel_fro(got, o) <= TOL["bf16"]
