"""bench.py's CPU legs on a tiny set (no GPU): the oracle baseline times the
whole set when it is small and one matrix per (m, n) bucket otherwise, and the
reference arm's steps each time one bucket's matrix, so its per-step wall time
is real while the set's rate is extrapolated by bucket counts."""
import json
import os
import subprocess
import sys

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

TINY = workloads.Config("tiny", "tiny test set", "bf16", 7,
                        ((16, 48), (48, 16), (16, 48), (32, 32), (8, 64)), "normal", grad_scale=1e-3)


def test_cpu_baseline_buckets_and_full_or_sampled():
    full = bench.cpu_baseline(TINY)
    assert not full["extrapolated"]
    assert [(b["m"], b["n"], b["count"], b["timed"]) for b in full["per_bucket"]] == \
        [(8, 64, 1, 1), (16, 48, 3, 3), (32, 32, 1, 1)]
    sampled = bench.cpu_baseline(TINY, full_limit_tflop=0.0)
    assert sampled["extrapolated"] and all(b["timed"] == 1 for b in sampled["per_bucket"])
    for name in ("16x48", "8x64", "32x32"):
        assert name in sampled["sample"]
    assert sampled["value"] > 0 and full["value"] > 0


def test_reference_arm_steps_are_real_and_bounded():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "4", "--warmup", "1",
           "--config", "c2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    # each step one matrix: its wall time is far below the set's extrapolated time
    assert d["ms_per_step"] < 1000.0 * d["set_seconds_extrapolated"]
    assert d["config"]["workload"].startswith("c2") and d["cpu_baseline"]["extrapolated"]
    assert "768x768" in d["cpu_baseline"]["sample"] and "768x3072" in d["cpu_baseline"]["sample"]
