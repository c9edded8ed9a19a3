"""Pins of the fp64 oracle against what the mathematics fixes (no GPU).

The pages print no worked example and no coefficients, so every pin here is a
closed form, an invariant, a special case or a brute-force computation that
does not reuse the oracle's own arithmetic:

* the Newton-Schulz result equals U f^T(S) V^T, f the scalar quintic,
  with U, S, V from a one-sided Jacobi SVD written here;
* its singular values land in the band the scalar map f^5 gives;
* Gram-space and direct NS agree (the identity behind the summary's
  section 2.2 "Gram Newton-Schulz iteration");
* an orthonormal input is mapped to f^5(m^-1/2) times itself;
* the golden table tests/golden/quintic_map.txt (f^k(s) iterated in exact
  rational arithmetic by tests/golden/make_quintic_map.py) on diagonal and
  rotated inputs;
* zero, rank-1, scaled and transposed inputs;
* the whole update (1 - lr wd) W - lr s O on an input of equal singular
  values, whose O is f^5(0.25) times its direction (golden table);
* bf16 round-to-nearest-even against hand-made halfway cases and torch;
* the planner rules against hand-worked bucket lists.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import plan as oplan

A, B, C = 3.4445, -4.7750, 2.0315


def f(s):
    return A * s + B * s ** 3 + C * s ** 5


def f_iter(s, t):
    for _ in range(t):
        s = f(s)
    return s


def jacobi_svd(a, sweeps=80):
    """One-sided (Hestenes) Jacobi SVD of a (m x n, m <= n): a = U diag(s) Vt."""
    bm = np.array(a, dtype=np.float64)
    m = bm.shape[0]
    u = np.eye(m)
    for _ in range(sweeps):
        rotated = False
        for i in range(m - 1):
            for j in range(i + 1, m):
                alpha = bm[i] @ bm[i]
                beta = bm[j] @ bm[j]
                gamma = bm[i] @ bm[j]
                if abs(gamma) <= 1e-15 * math.sqrt(alpha * beta):
                    continue
                rotated = True
                zeta = (beta - alpha) / (2.0 * gamma)
                t = (1.0 if zeta >= 0 else -1.0) / (abs(zeta) + math.sqrt(1.0 + zeta * zeta))
                c = 1.0 / math.sqrt(1.0 + t * t)
                s = c * t
                bi, bj = bm[i].copy(), bm[j].copy()
                bm[i], bm[j] = c * bi - s * bj, s * bi + c * bj
                ui, uj = u[:, i].copy(), u[:, j].copy()
                u[:, i], u[:, j] = c * ui - s * uj, s * ui + c * uj
        if not rotated:
            break
    sig = np.sqrt(np.sum(bm * bm, axis=1))
    return u, sig, bm / sig[:, None]


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(b))


# ---------------------------------------------------------------- rounding


def test_bf16_rounding_halfway_and_limits():
    r = oracle.round_to_bf16
    # halfway between 1 and 1+2^-7 goes to the even neighbour 1
    assert r(1.0 + 2.0 ** -8) == 1.0
    # halfway between 1+2^-7 and 1+2^-6 goes to 1+2^-6 (even significand)
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # just above halfway rounds up
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert r(-(1.0 + 2.0 ** -8)) == -1.0
    # subnormals: quantum 2^-133
    assert r(2.0 ** -134) == 0.0
    assert r(3 * 2.0 ** -134) == 2.0 ** -132
    assert r(2.0 ** -133) == 2.0 ** -133
    # largest finite bf16 and overflow
    bmax = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert r(bmax) == bmax
    assert r(bmax + 2.0 ** 119) == math.inf
    assert r(bmax + 2.0 ** 118) == bmax
    assert math.isnan(r(math.nan))
    assert r(0.0) == 0.0


def test_bf16_rounding_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 10)
    want = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(x.to(torch.float64).numpy())
    assert np.array_equal(got, want)


def test_bf16_rounding_is_nearest():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)
    y = oracle.round_to_bf16(x)
    bits = y.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)                         # representable in bf16
    _, e = np.frexp(x)
    half_ulp = np.ldexp(1.0, np.maximum(e, -125) - 9)
    assert np.all(np.abs(y - x) <= half_ulp)


# ---------------------------------------------------------------- momentum


def test_nesterov_worked_example():
    mom_new, u = oracle.nesterov_momentum(np.array([[1.0]]), np.array([[2.0]]), 0.5)
    assert mom_new[0, 0] == 2.0            # 0.5*2 + 1
    assert u[0, 0] == 2.0                  # 1 + 0.5*2
    mom_new, u = oracle.nesterov_momentum(np.array([[3.0]]), np.array([[-4.0]]), 0.25, nesterov=False)
    assert mom_new[0, 0] == 2.0 and u[0, 0] == 2.0


# ---------------------------------------------------------------- NS core


@pytest.mark.parametrize("m,n,seed", [(8, 16, 0), (16, 64, 1), (8, 8, 2)])
def test_ns_closed_form_jacobi(m, n, seed):
    rng = np.random.default_rng(seed)
    x0 = oracle.frobenius_normalise(rng.standard_normal((m, n)))
    u, s, vt = jacobi_svd(x0)
    assert np.allclose(u @ np.diag(s) @ vt, x0, atol=1e-14)
    want = u @ np.diag(f_iter(s, 5)) @ vt
    assert rel(oracle.ns_direct(x0, 5), want) < 1e-12
    assert rel(oracle.ns_gram(x0, 5), want) < 1e-12
    want3 = u @ np.diag(f_iter(s, 3)) @ vt
    assert rel(oracle.ns_direct(x0, 3), want3) < 1e-12


def test_ns_band():
    grid = np.linspace(0.01, 1.0, 200001)
    img = f_iter(grid, 5)
    lo, hi = img.min(), img.max()
    assert 0.68 < lo < 0.69 and 1.13 < hi < 1.14           # attracting band of the quintic
    rng = np.random.default_rng(3)
    for m, n in [(8, 16), (32, 48), (16, 256)]:
        x = rng.standard_normal((m, n))
        x0 = oracle.frobenius_normalise(x)
        s0 = np.linalg.svd(x0, compute_uv=False)
        out = np.linalg.svd(oracle.ns_direct(x0, 5), compute_uv=False)
        keep = s0 >= 0.01
        assert np.all(out[keep] >= lo - 1e-9) and np.all(out[keep] <= hi + 1e-9)


def test_ns_band_vs_uv():
    # The quintic does not reach U V^T exactly: distance about 0.2 relative on a Gaussian 8x16.
    rng = np.random.default_rng(0)
    x0 = oracle.frobenius_normalise(rng.standard_normal((8, 16)))
    u, s, vt = jacobi_svd(x0)
    d = rel(oracle.ns_direct(x0, 5), u @ vt)
    assert 0.02 < d < 0.35


@pytest.mark.parametrize("m,n", [(8, 16), (16, 64), (64, 64), (5, 37)])
def test_gram_equals_direct(m, n):
    rng = np.random.default_rng(m * 1000 + n)
    x0 = oracle.frobenius_normalise(rng.standard_normal((m, n)))
    assert rel(oracle.ns_gram(x0, 5), oracle.ns_direct(x0, 5)) < 1e-12


def test_orthonormal_input():
    rng = np.random.default_rng(7)
    q, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    o = q[:8]                                   # orthonormal rows, 8 x 16
    x0 = oracle.frobenius_normalise(o)
    k = f_iter(1.0 / (math.sqrt(8.0) + 1e-7), 5)
    assert abs(f_iter(1.0 / math.sqrt(8.0), 5) - 1.066968) < 1e-6
    assert rel(oracle.ns_direct(x0, 5), k * o) < 1e-12


def test_gram_symmetric_bitwise():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((40, 70))
    g = x @ x.T
    assert np.array_equal(g, g.T)


# ---------------------------------------------------------------- full step


def _f32(v):
    return float(np.float32(v))


def test_zero_input():
    w = oracle.round_to_bf16(np.random.default_rng(0).standard_normal((6, 9)) * 0.02)
    z = np.zeros((6, 9))
    lr, wd, beta = _f32(0.02), _f32(0.01), _f32(0.95)
    out = oracle.muon_step(w, z, z, lr=lr, beta=beta, wd=wd)
    assert np.all(out["O"] == 0.0)
    assert np.array_equal(out["W"], oracle.round_to_bf16((1.0 - lr * wd) * w))
    assert np.all(out["M"] == 0.0)


def test_rank_one():
    rng = np.random.default_rng(2)
    a = rng.standard_normal(6)
    a /= np.linalg.norm(a)
    b = rng.standard_normal(10)
    b /= np.linalg.norm(b)
    grad = 5.0 * np.outer(a, b)
    out = oracle.muon_step(np.zeros((6, 10)), grad, np.zeros((6, 10)), lr=1.0, beta=0.0, wd=0.0,
                           dtype="fp32")
    s0 = 5.0 / (5.0 + 1e-7)
    assert rel(out["O"], f_iter(s0, 5) * np.outer(a, b)) < 1e-12


def test_scale_invariance_and_transpose():
    rng = np.random.default_rng(4)
    grad = rng.standard_normal((12, 30))
    z = np.zeros_like(grad)
    kw = dict(lr=1.0, beta=0.0, wd=0.0, dtype="fp32")
    o1 = oracle.muon_step(z, grad, z, **kw)["O"]
    o2 = oracle.muon_step(z, 1000.0 * grad, z, **kw)["O"]
    assert rel(o2, o1) < 1e-7
    ot = oracle.muon_step(z.T, grad.T, z.T, **kw)["O"]
    assert np.array_equal(ot, o1.T)


def test_update_and_scale_rules():
    rng = np.random.default_rng(9)
    rows, cols = 20, 5                      # tall: s = sqrt(4) = 2
    w = oracle.round_to_fp32(rng.standard_normal((rows, cols)) * 0.02)
    grad = oracle.round_to_fp32(rng.standard_normal((rows, cols)))
    mom = oracle.round_to_fp32(rng.standard_normal((rows, cols)) * 1e-3)
    lr, beta, wd = 0.02, 0.95, 0.01
    out = oracle.muon_step(w, grad, mom, lr=lr, beta=beta, wd=wd, dtype="fp32")
    assert oracle.shape_scale(rows, cols) == 2.0
    assert oracle.shape_scale(cols, rows) == 1.0
    assert oracle.shape_scale(rows, cols, "rms") == pytest.approx(0.2 * math.sqrt(20))
    mom_new = beta * mom + grad
    u = grad + beta * mom_new
    want_o = oracle.ns_direct(oracle.frobenius_normalise(u.T), 5).T
    assert rel(out["O"], want_o) < 1e-14
    assert np.array_equal(out["M"], oracle.round_to_fp32(mom_new))
    assert np.array_equal(out["W"], oracle.round_to_fp32((1 - lr * wd) * w - lr * 2.0 * want_o))
    # Nesterov off: the direction is M' itself
    out2 = oracle.muon_step(w, grad, mom, lr=lr, beta=beta, wd=wd, dtype="fp32", nesterov=False)
    want2 = oracle.ns_direct(oracle.frobenius_normalise(mom_new.T), 5).T
    assert rel(out2["O"], want2) < 1e-14


@pytest.mark.parametrize("dtype,scale_rule", [("fp32", "aspect"), ("bf16", "aspect"), ("fp32", "rms")])
def test_update_term_closed_form(dtype, scale_rule):
    # The whole update W' = (1 - lr wd) W - lr s O against a closed form, with
    # W != 0, lr != 1, wd != 0 and beta != 0, so that every term is visible.
    # The gradient is k V with V (40 x 16, tall) of orthonormal columns: the
    # step transposes it to X = (1 + beta) k V^T, whose 16 singular values are
    # all equal, and normalisation makes each one 0.25 (to 2.5e-13 for the
    # chosen k).  Newton-Schulz then maps V^T to f^5(0.25) V^T, f^5(0.25) read
    # from the exact-rational golden table, so O = f^5(0.25) V.  The expected
    # W' below is written from these facts alone; a dropped lr, a flipped
    # sign, a wrong decay or scale, or a missing transpose moves W' by far
    # more than one storage ulp.
    rows, cols = 40, 16
    rng = np.random.default_rng(31)
    v, _ = np.linalg.qr(rng.standard_normal((rows, cols)))   # orthonormal columns
    lr, wd, beta = _f32(0.02), _f32(0.01), _f32(0.9)
    big = 1e5 / (1.0 + beta)                                   # (1 + beta) k = 1e5
    grad = big * v
    w = oracle.round_to_storage(rng.standard_normal((rows, cols)) * 0.02, dtype)
    out = oracle.muon_step(w, grad, np.zeros_like(grad), lr=lr, beta=beta, wd=wd, dtype="fp32" if dtype == "fp32"
                           else "bf16", scale_rule=scale_rule)
    table = dict((s, vals) for s, vals in _quintic_table())
    f5 = table[0.25][4]
    s = math.sqrt(rows / cols) if scale_rule == "aspect" else 0.2 * math.sqrt(max(rows, cols))
    exact = (1.0 - lr * wd) * w - lr * s * f5 * v
    assert rel(out["O"], f5 * v) < 1e-10
    want = oracle.round_to_storage(exact, dtype)
    st = torch.float32 if dtype == "fp32" else torch.bfloat16
    got_t, want_t = torch.from_numpy(out["W"]).to(st), torch.from_numpy(want).to(st)
    # both round values that agree to ~1e-11 relative: equal unless within that of a tie
    bits = torch.int32 if dtype == "fp32" else torch.int16
    d = (got_t.view(bits).to(torch.int64) - want_t.view(bits).to(torch.int64)).abs()
    assert int(d.max()) <= 1 and float((d == 0).double().mean()) >= 0.99
    # the decay term alone and the update term alone are each far above one ulp here
    assert np.sqrt(np.mean((lr * wd * w) ** 2)) > 1e-6 and np.sqrt(np.mean((lr * s * f5 * v) ** 2)) > 1e-4


def test_gram_method_in_step_matches_direct():
    rng = np.random.default_rng(12)
    grad = rng.standard_normal((24, 10))
    z = np.zeros_like(grad)
    kw = dict(lr=1.0, beta=0.9, wd=0.0, dtype="fp32")
    assert rel(oracle.muon_step(z, grad, z, method="gram", **kw)["O"],
               oracle.muon_step(z, grad, z, **kw)["O"]) < 1e-12


# ---------------------------------------------------------------- planner rules


def test_plan_small_transformer_buckets():
    shapes = [(768, 2304, 0), (768, 768, 0), (768, 3072, 0), (3072, 768, 0)] * 12
    buckets, waves = oplan.plan_buckets(shapes)
    got = [(b["m"], b["n"], len(b["members"]), b["route"], b["engine"]) for b in buckets]
    assert got == [(768, 768, 12, oplan.BUCKET_DIRECT, oplan.ENGINE_TC_BF16),
                   (768, 2304, 12, oplan.BUCKET_GRAM, oplan.ENGINE_TC_BF16),
                   (768, 3072, 24, oplan.BUCKET_GRAM, oplan.ENGINE_TC_BF16)]
    assert buckets[2]["members"][:4] == [2, 3, 6, 7]        # input order, wide and tall mixed
    assert waves == [[(0, 0, 12), (1, 0, 12), (2, 0, 24)]]


def test_plan_per_matrix_bytes_hand_worked():
    # m=3, n=5 Gram bucket on tensor cores: ldm = ldn = 8
    # u: 3*8*2=48 -> 256; five bf16 m x m: 48 -> 256 each;
    # partials (8 per tile, one tile) 32 -> 256
    assert oplan.per_matrix_bytes(3, 5, oplan.PREC_BF16, oplan.BUCKET_GRAM, oplan.ENGINE_TC_BF16) == 7 * 256
    # direct bucket, bf16: u, X1, A, B -> 4 * 256, partials 256
    assert oplan.per_matrix_bytes(3, 5, oplan.PREC_BF16, oplan.BUCKET_DIRECT, oplan.ENGINE_TC_BF16) == 5 * 256
    # 1024 x 4096 bf16 Gram, tensor cores
    m, n = 1024, 4096
    want = m * n * 2 + 5 * m * m * 2 + 4 * 8 * 16 * 64
    assert oplan.per_matrix_bytes(m, n, oplan.PREC_BF16, oplan.BUCKET_GRAM, oplan.ENGINE_TC_BF16) == want


def test_plan_per_matrix_bytes_split_engine_hand_worked():
    # m=100, n=700 bf16 Gram bucket with split m x m operands: ldn = 704,
    # ldm = 104; each split operand row is [hi | lo] with both parts 128 long
    # u: 100*704*2 = 140800 -> 140800 (550 * 256); Rf: 100*104*4 = 41600 -> 41728;
    # five split operands: 100*256*2 = 51200 (= 200 * 256) each;
    # partials: 2 x 11 tiles, 8 floats each: 704 -> 768
    want = 140800 + 41728 + 5 * 51200 + 768
    assert oplan.per_matrix_bytes(100, 700, oplan.PREC_BF16, oplan.BUCKET_GRAM, oplan.ENGINE_TC_SPLIT) == want
    b, _ = oplan.plan_buckets([(700, 100, 0)])
    assert (b[0]["route"], b[0]["engine"], b[0]["per_matrix_bytes"]) == (oplan.BUCKET_GRAM, oplan.ENGINE_TC_SPLIT,
                                                                        want)


def test_plan_waves_split_buckets():
    shapes = [(64, 64, 0)] * 5 + [(64, 128, 0)] * 3
    b0, _ = oplan.plan_buckets(shapes)
    p0, p1 = b0[0]["per_matrix_bytes"], b0[1]["per_matrix_bytes"]
    budget = 2 * p0 + p1 // 2                      # two of the first kind fit, no second kind alone
    budget = max(budget, p1)
    buckets, waves = oplan.plan_buckets(shapes, budget=budget)
    flat = [pc for w in waves for pc in w]
    assert sum(c for b, s, c in flat if b == 0) == 5
    assert sum(c for b, s, c in flat if b == 1) == 3
    for w in waves:
        assert sum(c * buckets[b]["per_matrix_bytes"] for b, s, c in w) <= budget
    with pytest.raises(ValueError):
        oplan.plan_buckets(shapes, budget=p0 - 1)


def test_plan_fp32_and_forced_routes():
    shapes = [(100, 100, 1), (10, 300, 1), (300, 10, 0)]
    b, _ = oplan.plan_buckets(shapes, precision=oplan.PREC_FP32)
    assert [x["route"] for x in b] == [oplan.BUCKET_GRAM] * 3
    assert all(x["engine"] == oplan.ENGINE_SIMT_FP32 for x in b)
    b, _ = oplan.plan_buckets(shapes, route=oplan.ROUTE_DIRECT)
    assert [x["route"] for x in b] == [oplan.BUCKET_DIRECT] * 3
    b, _ = oplan.plan_buckets([(600, 700, 0), (200, 210, 0)], small_m=-1)
    assert [x["route"] for x in b] == [oplan.BUCKET_DIRECT, oplan.BUCKET_DIRECT]
    b, _ = oplan.plan_buckets([(600, 700, 0), (200, 210, 0)])
    assert [(x["route"], x["engine"]) for x in b] == [(oplan.BUCKET_GRAM, oplan.ENGINE_TC_SPLIT),
                                                      (oplan.BUCKET_DIRECT, oplan.ENGINE_TC_BF16)]


def _quintic_table():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "quintic_map.txt")
    rows = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        rows.append((float(parts[0]), [float(x) for x in parts[1:]]))
    return rows


@pytest.mark.parametrize("route", ["direct", "gram"])
def test_ns_singular_values_follow_the_exact_scalar_map(route):
    # golden table: f^k(s) iterated in exact rational arithmetic by
    # tests/golden/make_quintic_map.py.  Diagonal input: the singular values
    # are the starting values, and k steps map each one to f^k(s) exactly
    # (up to fp64 rounding).  Rotated input: the same singular values.
    rows = _quintic_table()
    s = np.array([r[0] for r in rows])
    m, n = len(s), len(s) + 7
    rng = np.random.default_rng(5)
    u, _ = np.linalg.qr(rng.standard_normal((m, m)))
    v, _ = np.linalg.qr(rng.standard_normal((n, n)))
    ns = oracle.ns_direct if route == "direct" else oracle.ns_gram
    for k in range(1, 7):
        want = np.array([r[1][k - 1] for r in rows])
        x0 = np.zeros((m, n))
        x0[np.arange(m), np.arange(m)] = s
        out = ns(x0, k)
        np.testing.assert_allclose(np.diag(out[:, :m]), want, rtol=1e-12, atol=1e-15)
        assert np.abs(out[:, m:]).max() == 0.0
        rot = ns(u @ x0 @ v.T, k)
        np.testing.assert_allclose(np.sort(np.linalg.svd(rot, compute_uv=False)), np.sort(want), rtol=1e-10)
