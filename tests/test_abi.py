"""C ABI checks that need no GPU: exports, planner bit-exactness, host-side errors."""
import ctypes
import os
import re

import pytest
import torch

import workloads
from matrix_orthogonalising_optimizer_gb300 import Muon, _lib
from oracle import plan as oplan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "dmuon.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dmuon_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = header_functions()
    assert len(names) >= 18
    for n in names:
        assert n in _lib.SIGNATURES, n
        assert hasattr(lib, n), n
    assert set(_lib.SIGNATURES) == set(names)


def _lib_plan(shapes, **kw):
    m = Muon(shapes, **kw)
    return m, m.buckets(), m.waves()


def _check_same(shapes, precision="bf16", route="auto", small_m=0, budget=0, tile="auto"):
    pmap = {"bf16": oplan.PREC_BF16, "fp32": oplan.PREC_FP32}
    rmap = {"auto": oplan.ROUTE_AUTO, "gram": oplan.ROUTE_GRAM, "direct": oplan.ROUTE_DIRECT}
    tmap = {"auto": oplan.TILE_AUTO, "packed": oplan.TILE_PACKED, "single": oplan.TILE_SINGLE}
    want_b, want_w = oplan.plan_buckets(shapes, precision=pmap[precision], route=rmap[route], small_m=small_m,
                                        budget=budget, tile=tmap[tile])
    _, got_b, got_w = _lib_plan(shapes, precision=precision, route=route, small_m=small_m,
                                workspace_budget=budget, tile=tile)
    assert len(got_b) == len(want_b)
    for g, w in zip(got_b, want_b):
        for k in ("dtype", "m", "n", "members", "route", "engine", "tile", "per_matrix_bytes"):
            assert g[k] == w[k], (k, g, w)
    assert got_w == [list(x) for x in want_w]


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_planner_matches_oracle_on_configs(name):
    cfg = workloads.get(name)
    dt = 0 if cfg.dtype == "bf16" else 1
    shapes = [(r, c, dt) for r, c in cfg.shapes]
    _check_same(shapes, precision=cfg.precision)


@pytest.mark.parametrize("seed", range(6))
def test_planner_matches_oracle_random(seed):
    g = torch.Generator().manual_seed(seed)
    shapes = [(r, c, int(torch.randint(0, 2, (1,), generator=g))) for r, c in
              workloads.random_shapes(seed, 150, 1, 700)]
    # repeat some shapes so buckets hold several matrices
    shapes = shapes + shapes[: 40]
    for prec in ("bf16", "fp32"):
        for route in ("auto", "gram", "direct"):
            _check_same(shapes, precision=prec, route=route)
    _check_same(shapes, small_m=-1)
    _check_same(shapes, small_m=100)
    b, _ = oplan.plan_buckets(shapes)
    big = max(x["per_matrix_bytes"] for x in b)
    for mult in (1, 3, 17):
        _check_same(shapes, budget=big * mult + 12345)


@pytest.mark.parametrize("seed", range(4))
def test_planner_per_shape_routes_match_oracle(seed):
    # a shape's own route overrides the plan's rule; equal shapes with
    # different routes land in different buckets (Gram before direct)
    g = torch.Generator().manual_seed(100 + seed)
    base = [(r, c, int(torch.randint(0, 2, (1,), generator=g))) for r, c in
            workloads.random_shapes(seed, 80, 1, 600)]
    base = base + base[:30]
    shapes = [s + (int(torch.randint(0, 3, (1,), generator=g)),) for s in base]
    for prec in ("bf16", "fp32"):
        for route in ("auto", "gram", "direct"):
            _check_same(shapes, precision=prec, route=route)
    b, _ = oplan.plan_buckets(shapes)
    _check_same(shapes, budget=max(x["per_matrix_bytes"] for x in b) * 5 + 999)
    # forcing a route per shape equals forcing it for the plan
    for r, name in ((1, "gram"), (2, "direct")):
        _, got, _ = _lib_plan([s[:3] + (r,) for s in base])
        _, want, _ = _lib_plan(base, route=name)
        assert got == want


@pytest.mark.parametrize("seed", range(3))
def test_planner_per_shape_tiles_match_oracle(seed):
    # a shape's own tile rule overrides the plan's; it splits buckets only where
    # packing applies (bf16, m <= 128)
    g = torch.Generator().manual_seed(200 + seed)
    base = [(r, c, 0) for r, c in workloads.random_shapes(seed, 90, 1, 300)]
    base = base + base[:40]
    shapes = [s + (int(torch.randint(0, 3, (1,), generator=g)), int(torch.randint(0, 3, (1,), generator=g)))
              for s in base]
    for prec in ("bf16", "fp32"):
        for tile in ("auto", "packed", "single"):
            _check_same(shapes, precision=prec, tile=tile)
    _, got, _ = _lib_plan(shapes)
    assert {b["tile"] for b in got if b["m"] > 128} <= {oplan.TILE_SINGLE}
    assert {b["tile"] for b in got if b["m"] <= 128} == {oplan.TILE_PACKED, oplan.TILE_SINGLE}
    # forcing a tile rule per shape equals forcing it for the plan
    for t, name in ((1, "packed"), (2, "single")):
        _, got, _ = _lib_plan([s[:3] + (0, t) for s in base])
        _, want, _ = _lib_plan(base, tile=name)
        assert got == want


def test_planner_is_order_independent_up_to_members():
    shapes = [(r, c, 0) for r, c in workloads.random_shapes(3, 80, 1, 300)]
    perm = list(reversed(range(len(shapes))))
    _, b1, _ = _lib_plan(shapes)
    _, b2, _ = _lib_plan([shapes[i] for i in perm])
    assert [(x["m"], x["n"], len(x["members"])) for x in b1] == [(x["m"], x["n"], len(x["members"])) for x in b2]
    for x, y in zip(b1, b2):
        assert sorted(x["members"]) == sorted(perm[i] for i in y["members"])


def test_plan_errors(lib):
    def plan(rows, cols, dtype=0, shape_route=0, shape_tile=0, shape_reserved=0, **kw):
        arr = (_lib.Shape * 1)()
        arr[0].rows, arr[0].cols, arr[0].dtype, arr[0].route = rows, cols, dtype, shape_route
        arr[0].tile, arr[0].reserved = shape_tile, shape_reserved
        opt = _lib.Options()
        for k, v in kw.items():
            setattr(opt, k, v)
        return lib.dmuon_plan_ex(arr, 1, ctypes.byref(opt))

    assert plan(4, 4)
    for bad in [dict(rows=0, cols=4), dict(rows=4, cols=-1), dict(rows=1 << 21, cols=1),
                dict(rows=1 << 20, cols=1 << 20), dict(rows=4, cols=4, dtype=7), dict(rows=4, cols=4, shape_route=3),
                dict(rows=4, cols=4, shape_route=-1),
                dict(rows=4, cols=4, precision=9), dict(rows=4, cols=4, route=5), dict(rows=4, cols=4, eps=-1.0),
                dict(rows=4, cols=4, scale_rule=3), dict(rows=4, cols=4, no_nesterov=2),
                dict(rows=4, cols=4, shape_tile=3), dict(rows=4, cols=4, shape_tile=-1),
                dict(rows=4, cols=4, shape_reserved=1), dict(rows=4, cols=4, tile_rule=3)]:
        assert not plan(**bad), bad
        assert lib.dmuon_last_error()
    assert not lib.dmuon_plan(None, 1)
    arr = (_lib.Shape * 1)()
    arr[0].rows, arr[0].cols = 4, 4
    assert not lib.dmuon_plan(arr, 0)
    # a budget below one matrix is refused
    assert not plan(64, 64, workspace_budget=1000)


def test_step_host_errors(lib):
    m = Muon([(8, 16), (16, 8)])
    p = (ctypes.c_void_p * 2)(16, 32)
    st = lib.dmuon_step(m.handle, p, p, p, 0.02, 0.95, 0.01, 5, None)
    assert st == _lib.ERR_NO_WORKSPACE
    assert lib.dmuon_step(None, p, p, p, 0.02, 0.95, 0.01, 5, None) == _lib.ERR_INVALID_ARG
    assert lib.dmuon_bind_workspace(m.handle, ctypes.c_void_p(0x1001), 1 << 30) == _lib.ERR_WORKSPACE_TOO_SMALL
    assert lib.dmuon_bind_workspace(m.handle, ctypes.c_void_p(0x100000), 16) == _lib.ERR_WORKSPACE_TOO_SMALL
    assert lib.dmuon_device_status(m.handle, None) == _lib.ERR_NO_WORKSPACE
    assert lib.dmuon_status_string(_lib.ERR_ALIGN) == b"pointer not 16-byte aligned"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_bind_refuses_without_gpu(lib):
    m = Muon([(8, 16)])
    st = lib.dmuon_bind_workspace(m.handle, ctypes.c_void_p(1 << 20), m.workspace_bytes())
    assert st in (_lib.ERR_CUDA, _lib.ERR_UNSUPPORTED_DEVICE)


def test_plan_flops_formula():
    cfg = workloads.get("c3")
    m = Muon([(r, c, 0) for r, c in cfg.shapes])
    total, tc = m.flops(5)
    # c3: 64 x 1024x4096 Gram, 64 x 4096^2 direct, 96 x 4096x14336 Gram
    want = 64 * (3 * 1024 ** 2 * 4096 + 17 * 1024 ** 3) + 64 * 5 * (3 * 4096 ** 3 + 4096 ** 3) \
        + 96 * (3 * 4096 ** 2 * 14336 + 17 * 4096 ** 3)
    assert total == pytest.approx(want, rel=1e-12)
    assert tc == pytest.approx(want, rel=1e-12)
    assert m.workspace_bytes() > 0
