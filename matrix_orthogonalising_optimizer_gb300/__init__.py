"""GB300 batched Gram-space Newton-Schulz Muon step.

A thin binding over the C ABI of ``include/dmuon.h`` (``libdmuon.so``): it
only marshals arguments.  Every step of the computation runs in the CUDA
kernels; PyTorch supplies device memory (the workspace) and streams.  There
is no CPU fallback: without the built library every call raises.

Subject: "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead"
(arXiv 2606.27153), the per-owner Gram Newton-Schulz engine of its section
2.2 (gist.science technical summary), on one GPU.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (  # noqa: F401
    BF16, FP32, PREC_BF16, PREC_FP32, ROUTE_AUTO, ROUTE_GRAM, ROUTE_DIRECT, BUCKET_GRAM, BUCKET_DIRECT,
    ENGINE_TC_BF16, ENGINE_SIMT_FP32, ENGINE_TC_SPLIT, TILE_AUTO, TILE_PACKED, TILE_SINGLE, SCALE_ASPECT, SCALE_RMS, TIMER_NAMES, ASSIGN_GREEDY, ASSIGN_EXACT, DmuonError,
)

__all__ = ["Muon", "dmuon_plan", "dmuon_step", "assign_owners", "adamw_step", "load"]

_DTYPES = {"bf16": BF16, "fp32": FP32}
_PREC = {"bf16": PREC_BF16, "fp32": PREC_FP32}
_ROUTES = {"auto": ROUTE_AUTO, "gram": ROUTE_GRAM, "direct": ROUTE_DIRECT}
_SCALES = {"aspect": SCALE_ASPECT, "rms": SCALE_RMS}
_TILES = {"auto": TILE_AUTO, "packed": TILE_PACKED, "single": TILE_SINGLE}


def load():
    return _lib.load()


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def dmuon_plan(shapes, dtype="bf16", precision="bf16", route="auto", coeffs=None, eps=0.0,
               scale_rule="aspect", nesterov=True, small_m=0, workspace_budget=0, tile="auto"):
    """dmuon_plan_ex: shapes is a list of (rows, cols[, dtype[, route[, tile]]]); a shape's
    route ("auto" / 0 = the plan's ``route``, "gram", "direct") and tile rule ("auto" / 0 =
    the plan's ``tile``, "packed", "single") override the plan's rules."""
    lib = _lib.load()
    arr = (_lib.Shape * len(shapes))()
    for i, s in enumerate(shapes):
        dt = s[2] if len(s) > 2 else dtype
        arr[i].rows, arr[i].cols = int(s[0]), int(s[1])
        arr[i].dtype = _DTYPES[dt] if isinstance(dt, str) else int(dt)
        rt = s[3] if len(s) > 3 else 0
        arr[i].route = _ROUTES[rt] if isinstance(rt, str) else int(rt)
        tl = s[4] if len(s) > 4 else 0
        arr[i].tile = _TILES[tl] if isinstance(tl, str) else int(tl)
    opt = _lib.Options()
    opt.precision = _PREC[precision]
    opt.route = _ROUTES[route]
    if coeffs is not None:
        opt.ns_a, opt.ns_b, opt.ns_c = coeffs
    opt.eps = eps
    opt.scale_rule = _SCALES[scale_rule]
    opt.no_nesterov = 0 if nesterov else 1
    opt.small_m = small_m
    opt.tile_rule = _TILES[tile]
    opt.workspace_budget = workspace_budget
    h = lib.dmuon_plan_ex(arr, len(shapes), ctypes.byref(opt))
    if not h:
        raise DmuonError(_lib.ERR_INVALID_ARG, "dmuon_plan_ex")
    return h


def dmuon_step(h, params, grads, momenta, lr, beta, wd, ns_steps=5, stream=None, params_ready=None):
    """dmuon_step over lists of device tensors (or raw device pointers); with ``params_ready``
    (a recorded torch.cuda.Event) dmuon_step_ex: the first parameter write waits for it."""
    lib = _lib.load()
    n = len(params)

    def ptrs(xs):
        a = (ctypes.c_void_p * n)()
        for i, x in enumerate(xs):
            a[i] = x if isinstance(x, int) else x.data_ptr()
        return a

    if params_ready is None:
        st = lib.dmuon_step(h, ptrs(params), ptrs(grads), ptrs(momenta), lr, beta, wd, ns_steps,
                            _stream_handle(stream))
    else:
        ev = params_ready if isinstance(params_ready, int) else params_ready.cuda_event
        st = lib.dmuon_step_ex(h, ptrs(params), ptrs(grads), ptrs(momenta), lr, beta, wd, ns_steps,
                               _stream_handle(stream), ctypes.c_void_p(ev))
    _lib.check(st, "dmuon_step")


_ASSIGN = {"greedy": ASSIGN_GREEDY, "exact": ASSIGN_EXACT}


def adamw_step(params, grads, exp_avgs, exp_avg_sqs, lr, beta1, beta2, eps, wd, step, stream=None):
    """dmuon_adamw_step over lists of device tensors of one dtype each (bf16 or fp32)."""
    import torch
    lib = _lib.load()
    n = len(params)
    dts = {torch.bfloat16: BF16, torch.float32: FP32}

    def ptrs(xs):
        a = (ctypes.c_void_p * max(n, 1))()
        for i, x in enumerate(xs):
            a[i] = x.data_ptr()
        return a

    numel = (ctypes.c_int64 * max(n, 1))(*[p.numel() for p in params])
    dtype = (ctypes.c_int32 * max(n, 1))(*[dts.get(p.dtype, -1) for p in params])
    st = lib.dmuon_adamw_step(ptrs(params), ptrs(grads), ptrs(exp_avgs), ptrs(exp_avg_sqs), numel, dtype, n,
                              lr, beta1, beta2, eps, wd, int(step), _stream_handle(stream))
    _lib.check(st, "dmuon_adamw_step")


def assign_owners(costs, ranks, method="greedy"):
    """dmuon_assign_owners: (owner rank per matrix, makespan) for predicted costs."""
    lib = _lib.load()
    n = len(costs)
    arr = (ctypes.c_double * max(n, 1))(*[float(c) for c in costs])
    owner = (ctypes.c_int32 * max(n, 1))()
    ms = ctypes.c_double()
    _lib.check(lib.dmuon_assign_owners(arr, n, int(ranks), _ASSIGN[method], owner, ctypes.byref(ms)),
               "dmuon_assign_owners")
    return [int(owner[i]) for i in range(n)], ms.value


class Muon:
    """One plan bound to a workspace: ``Muon(shapes).step(params, grads, moms, lr, beta, wd)``.

    ``shapes``: list of (rows, cols[, dtype]).  The workspace is a torch uint8
    tensor on the current CUDA device unless one is passed to ``bind``.
    """

    def __init__(self, shapes, **plan_kw):
        self.lib = _lib.load()
        self.shapes = [tuple(s) for s in shapes]
        self.handle = dmuon_plan(shapes, **plan_kw)
        self.workspace = None

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            self.lib.dmuon_destroy(h)
            self.handle = None

    # ---- plan queries
    def workspace_bytes(self) -> int:
        return int(self.lib.dmuon_workspace_bytes(self.handle))

    def buckets(self):
        out = []
        for b in range(self.lib.dmuon_plan_num_buckets(self.handle)):
            info = _lib.BucketInfo()
            _lib.check(self.lib.dmuon_plan_bucket(self.handle, b, ctypes.byref(info)), "dmuon_plan_bucket")
            mem = (ctypes.c_int64 * info.count)()
            _lib.check(self.lib.dmuon_plan_bucket_members(self.handle, b, mem), "dmuon_plan_bucket_members")
            out.append({"dtype": info.dtype, "m": info.m, "n": info.n, "route": info.route,
                        "engine": info.mm_engine, "tile": info.tile, "per_matrix_bytes": info.per_matrix_bytes,
                        "members": list(mem)})
        return out

    def waves(self):
        out = []
        for w in range(self.lib.dmuon_plan_num_waves(self.handle)):
            pieces = []
            for p in range(self.lib.dmuon_plan_wave_num_pieces(self.handle, w)):
                b, s, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
                _lib.check(self.lib.dmuon_plan_wave_piece(self.handle, w, p, ctypes.byref(b), ctypes.byref(s),
                                                          ctypes.byref(c)), "dmuon_plan_wave_piece")
                pieces.append((b.value, s.value, c.value))
            out.append(pieces)
        return out

    def flops(self, ns_steps=5):
        out = (ctypes.c_double * 2)()
        _lib.check(self.lib.dmuon_plan_flops(self.handle, ns_steps, out), "dmuon_plan_flops")
        return out[0], out[1]

    def matrix_flops(self, ns_steps=5):
        """Per-matrix algorithmic FLOPs of one step, in the order of the shapes."""
        out = (ctypes.c_double * max(len(self.shapes), 1))()
        _lib.check(self.lib.dmuon_plan_matrix_flops(self.handle, ns_steps, out), "dmuon_plan_matrix_flops")
        return [out[i] for i in range(len(self.shapes))]

    # ---- device
    def bind(self, workspace=None):
        import torch
        nbytes = self.workspace_bytes()
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.workspace = workspace
        _lib.check(self.lib.dmuon_bind_workspace(self.handle, ctypes.c_void_p(workspace.data_ptr()),
                                                 workspace.numel() * workspace.element_size()),
                   "dmuon_bind_workspace")
        return self

    def step(self, params, grads, momenta, lr, beta, wd, ns_steps=5, stream=None, params_ready=None):
        dmuon_step(self.handle, params, grads, momenta, lr, beta, wd, ns_steps, stream, params_ready)

    def device_status(self, stream=None) -> int:
        return int(self.lib.dmuon_device_status(self.handle, _stream_handle(stream)))

    def set_timing(self, enable: bool):
        _lib.check(self.lib.dmuon_set_timing(self.handle, 1 if enable else 0), "dmuon_set_timing")

    def timing(self):
        n = len(TIMER_NAMES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        _lib.check(self.lib.dmuon_get_timing(self.handle, ms, cnt, n), "dmuon_get_timing")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(TIMER_NAMES)}

    def debug_buffer(self, wave, piece, which):
        """(byte offset, leading dimension, batch stride, dtype 'bf16'|'fp32') of a workspace buffer."""
        off, ld, bs, et = ctypes.c_uint64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _lib.check(self.lib.dmuon_debug_buffer(self.handle, wave, piece, which, ctypes.byref(off), ctypes.byref(ld),
                                               ctypes.byref(bs), ctypes.byref(et)), "dmuon_debug_buffer")
        return off.value, ld.value, bs.value, "bf16" if et.value == BF16 else "fp32"
