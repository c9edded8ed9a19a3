"""ctypes declarations of the C ABI in include/dmuon.h (marshalling only)."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdmuon.so")

# constants of include/dmuon.h
BF16, FP32 = 0, 1
PREC_BF16, PREC_FP32 = 0, 1
ROUTE_AUTO, ROUTE_GRAM, ROUTE_DIRECT = 0, 1, 2
BUCKET_GRAM, BUCKET_DIRECT = 1, 2
ENGINE_TC_BF16, ENGINE_SIMT_FP32, ENGINE_TC_SPLIT = 0, 1, 2
TILE_AUTO, TILE_PACKED, TILE_SINGLE = 0, 1, 2
SCALE_ASPECT, SCALE_RMS = 0, 1
OK = 0
ERR_INVALID_ARG, ERR_ALIGN, ERR_NO_WORKSPACE, ERR_UNSUPPORTED_DTYPE = -1, -2, -3, -4
ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_UNSUPPORTED_DEVICE, ERR_WORKSPACE_TOO_SMALL = -5, -6, -7, -8
MAX_NS_STEPS = 16
TIMER_NAMES = ("momentum", "norm", "syrk", "ns", "final", "tc", "simt")
BUF_X, BUF_RF, BUF_R_OPERAND = 0, 1, 2
ASSIGN_GREEDY, ASSIGN_EXACT = 0, 1


class Shape(ctypes.Structure):
    _fields_ = [("rows", c_int64), ("cols", c_int64), ("dtype", c_int32), ("route", c_int32), ("tile", c_int32),
                ("reserved", c_int32)]


class Options(ctypes.Structure):
    _fields_ = [("precision", c_int32), ("route", c_int32), ("ns_a", c_float), ("ns_b", c_float),
                ("ns_c", c_float), ("eps", c_float), ("scale_rule", c_int32), ("no_nesterov", c_int32),
                ("small_m", c_int32), ("tile_rule", c_int32), ("workspace_budget", c_uint64)]


class BucketInfo(ctypes.Structure):
    _fields_ = [("dtype", c_int32), ("route", c_int32), ("mm_engine", c_int32), ("tile", c_int32),
                ("m", c_int64), ("n", c_int64), ("count", c_int64), ("per_matrix_bytes", c_int64)]


# name -> (restype, argtypes); every function include/dmuon.h declares
SIGNATURES = {
    "dmuon_plan": (c_void_p, [POINTER(Shape), c_int64]),
    "dmuon_plan_ex": (c_void_p, [POINTER(Shape), c_int64, POINTER(Options)]),
    "dmuon_destroy": (None, [c_void_p]),
    "dmuon_plan_num_buckets": (c_int64, [c_void_p]),
    "dmuon_plan_bucket": (c_int, [c_void_p, c_int64, POINTER(BucketInfo)]),
    "dmuon_plan_bucket_members": (c_int, [c_void_p, c_int64, POINTER(c_int64)]),
    "dmuon_plan_num_waves": (c_int64, [c_void_p]),
    "dmuon_plan_wave_num_pieces": (c_int64, [c_void_p, c_int64]),
    "dmuon_plan_wave_piece": (c_int, [c_void_p, c_int64, c_int64, POINTER(c_int64), POINTER(c_int64),
                                      POINTER(c_int64)]),
    "dmuon_plan_flops": (c_int, [c_void_p, c_int32, POINTER(c_double)]),
    "dmuon_workspace_bytes": (c_size_t, [c_void_p]),
    "dmuon_bind_workspace": (c_int, [c_void_p, c_void_p, c_size_t]),
    "dmuon_step": (c_int, [c_void_p, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p), c_float, c_float,
                           c_float, c_int32, c_void_p]),
    "dmuon_step_ex": (c_int, [c_void_p, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p), c_float,
                              c_float, c_float, c_int32, c_void_p, c_void_p]),
    "dmuon_device_status": (c_int, [c_void_p, c_void_p]),
    "dmuon_set_timing": (c_int, [c_void_p, c_int32]),
    "dmuon_get_timing": (c_int, [c_void_p, POINTER(c_double), POINTER(c_int64), c_int32]),
    "dmuon_last_error": (c_char_p, []),
    "dmuon_status_string": (c_char_p, [c_int]),
    "dmuon_debug_buffer": (c_int, [c_void_p, c_int64, c_int64, c_int32, POINTER(c_uint64), POINTER(c_int64),
                                   POINTER(c_int64), POINTER(c_int32)]),
    "dmuon_assign_owners": (c_int, [POINTER(c_double), c_int64, c_int32, c_int32, POINTER(c_int32),
                                    POINTER(c_double)]),
    "dmuon_plan_matrix_flops": (c_int, [c_void_p, c_int32, POINTER(c_double)]),
    "dmuon_adamw_step": (c_int, [POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                 POINTER(c_int64), POINTER(c_int32), c_int64, c_float, c_float, c_float, c_float,
                                 c_float, c_int64, c_void_p]),
    "dmuon_adamw_status": (c_int, []),
    "dmuon_step_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int32, c_float, c_float,
                                   c_float, c_int32, c_void_p]),
}

_lib = None


def load(build_if_missing: bool = False):
    """The loaded library; raises if it is not built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        from . import build as _build
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                           "(python -m matrix_orthogonalising_optimizer_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class DmuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.dmuon_last_error().decode(errors="replace")
        super().__init__(f"{where}: {lib.dmuon_status_string(status).decode()} ({status}): {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise DmuonError(status, where)
