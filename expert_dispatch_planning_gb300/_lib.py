"""ctypes view of ``libmoe_dispatch.so`` (declarations mirror include/moe_dispatch.h)."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_dispatch.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_INDEX = 6
MOE_ERR_WORKSPACE = 7
MOE_ERR_DEVICE_CAPACITY = 8

MOE_SCORING_SOFTMAX = 0
MOE_SCORING_SIGMOID = 1

_P = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_size = ctypes.c_size_t


class MoePlanOut(ctypes.Structure):
    _fields_ = [(name, _P) for name in (
        "tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "pairs_per_rank", "tokens_per_rank",
        "rank_prefix", "rank_slot_offsets", "is_token_in_rank", "dst", "src_of_slot", "dup_groups",
        "dup_loffs", "dup_counts", "status")]


class MoeBalancedPlanOut(ctypes.Structure):
    _fields_ = [(name, _P) for name in (
        "z", "alloc", "alloc_cumsum", "experts_to_copy", "remote_stats", "rank_cu_seqlens", "rank_zero_fill",
        "expert_offsets", "dst")]


# (name, restype, argtypes) for every function include/moe_dispatch.h declares
SIGNATURES = [
    ("moe_status_string", ctypes.c_char_p, [_i32]),
    ("moe_route_topk", _i32, [_P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _P, _P, _P]),
    ("moe_plan_capacity_rows", _i64, [_i32, _i32, _i32, _i32]),
    ("moe_plan_workspace_size", _size, [_i32, _i32, _i32, _i32]),
    ("moe_plan_launch_count", _i32, [_i32, _i32, _i32, _i32]),
    ("moe_plan_workspace_init", _i32, [_P, _size, _P]),
    ("moe_plan", _i32, [_P, _i32, _i32, _i32, _i32, _i32, _P, _size, ctypes.POINTER(MoePlanOut), _P]),
    ("moe_plan_no_alloc", _i32, [_P, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(MoePlanOut), _P]),
    ("moe_plan_copy", _i32, [ctypes.POINTER(MoePlanOut), ctypes.POINTER(MoePlanOut), _i32, _i32, _i32, _i32, _i32,
                             _P]),
    ("moe_plan_balanced", _i32, [ctypes.POINTER(MoePlanOut), _P, _i32, _i32, _i32, _i32, _i32, ctypes.c_int32,
                                 _i32, ctypes.c_int32, ctypes.POINTER(MoeBalancedPlanOut), _P]),
    ("moe_tile_map", _i32, [ctypes.POINTER(MoePlanOut), _i32, _i32, _P, _P, _i64, _P, _P]),
    ("moe_rank_layout_workspace_size", _size, [_i32, _i32]),
    ("moe_rank_layout", _i32, [ctypes.POINTER(MoePlanOut), _i32, _i32, _i32, _P, _size, _P, _P, _P]),
    ("moe_route_plan", _i32, [_P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _P, _P, _i32, _i32,
                              _P, ctypes.c_size_t, ctypes.POINTER(MoePlanOut), _P]),
    ("moe_route_plan_fused", _i32, [_i32, _i32, _i32, _i32, _i32]),
    ("moe_permute", _i32, [_P, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(MoePlanOut), _P, _i32, _P]),
    ("moe_combine", _i32, [_P, _P, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(MoePlanOut), _P, _P]),
    ("moe_get_status", _i32, [ctypes.POINTER(MoePlanOut), ctypes.POINTER(ctypes.c_int32), _P]),
    ("moe_debug_set_plan_fault", _i32, [_i32, _i64]),
    ("moe_debug_route_sigmoid_error", _i32, [_P, _P]),
]

_lock = threading.Lock()
_lib = None


MOE_PERMUTE_EARLY_X = 1  # moe_permute flag (include/moe_dispatch.h)


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s (%d)" % (fn, status_string(code), code))
        self.code = code


def load() -> ctypes.CDLL:
    """Load the in-tree library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    "libmoe_dispatch.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` first" % LIB_PATH)
            lib = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    try:
        return load().moe_status_string(int(code)).decode()
    except ImportError:
        return "status %d" % code


def check(fn: str, code: int) -> None:
    if code != MOE_OK:
        raise MoeError(fn, code)
