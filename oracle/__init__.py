"""CPU oracle for the MoE route / plan / permute / combine hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  It shares no code
with ``expert_dispatch_planning_gb300`` and imports nothing from it; the
product library never loads it.

The arithmetic lives in ``moe_oracle.c`` (plain C, built with
``-O2 -ffp-contract=off``, no fast-math).  This module only marshals numpy
arrays through ctypes.  Every function is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force on tiny inputs and
hand-derived worked examples; the dedup-structure layout is a reading the
pages do not fix (its parity against MoonEP's builder is unpinned, its
invariants are pinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EUNSUP, ECAP = 0, 1, 2, 3

SCORING_SOFTMAX = 0
SCORING_SIGMOID = 1


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``libmoe_oracle.so`` next to it."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f32.restype = f32
            lib.orc_f32_to_bf16.argtypes = [f32]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_exp_f32.argtypes = [f32]
            lib.orc_exp_f32.restype = f32
            lib.orc_sigmoid_f32.argtypes = [f32]
            lib.orc_sigmoid_f32.restype = f32
            lib.orc_route_topk.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, f32, P, P]
            lib.orc_route_topk.restype = i32
            lib.orc_plan_capacity_rows.argtypes = [i32, i32, i32, i32]
            lib.orc_plan_capacity_rows.restype = i64
            lib.orc_plan.argtypes = [P, i32, i32, i32, i32, i32] + [P] * 10 + [i64, P, i64, P, i64, P]
            lib.orc_plan.restype = i32
            lib.orc_permute.argtypes = [P, i32, i32, i32, P, P, i32, P]
            lib.orc_permute.restype = None
            lib.orc_combine.argtypes = [P, P, P, i32, i32, i32, P]
            lib.orc_combine.restype = None
            lib.orc_combine_rows.argtypes = [P, P, P, P, i32, i32, i32, P]
            lib.orc_combine_rows.restype = None
            lib.orc_plan_balanced.argtypes = [P, i32, i32, i32, i32, i32, ctypes.c_int32, i32, ctypes.c_int32] + [P] * 9
            lib.orc_plan_balanced.restype = i32
            lib.orc_tile_map.argtypes = [P, i32, i32, P, P, i64, P]
            lib.orc_tile_map.restype = i32
            lib.orc_rank_layout.argtypes = [P, i32, i32, i32, P, P]
            lib.orc_rank_layout.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__("oracle returned status %d" % code)
        self.code = code


# ---------------------------------------------------------------- scalars
def exp_f32(t: float) -> np.float32:
    return np.float32(_load().orc_exp_f32(float(t)))


def sigmoid_f32(x: float) -> np.float32:
    return np.float32(_load().orc_sigmoid_f32(float(x)))


def sigmoid_f32_array(x) -> np.ndarray:
    f = _load().orc_sigmoid_f32
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in x], dtype=np.float32)


def exp_f32_array(t) -> np.ndarray:
    f = _load().orc_exp_f32
    t = np.asarray(t, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in t], dtype=np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    f = _load().orc_f32_to_bf16
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    f = _load().orc_bf16_to_f32
    b = np.asarray(b, dtype=np.uint16).ravel()
    return np.array([f(int(v)) for v in b], dtype=np.float32)


# ---------------------------------------------------------------- router
def route_topk(logits, K, scoring=SCORING_SOFTMAX, renormalize=True, bias=None,
               n_group=1, topk_group=1, routed_scaling=1.0):
    """Return (topk_idx int32[N,K], topk_w float64[N,K])."""
    logits = _c(logits, np.float32)
    N, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((N, K), dtype=np.int32)
    w = np.empty((N, K), dtype=np.float64)
    rc = _load().orc_route_topk(_ptr(logits), _ptr(b), N, E, K, int(scoring),
                                int(bool(renormalize)), int(n_group), int(topk_group),
                                float(routed_scaling), _ptr(idx), _ptr(w))
    if rc != OK:
        raise OracleError(rc)
    return idx, w


# ---------------------------------------------------------------- plan
def capacity_rows(N, E, K, alignment) -> int:
    return int(_load().orc_plan_capacity_rows(N, E, K, alignment))


def plan(topk_idx, E, R, alignment):
    """Return a dict of every plan output (numpy arrays, exact lengths)."""
    topk = _c(topk_idx, np.int32)
    N, K = topk.shape
    cap = capacity_rows(N, E, K, alignment)
    out = dict(
        tokens_per_expert=np.empty(E, np.int32),
        cu_seqlens=np.empty(E + 1, np.int32),
        zero_fill_ranges=np.empty((E, 2), np.int32),
        pairs_per_rank=np.empty(R, np.int32),
        tokens_per_rank=np.empty(R, np.int32),
        rank_prefix=np.empty(R + 1, np.int32),
        rank_slot_offsets=np.empty(R + 1, np.int32),
        is_token_in_rank=np.empty((N, R), np.uint8),
        dst=np.empty((N, K), np.int32),
        src_of_slot=np.empty(max(cap, 1), np.int32),
    )
    gcap = N * (K // 2)
    dcap = N * (K - 1)
    dup_groups = np.empty((max(gcap, 1), 3), np.int32)
    dup_loffs = np.empty(max(dcap, 1), np.int32)
    dup_counts = np.empty(2, np.int32)
    rc = _load().orc_plan(
        _ptr(topk), N, E, K, R, alignment,
        _ptr(out["tokens_per_expert"]), _ptr(out["cu_seqlens"]), _ptr(out["zero_fill_ranges"]),
        _ptr(out["pairs_per_rank"]), _ptr(out["tokens_per_rank"]), _ptr(out["rank_prefix"]),
        _ptr(out["rank_slot_offsets"]), _ptr(out["is_token_in_rank"]), _ptr(out["dst"]),
        _ptr(out["src_of_slot"]), cap, _ptr(dup_groups), gcap, _ptr(dup_loffs), dcap,
        _ptr(dup_counts))
    if rc != OK:
        raise OracleError(rc)
    out["src_of_slot"] = out["src_of_slot"][:cap]
    out["dup_counts"] = dup_counts
    out["dup_groups"] = dup_groups[: dup_counts[0]].copy()
    out["dup_loffs"] = dup_loffs[: dup_counts[1]].copy()
    out["P"] = int(out["cu_seqlens"][-1])
    out["P_cap"] = cap
    return out


# ---------------------------------------------------------------- rows
def permute(x_bits, dst, zero_fill_ranges, K, P_cap, fill=None):
    """x_bits uint16[N,H] (bf16 bit patterns) -> permuted uint16[P_cap,H].

    Rows the permute does not write keep ``fill`` (default: zero)."""
    x = _c(x_bits, np.uint16)
    N, H = x.shape
    d = _c(dst, np.int32)
    z = _c(zero_fill_ranges, np.int32)
    if fill is None:
        out = np.zeros((P_cap, H), np.uint16)
    else:
        out = np.array(fill, dtype=np.uint16, copy=True).reshape(P_cap, H)
    _load().orc_permute(_ptr(x), N, H, K, _ptr(d), _ptr(z), z.shape[0], _ptr(out))
    return out


def combine(y_bits, w, dst):
    """y_bits uint16[P_cap,H], w float32[N,K], dst int32[N,K] -> uint16[N,H]."""
    y = _c(y_bits, np.uint16)
    wf = _c(w, np.float32)
    d = _c(dst, np.int32)
    N, K = d.shape
    H = y.shape[1]
    out = np.empty((N, H), np.uint16)
    _load().orc_combine(_ptr(y), _ptr(wf), _ptr(d), N, K, H, _ptr(out))
    return out


def combine_rows(y_bits, w, dst, tokens):
    """The combine for the listed tokens only -> uint16[len(tokens),H]."""
    y = _c(y_bits, np.uint16)
    wf = _c(w, np.float32)
    d = _c(dst, np.int32)
    t = _c(tokens, np.int64)
    K = d.shape[1]
    H = y.shape[1]
    out = np.empty((t.shape[0], H), np.uint16)
    _load().orc_combine_rows(_ptr(y), _ptr(wf), _ptr(d), _ptr(t), t.shape[0], K, H, _ptr(out))
    return out


# ---------------------------------------------------------------- balanced plan
def plan_balanced(topk_idx, E, R, token_padding, capacity, B, NvS):
    """Capacity-balanced plan with redundant experts (single source rank).

    Returns dict(z[R,R], alloc[R,E], alloc_cumsum[E,R], experts_to_copy[R,B],
    remote_stats[R,2], rank_cu_seqlens[R,E+B], rank_zero_fill[R,E+B,2],
    expert_offsets[R,E], dst[N,K])."""
    topk = _c(topk_idx, np.int32)
    N, K = topk.shape
    out = dict(z=np.empty((R, R), np.int32), alloc=np.empty((R, E), np.int32),
               alloc_cumsum=np.empty((E, R), np.int32), experts_to_copy=np.empty((R, max(B, 0)), np.int32),
               remote_stats=np.empty((R, 2), np.int32), rank_cu_seqlens=np.empty((R, E + B), np.int32),
               rank_zero_fill=np.empty((R, E + B, 2), np.int32), expert_offsets=np.empty((R, E), np.int32),
               dst=np.empty((N, K), np.int32))
    rc = _load().orc_plan_balanced(
        _ptr(topk), N, E, K, R, token_padding, int(capacity), B, int(NvS),
        *[_ptr(out[k]) for k in ("z", "alloc", "alloc_cumsum", "experts_to_copy", "remote_stats",
                                 "rank_cu_seqlens", "rank_zero_fill", "expert_offsets", "dst")])
    if rc != OK:
        raise OracleError(rc)
    return out


# ---------------------------------------------------------------- tile map / rank layout
def tile_map(tokens_per_expert, tile, max_tiles):
    """Grouped-GEMM tiles: (tile_expert[max_tiles], tile_row_limit[max_tiles], (num_tiles, size))."""
    c = _c(tokens_per_expert, np.int32)
    te = np.empty(max_tiles, np.int32)
    tl = np.empty(max_tiles, np.int32)
    sizes = np.empty(2, np.int32)
    rc = _load().orc_tile_map(_ptr(c), c.size, int(tile), _ptr(te), _ptr(tl), int(max_tiles), _ptr(sizes))
    if rc != OK:
        raise OracleError(rc)
    return te, tl, sizes


def rank_layout(is_token_in_rank, num_channels):
    """(channel_prefix_matrix[R, C], token_rank_slot[N, R]) from is_token_in_rank[N, R]."""
    itr = _c(is_token_in_rank, np.uint8)
    N, R = itr.shape
    cpm = np.empty((R, num_channels), np.int32)
    trs = np.empty((N, R), np.int32)
    rc = _load().orc_rank_layout(_ptr(itr), N, R, int(num_channels), _ptr(cpm), _ptr(trs))
    if rc != OK:
        raise OracleError(rc)
    return cpm, trs
