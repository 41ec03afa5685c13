"""Python binding of the C ABI: argument marshalling only.

Torch supplies device memory and the current CUDA stream; every step of the
routing / planning / row-movement path runs in the library's own kernels.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import torch

from . import _lib
from ._lib import MOE_PERMUTE_EARLY_X, MoeBalancedPlanOut, MoePlanOut, check, load

SCORING = {"softmax": _lib.MOE_SCORING_SOFTMAX, "sigmoid": _lib.MOE_SCORING_SIGMOID,
           0: 0, 1: 1}


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s (got %s %s)" % (
            name, dtype, tuple(shape), t.dtype, tuple(t.shape)))


# ---------------------------------------------------------------- router
def route_topk(logits: torch.Tensor, K: int, scoring="softmax", renormalize: bool = True,
               bias: torch.Tensor | None = None, n_group: int = 1, topk_group: int = 1,
               routed_scaling: float = 1.0, topk_idx: torch.Tensor | None = None,
               topk_w: torch.Tensor | None = None, stream=None):
    """Router top-K: returns (topk_idx int32[N,K], topk_w float32[N,K])."""
    N, E = logits.shape
    _need(logits, torch.float32, (N, E), "logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((N, K), dtype=torch.float32, device=logits.device)
    _need(topk_idx, torch.int32, (N, K), "topk_idx")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    rc = load().moe_route_topk(_ptr(logits), _ptr(bias), N, E, K, SCORING[scoring], int(bool(renormalize)),
                               n_group, topk_group, float(routed_scaling), _ptr(topk_idx), _ptr(topk_w),
                               _stream(stream))
    check("moe_route_topk", rc)
    return topk_idx, topk_w


# ---------------------------------------------------------------- plan
@dataclass
class Plan:
    """Caller-owned plan buffers (device tensors) plus the plan workspace."""
    N: int
    E: int
    K: int
    R: int
    alignment: int
    tokens_per_expert: torch.Tensor
    cu_seqlens: torch.Tensor
    zero_fill_ranges: torch.Tensor
    pairs_per_rank: torch.Tensor
    tokens_per_rank: torch.Tensor
    rank_prefix: torch.Tensor
    rank_slot_offsets: torch.Tensor
    is_token_in_rank: torch.Tensor
    dst: torch.Tensor
    src_of_slot: torch.Tensor
    dup_groups: torch.Tensor
    dup_loffs: torch.Tensor
    dup_counts: torch.Tensor
    status: torch.Tensor
    workspace: torch.Tensor
    c_struct: MoePlanOut = field(default=None, repr=False)

    @property
    def P_cap(self) -> int:
        return self.src_of_slot.numel()

    @classmethod
    def allocate(cls, N, E, K, R, alignment, device="cuda", stream=None) -> "Plan":
        lib = load()
        cap = int(lib.moe_plan_capacity_rows(N, E, K, alignment))
        ws = int(lib.moe_plan_workspace_size(N, E, K, R))
        if cap < 0 or ws == 0:
            raise ValueError("unsupported plan sizes N=%d E=%d K=%d R=%d alignment=%d" % (N, E, K, R, alignment))
        i32 = dict(dtype=torch.int32, device=device)
        p = cls(N=N, E=E, K=K, R=R, alignment=alignment,
                tokens_per_expert=torch.empty(E, **i32), cu_seqlens=torch.empty(E + 1, **i32),
                zero_fill_ranges=torch.empty((E, 2), **i32), pairs_per_rank=torch.empty(R, **i32),
                tokens_per_rank=torch.empty(R, **i32), rank_prefix=torch.empty(R + 1, **i32),
                rank_slot_offsets=torch.empty(R + 1, **i32),
                is_token_in_rank=torch.empty((N, R), dtype=torch.uint8, device=device),
                dst=torch.empty((N, K), **i32), src_of_slot=torch.empty(cap, **i32),
                dup_groups=torch.empty((max(1, N * (K // 2)), 3), **i32),
                dup_loffs=torch.empty(max(1, N * (K - 1)), **i32), dup_counts=torch.empty(2, **i32),
                status=torch.zeros(4, **i32), workspace=torch.empty(ws, dtype=torch.uint8, device=device))
        check("moe_plan_workspace_init", lib.moe_plan_workspace_init(_ptr(p.workspace), ws, _stream(stream)))
        p.c_struct = MoePlanOut(*[t.data_ptr() for t in (
            p.tokens_per_expert, p.cu_seqlens, p.zero_fill_ranges, p.pairs_per_rank, p.tokens_per_rank,
            p.rank_prefix, p.rank_slot_offsets, p.is_token_in_rank, p.dst, p.src_of_slot, p.dup_groups,
            p.dup_loffs, p.dup_counts, p.status)])
        return p

    def clone(self, stream=None) -> "Plan":
        """A copy of this plan in new buffers (moe_plan_copy)."""
        c = Plan.allocate(self.N, self.E, self.K, self.R, self.alignment, device=self.dst.device, stream=stream)
        check("moe_plan_copy", load().moe_plan_copy(ctypes.byref(self.c_struct), ctypes.byref(c.c_struct), self.N,
                                                   self.E, self.K, self.R, self.alignment, _stream(stream)))
        return c

    def to_host(self) -> dict:
        """Copy every output to numpy (synchronises); dedup arrays cut to their counts."""
        out = {k: getattr(self, k).cpu().numpy() for k in (
            "tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "pairs_per_rank", "tokens_per_rank",
            "rank_prefix", "rank_slot_offsets", "is_token_in_rank", "dst", "src_of_slot", "dup_counts")}
        g, d = int(out["dup_counts"][0]), int(out["dup_counts"][1])
        out["dup_groups"] = self.dup_groups[:g].cpu().numpy()
        out["dup_loffs"] = self.dup_loffs[:d].cpu().numpy()
        out["P"] = int(out["cu_seqlens"][-1])
        out["P_cap"] = self.P_cap
        return out


def plan(topk_idx: torch.Tensor, E: int, R: int, alignment: int, out: Plan | None = None,
         stream=None) -> Plan:
    """Dispatch plan for topk_idx int32[N,K] (written into `out` if given)."""
    N, K = topk_idx.shape
    _need(topk_idx, torch.int32, (N, K), "topk_idx")
    if out is None:
        out = Plan.allocate(N, E, K, R, alignment, device=topk_idx.device, stream=stream)
    if (out.N, out.E, out.K, out.R, out.alignment) != (N, E, K, R, alignment):
        raise ValueError("plan buffers were allocated for other sizes")
    rc = load().moe_plan(_ptr(topk_idx), N, E, K, R, alignment, _ptr(out.workspace), out.workspace.numel(),
                         ctypes.byref(out.c_struct), _stream(stream))
    check("moe_plan", rc)
    return out


def route_plan(logits: torch.Tensor, K: int, R: int, alignment: int, scoring="softmax", renormalize: bool = True,
               bias: torch.Tensor | None = None, n_group: int = 1, topk_group: int = 1,
               routed_scaling: float = 1.0, topk_idx: torch.Tensor | None = None,
               topk_w: torch.Tensor | None = None, out: Plan | None = None, stream=None):
    """route_topk then plan in one call (one launch where route_plan_fused says so):
    returns (topk_idx, topk_w, plan), identical to the two calls."""
    N, E = logits.shape
    _need(logits, torch.float32, (N, E), "logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((N, K), dtype=torch.float32, device=logits.device)
    _need(topk_idx, torch.int32, (N, K), "topk_idx")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    if out is None:
        out = Plan.allocate(N, E, K, R, alignment, device=logits.device, stream=stream)
    if (out.N, out.E, out.K, out.R, out.alignment) != (N, E, K, R, alignment):
        raise ValueError("plan buffers were allocated for other sizes")
    rc = load().moe_route_plan(_ptr(logits), _ptr(bias), N, E, K, SCORING[scoring], int(bool(renormalize)),
                               n_group, topk_group, float(routed_scaling), _ptr(topk_idx), _ptr(topk_w), R, alignment,
                               _ptr(out.workspace), out.workspace.numel(), ctypes.byref(out.c_struct), _stream(stream))
    check("moe_route_plan", rc)
    return topk_idx, topk_w, out


def route_plan_launches(N: int, E: int, K: int, R: int, n_group: int = 1) -> int:
    """Kernel launches route_plan makes for these sizes on the current device."""
    f = int(load().moe_route_plan_fused(N, E, K, R, n_group))
    if f < 0:
        raise ValueError("unsupported sizes")
    if N == 0:      # nothing to route: the plan's launch alone
        return plan_launches(N, E, K, R)
    return 1 if f == 1 else 1 + plan_launches(N, E, K, R)


def plan_launches(N: int, E: int, K: int, R: int) -> int:
    """Kernel launches moe_plan makes for these sizes on the current device."""
    n = int(load().moe_plan_launch_count(N, E, K, R))
    if n < 0:
        raise ValueError("unsupported plan sizes")
    return n


@dataclass
class BalancedPlan:
    """Caller-owned outputs of the capacity-balanced plan (device tensors)."""
    N: int
    E: int
    K: int
    R: int
    B: int
    z: torch.Tensor
    alloc: torch.Tensor
    alloc_cumsum: torch.Tensor
    experts_to_copy: torch.Tensor
    remote_stats: torch.Tensor
    rank_cu_seqlens: torch.Tensor
    rank_zero_fill: torch.Tensor
    expert_offsets: torch.Tensor
    dst: torch.Tensor
    c_struct: MoeBalancedPlanOut = field(default=None, repr=False)

    FIELDS = ("z", "alloc", "alloc_cumsum", "experts_to_copy", "remote_stats", "rank_cu_seqlens",
              "rank_zero_fill", "expert_offsets", "dst")

    @classmethod
    def allocate(cls, N, E, K, R, B, device="cuda") -> "BalancedPlan":
        i32 = dict(dtype=torch.int32, device=device)
        b = cls(N=N, E=E, K=K, R=R, B=B, z=torch.empty((R, R), **i32), alloc=torch.empty((R, E), **i32),
                alloc_cumsum=torch.empty((E, R), **i32), experts_to_copy=torch.empty((R, max(B, 1)), **i32),
                remote_stats=torch.empty((R, 2), **i32), rank_cu_seqlens=torch.empty((R, E + B), **i32),
                rank_zero_fill=torch.empty((R, E + B, 2), **i32), expert_offsets=torch.empty((R, E), **i32),
                dst=torch.empty((N, K), **i32))
        b.c_struct = MoeBalancedPlanOut(*[getattr(b, k).data_ptr() for k in cls.FIELDS])
        return b

    def to_host(self) -> dict:
        out = {k: getattr(self, k).cpu().numpy() for k in self.FIELDS}
        out["experts_to_copy"] = out["experts_to_copy"][:, : self.B]
        return out


def plan_balanced(topk_idx: torch.Tensor, p: Plan, token_padding: int, capacity: int, B: int, NvS: int,
                  out: BalancedPlan | None = None, stream=None) -> BalancedPlan:
    """Capacity-balanced plan with redundant experts on top of the plain plan `p`."""
    N, K = topk_idx.shape
    _need(topk_idx, torch.int32, (p.N, p.K), "topk_idx")
    if out is None:
        out = BalancedPlan.allocate(N, p.E, K, p.R, B, device=topk_idx.device)
    rc = load().moe_plan_balanced(ctypes.byref(p.c_struct), _ptr(topk_idx), N, p.E, K, p.R, int(token_padding),
                                  int(capacity), int(B), int(NvS), ctypes.byref(out.c_struct), _stream(stream))
    check("moe_plan_balanced", rc)
    return out


def tile_map(p: Plan, max_tiles: int | None = None, out=None, stream=None):
    """Grouped-GEMM tiles of `p.alignment` rows: (tile_expert, tile_row_limit, sizes[num_tiles, P])."""
    dev = p.dst.device
    if out is None:
        if max_tiles is None:
            max_tiles = max(1, p.P_cap // p.alignment)
        out = (torch.empty(max_tiles, dtype=torch.int32, device=dev),
               torch.empty(max_tiles, dtype=torch.int32, device=dev), torch.empty(2, dtype=torch.int32, device=dev))
    te, tl, sizes = out
    max_tiles = te.numel()
    _need(tl, torch.int32, (max_tiles,), "tile_row_limit")
    _need(sizes, torch.int32, (2,), "sizes")
    check("moe_tile_map", load().moe_tile_map(ctypes.byref(p.c_struct), p.E, p.alignment, _ptr(te), _ptr(tl),
                                             int(max_tiles), _ptr(sizes), _stream(stream)))
    return te, tl, sizes


def rank_layout_workspace(N: int, R: int, device="cuda") -> torch.Tensor:
    """A workspace for rank_layout of these sizes (reusable across calls)."""
    n = int(load().moe_rank_layout_workspace_size(N, R))
    if n == 0:
        raise ValueError("unsupported rank layout sizes N=%d R=%d" % (N, R))
    return torch.empty(n, dtype=torch.uint8, device=device)


def rank_layout(p: Plan, num_channels: int, workspace: torch.Tensor | None = None, out=None, stream=None):
    """(channel_prefix_matrix[R, C], token_rank_slot[N, R]) of a plan."""
    dev = p.dst.device
    if workspace is None:
        workspace = rank_layout_workspace(p.N, p.R, device=dev)
    if out is None:
        out = (torch.empty((p.R, num_channels), dtype=torch.int32, device=dev),
               torch.empty((p.N, p.R), dtype=torch.int32, device=dev))
    cpm, trs = out
    _need(cpm, torch.int32, (p.R, num_channels), "channel_prefix_matrix")
    _need(trs, torch.int32, (p.N, p.R), "token_rank_slot")
    check("moe_rank_layout", load().moe_rank_layout(ctypes.byref(p.c_struct), p.N, p.R, int(num_channels),
                                                   _ptr(workspace), workspace.numel(), _ptr(cpm), _ptr(trs),
                                                   _stream(stream)))
    return cpm, trs


def permute(x: torch.Tensor, p: Plan, out: torch.Tensor | None = None, stream=None,
            early_x: bool = False) -> torch.Tensor:
    """Expert-contiguous copy of x bf16[N,H] -> bf16[P_cap,H] (rows >= P untouched).

    early_x: start loading x before the previous kernel on the stream ends
    (MOE_PERMUTE_EARLY_X); only when that kernel does not write x, e.g.
    directly after the plan() call that built p, with x produced before it.
    """
    N, H = x.shape
    _need(x, torch.bfloat16, (p.N, H), "x")
    if out is None:
        out = torch.empty((p.P_cap, H), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (p.P_cap, H), "permuted")
    rc = load().moe_permute(_ptr(x), N, H, p.K, p.E, p.alignment, ctypes.byref(p.c_struct), _ptr(out),
                            MOE_PERMUTE_EARLY_X if early_x else 0, _stream(stream))
    check("moe_permute", rc)
    return out


def combine(y: torch.Tensor, topk_w: torch.Tensor, p: Plan, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Weighted combine of expert rows y bf16[P_cap,H] back to token order bf16[N,H]."""
    H = y.shape[1]
    _need(y, torch.bfloat16, (p.P_cap, H), "y")
    _need(topk_w, torch.float32, (p.N, p.K), "topk_w")
    if out is None:
        out = torch.empty((p.N, H), dtype=torch.bfloat16, device=y.device)
    _need(out, torch.bfloat16, (p.N, H), "out")
    rc = load().moe_combine(_ptr(y), _ptr(topk_w), p.N, p.K, H, p.E, p.alignment, ctypes.byref(p.c_struct),
                            _ptr(out), _stream(stream))
    check("moe_combine", rc)
    return out


def get_status(p: Plan, stream=None) -> int:
    """Synchronise and return (then clear) the plan's device status code."""
    v = ctypes.c_int32(0)
    check("moe_get_status", load().moe_get_status(ctypes.byref(p.c_struct), ctypes.byref(v), _stream(stream)))
    return int(v.value)


def set_plan_fault(skip_tile: int = -1, timeout_ns: int = 0) -> None:
    """Test hook: make one planning tile withhold its counts (see the C header)."""
    check("moe_debug_set_plan_fault", load().moe_debug_set_plan_fault(int(skip_tile), int(timeout_ns)))
