"""GB300 (sm_103a) Mixture-of-Experts routing and dispatch planning.

Four steps, each one C-ABI call into ``libmoe_dispatch.so``:
``route_topk`` -> ``plan`` -> ``permute`` -> (experts) -> ``combine``
(``route_plan`` does the first two in one call, one launch where it can).
"""
from ._lib import MoeError, load  # noqa: F401
from .api import (BalancedPlan, Plan, combine, get_status, permute, plan, plan_balanced,  # noqa: F401
                  plan_launches, rank_layout, rank_layout_workspace, route_plan, route_plan_launches, route_topk, set_plan_fault, tile_map)

__all__ = ["BalancedPlan", "MoeError", "Plan", "plan_balanced", "combine", "get_status", "load", "permute", "plan", "plan_launches",
           "rank_layout", "rank_layout_workspace", "route_plan", "route_plan_launches", "route_topk", "set_plan_fault", "tile_map"]
