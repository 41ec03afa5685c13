"""GB300 (sm_103a) Mixture-of-Experts routing and dispatch planning.

Four steps, each one C-ABI call into ``libmoe_dispatch.so``:
``route_topk`` -> ``plan`` -> ``permute`` -> (experts) -> ``combine``.
"""
from ._lib import MoeError, load  # noqa: F401
from .api import (Plan, combine, get_status, permute, plan, plan_launches, route_topk,  # noqa: F401
                  set_plan_fault)

__all__ = ["MoeError", "Plan", "combine", "get_status", "load", "permute", "plan", "plan_launches",
           "route_topk", "set_plan_fault"]
