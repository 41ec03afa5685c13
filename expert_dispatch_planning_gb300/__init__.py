"""GB300 (sm_103a) Mixture-of-Experts routing and dispatch planning.

Four steps, each one C-ABI call into ``libmoe_dispatch.so``:
``route_topk`` -> ``plan`` -> ``permute`` -> (experts) -> ``combine``.
"""
from ._lib import MoeError, load  # noqa: F401
from .api import Plan, combine, get_status, permute, plan, route_topk, set_plan_fault  # noqa: F401

__all__ = ["MoeError", "Plan", "combine", "get_status", "load", "permute", "plan", "route_topk",
           "set_plan_fault"]
