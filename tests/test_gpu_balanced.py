"""GPU parity of the capacity-balanced plan (moe_plan_balanced) against the
oracle: every output bit-exact, on the five workloads' routings with tight
capacities and on random shapes; plus the row-budget error."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from balanced_checks import check_balanced_invariants

pytestmark = pytest.mark.gpu

FIELDS = ["z", "alloc", "alloc_cumsum", "experts_to_copy", "remote_stats", "rank_cu_seqlens",
          "rank_zero_fill", "expert_offsets", "dst"]


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def run_both(m, topk, E, R, tp, cap, B, NvS, check_invariants=True):
    t = torch.from_numpy(topk).cuda()
    p = m.plan(t, E, R, 1)
    b = m.plan_balanced(t, p, tp, cap, B, NvS)
    got = b.to_host()
    assert m.get_status(p) == 0
    want = oracle.plan_balanced(topk, E, R, tp, cap, B, NvS)
    for k in FIELDS:
        assert np.array_equal(got[k].reshape(want[k].shape), want[k]), k
    if check_invariants:
        check_balanced_invariants(want, topk, E, R, tp, cap, B, NvS)


@pytest.mark.parametrize("name,B,slack", [("tiny", 1, 0.9), ("mixtral", 1, 0.8), ("qwen3", 4, 1.0),
                                          ("dsv3", 2, 0.9), ("large", 4, 1.0)])
def test_balanced_on_workloads(m, name, B, slack):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    topk, _ = oracle.route_topk(inp["logits"], w.K, scoring=w.scoring, renormalize=w.renormalize,
                                bias=inp["bias"], n_group=w.n_group, topk_group=w.topk_group,
                                routed_scaling=w.routed_scaling)
    cap = int(w.N * w.K / w.R * slack)
    NvS = w.N * w.K + (w.E + B) * (w.alignment - 1)
    run_both(m, topk, w.E, w.R, w.alignment, cap, B, NvS, check_invariants=name != "large")


@pytest.mark.parametrize("seed", range(10))
def test_balanced_random_shapes(m, seed):
    rng = np.random.default_rng(500 + seed)
    R = int(rng.choice([1, 2, 4, 8, 32, 128]))
    E = R * int(rng.choice([1, 2, 4, 8]))
    E = min(E, 1024)
    K = int(rng.integers(1, min(E, 8) + 1))
    N = int(rng.integers(1, 3000))
    tp = int(rng.choice([1, 4, 32, 128]))
    B = int(rng.integers(0, 9))
    total = N * K
    cap = int(max(0, total // R + rng.integers(-total // (2 * R) - 1, total // (2 * R) + 2)))
    NvS = total + (E + B) * tp
    topk = workloads.random_topk(rng, N, E, K, hot=float(rng.choice([0.0, 0.7])))
    run_both(m, topk, E, R, tp, cap, B, NvS, check_invariants=N * K < 4000)


def test_balanced_row_budget_error(m):
    topk = np.zeros((300, 1), np.int32)
    t = torch.from_numpy(topk).cuda()
    p = m.plan(t, 4, 2, 1)
    m.plan_balanced(t, p, 1, 1000, 1, 64)
    assert m.get_status(p) == 8
