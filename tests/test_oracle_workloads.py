"""Pins for the oracle at the five workloads' own inputs, at full size.

The other oracle pins use brute force and closed forms on small inputs; these
check the oracle's routing and plan on the seeded inputs the benchmark and
the GPU parity tests use, by means independent of the oracle's loops:
selection against numpy's lexicographic sort of the definition (group scores
as the sum of a group's two largest keys, the topk_group best groups, top-K
by (key descending, expert ascending)), weights against float64 closed
forms, and the plan against the size-independent invariants.  The sigmoid
keys come from the oracle's fixed sigmoid, which its own pins fix against
float64 and closed forms.
"""
import numpy as np
import pytest

import oracle
import workloads
from plan_checks import check_plan_invariants

NAMES = ["tiny", "mixtral", "qwen3", "dsv3", "large"]


def route(w, inp):
    return oracle.route_topk(inp["logits"], w.K, scoring=w.scoring, renormalize=w.renormalize, bias=inp["bias"],
                             n_group=w.n_group, topk_group=w.topk_group, routed_scaling=w.routed_scaling)


def selection_by_sort(w, logits, bias):
    """Expert ids by the routing definition, through numpy's sorts."""
    N, E = logits.shape
    if w.scoring == oracle.SCORING_SOFTMAX:
        keys = logits.astype(np.float32)
    else:
        sig = oracle.sigmoid_f32_array(logits).reshape(N, E)
        keys = (sig + (0 if bias is None else bias[None, :])).astype(np.float32)
    allowed = np.ones((N, E), bool)
    if w.n_group > 1:
        gs = E // w.n_group
        g = keys.reshape(N, w.n_group, gs)
        top2 = -np.sort(-g, axis=2)[:, :, :2]
        score = (top2[:, :, 0] + top2[:, :, 1]).astype(np.float32)  # one fp32 add, as defined
        gidx = np.broadcast_to(np.arange(w.n_group), score.shape)
        order = np.lexsort((gidx, -score.astype(np.float64)), axis=1)[:, : w.topk_group]
        kept = np.zeros((N, w.n_group), bool)
        np.put_along_axis(kept, order, True, axis=1)
        allowed = np.repeat(kept, gs, axis=1)
    masked = np.where(allowed, keys.astype(np.float64), -np.inf)
    eidx = np.broadcast_to(np.arange(E), (N, E))
    return np.lexsort((eidx, -masked), axis=1)[:, : w.K].astype(np.int32)


@pytest.mark.parametrize("name", NAMES)
def test_routing_at_the_workload(name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    idx, wt = route(w, inp)
    assert np.array_equal(idx, selection_by_sort(w, inp["logits"], inp["bias"]))
    x = np.take_along_axis(inp["logits"], idx, 1).astype(np.float64)
    if w.scoring == oracle.SCORING_SOFTMAX:       # renormalised softmax over the K winners
        e = np.exp(x - x[:, :1])
        want = e / e.sum(1, keepdims=True) * w.routed_scaling
    else:                                         # unbiased sigmoid scores, renormalised, scaled
        s = 1.0 / (1.0 + np.exp(-x))
        want = s / s.sum(1, keepdims=True) * w.routed_scaling
    np.testing.assert_allclose(wt, want, rtol=1e-12)
    np.testing.assert_allclose(wt.sum(1), w.routed_scaling, rtol=1e-12)


@pytest.mark.parametrize("name", NAMES)
def test_plan_at_the_workload(name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    idx, _ = route(w, inp)
    p = oracle.plan(idx, w.E, w.R, w.alignment)
    check_plan_invariants(p, idx, w.E, w.R, w.alignment)
    assert p["P"] == int(np.asarray(p["cu_seqlens"])[-1]) <= p["P_cap"]
    if name == "large":
        # the dedup-heavy shaping: most tokens send two or more pairs to one rank
        dst = np.asarray(p["dst"]).reshape(w.N, w.K)
        assert np.mean((dst < 0).any(axis=1)) > 0.5


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3"])
def test_permute_at_the_workload(name):
    """permuted[raw slot of pair f] = x[f // K]; padding rows +0; by numpy's
    fancy indexing (the workloads whose buffers stay under a few hundred MB)."""
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0)
    idx, _ = route(w, inp)
    p = oracle.plan(idx, w.E, w.R, w.alignment)
    dst = np.asarray(p["dst"], np.int64).ravel()
    raw = np.where(dst >= 0, dst, -dst - 1)
    want = np.zeros((p["P_cap"], w.H), np.uint16)
    want[raw] = inp["x_bits"][np.arange(w.N * w.K) // w.K]
    got = oracle.permute(inp["x_bits"], p["dst"], p["zero_fill_ranges"], w.K, p["P_cap"])
    assert np.array_equal(got, want)
