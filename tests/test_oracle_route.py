"""Pins for the oracle's router (softmax / sigmoid, group-limited top-K).

Selection is checked against brute force (Python's sort over (-key, index),
and exhaustive enumeration of group subsets) on tiny inputs chosen to force
ties; weights against closed forms and invariants; plus the hand-derived
worked examples in tests/golden/route_worked_examples.json.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle


def expected_topk(keys, K, allowed=None):
    E = len(keys)
    cand = [e for e in range(E) if allowed is None or allowed[e]]
    return sorted(cand, key=lambda e: (-float(keys[e]), e))[:K]


@pytest.fixture(scope="module")
def golden(golden_dir):
    with open(os.path.join(golden_dir, "route_worked_examples.json")) as f:
        return json.load(f)


def test_golden_softmax(golden):
    for name in ("softmax_tie", "softmax_closed_form"):
        case = golden[name]
        logits = np.array(case["logits"], np.float32)
        idx, w = oracle.route_topk(logits, case["K"])
        assert idx.tolist() == case["topk_idx"]
        np.testing.assert_allclose(w, np.array(case["topk_w"]), rtol=case.get("rtol", 0), atol=0)


def _keys_as_route_inputs(keys):
    # logits 0 give sigmoid exactly 0.5, so key = 0.5 + (key - 0.5) in fp32
    keys = np.asarray(keys, np.float32)
    logits = np.zeros((1, keys.size), np.float32)
    bias = (keys - np.float32(0.5)).astype(np.float32)
    return logits, bias


def test_golden_group_limited(golden):
    for name in ("group_limited", "group_sum_not_max"):
        case = golden[name]
        logits, bias = _keys_as_route_inputs(case["keys"])
        idx, w = oracle.route_topk(logits, case["K"], scoring=oracle.SCORING_SIGMOID,
                                   bias=bias, n_group=case["n_group"],
                                   topk_group=case["topk_group"])
        assert idx.tolist() == case["topk_idx"], name
        # every selected score is sigmoid(0) = 1/2: renormalised weights 1/K
        np.testing.assert_allclose(w, 1.0 / case["K"], rtol=1e-15)


def test_softmax_selection_brute_force():
    rng = np.random.default_rng(10)
    levels = np.array([-1.0, 0.0, 0.5, 1.0, 2.5], np.float32)
    for trial in range(400):
        E = int(rng.integers(1, 9))
        K = int(rng.integers(1, E + 1))
        N = 3
        logits = levels[rng.integers(0, levels.size, size=(N, E))]
        idx, _ = oracle.route_topk(logits, K)
        for s in range(N):
            assert idx[s].tolist() == expected_topk(logits[s], K), (logits[s], K)


def test_softmax_selection_negative_zero_ties_lower_index():
    logits = np.array([[-0.0, 0.0, -1.0]], np.float32)
    idx, _ = oracle.route_topk(logits, 2)
    assert idx.tolist() == [[0, 1]]


def test_softmax_weights_closed_forms():
    rng = np.random.default_rng(11)
    # equal logits: every weight is 1/K
    logits = np.full((4, 16), 0.3, np.float32)
    idx, w = oracle.route_topk(logits, 5)
    assert idx.tolist() == [[0, 1, 2, 3, 4]] * 4
    np.testing.assert_allclose(w, 0.2, rtol=1e-15)
    # full softmax (renormalize off) of equal logits is 1/E
    _, w = oracle.route_topk(logits, 5, renormalize=False)
    np.testing.assert_allclose(w, 1.0 / 16, rtol=1e-15)
    # invariants on random rows: weights sum to the scale, ratios are exp(l_i - l_j)
    logits = rng.standard_normal((50, 64)).astype(np.float32)
    idx, w = oracle.route_topk(logits, 8, routed_scaling=2.5)
    np.testing.assert_allclose(w.sum(1), 2.5, rtol=1e-13)
    sel = np.take_along_axis(logits, idx, 1).astype(np.float64)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-12)
    # non-renormalised weights equal the full-row softmax probability
    _, w0 = oracle.route_topk(logits, 8, renormalize=False)
    denom = np.exp(logits.astype(np.float64) - logits.max(1, keepdims=True)).sum(1)
    np.testing.assert_allclose(w0, np.exp(sel - sel[:, :1]) / denom[:, None], rtol=1e-12)


def test_sigmoid_selection_brute_force():
    rng = np.random.default_rng(12)
    for trial in range(200):
        E = int(rng.integers(2, 13))
        K = int(rng.integers(1, E + 1))
        logits = rng.choice(np.array([-2.0, 0.0, 1.0, 3.0], np.float32), size=(2, E))
        bias = rng.choice(np.array([0.0, 0.25, -0.25], np.float32), size=E)
        idx, _ = oracle.route_topk(logits, K, scoring=oracle.SCORING_SIGMOID, bias=bias)
        sig = oracle.sigmoid_f32_array(logits).reshape(logits.shape)
        keys = (sig + bias[None, :]).astype(np.float32)
        for s in range(2):
            assert idx[s].tolist() == expected_topk(keys[s], K)


def test_group_limited_brute_force():
    rng = np.random.default_rng(13)
    for trial in range(300):
        n_group = int(rng.integers(2, 6))
        gs = int(rng.integers(1, 5))
        E = n_group * gs
        topk_group = int(rng.integers(1, n_group + 1))
        K = int(rng.integers(1, topk_group * gs + 1))
        keys = rng.choice(np.array([0.1, 0.2, 0.3, 0.5, 0.7, 0.9], np.float32), size=E)
        logits, bias = _keys_as_route_inputs(keys)
        k32 = (np.float32(0.5) + bias).astype(np.float32)
        idx, _ = oracle.route_topk(logits, K, scoring=oracle.SCORING_SIGMOID, bias=bias,
                                   n_group=n_group, topk_group=topk_group)
        # brute force: enumerate every set of topk_group groups; the kept set
        # is the lexicographically best list of (score desc, index asc)
        scores = []
        for g in range(n_group):
            vals = sorted((float(v) for v in k32[g * gs:(g + 1) * gs]), reverse=True)
            scores.append(np.float32(vals[0]) if gs == 1 else np.float32(vals[0]) + np.float32(vals[1]))
        best = None
        for subset in itertools.combinations(range(n_group), topk_group):
            ordered = sorted(subset, key=lambda g: (-float(scores[g]), g))
            rank_key = [(-float(scores[g]), g) for g in ordered]
            if best is None or rank_key < best[0]:
                best = (rank_key, set(subset))
        allowed = [(e // gs) in best[1] for e in range(E)]
        assert idx[0].tolist() == expected_topk(k32, K, allowed), (keys, n_group, topk_group, K)


def test_sigmoid_weights_closed_forms():
    # all logits 0 -> every score 1/2; renormalised weights scale/K
    logits = np.zeros((3, 32), np.float32)
    bias = np.linspace(-0.1, 0.1, 32).astype(np.float32)
    idx, w = oracle.route_topk(logits, 4, scoring=1, bias=bias, routed_scaling=2.5)
    assert idx.tolist() == [[31, 30, 29, 28]] * 3   # bias decides the order
    np.testing.assert_allclose(w, 2.5 / 4, rtol=1e-15)
    _, w = oracle.route_topk(logits, 4, scoring=1, bias=bias, renormalize=False, routed_scaling=2.5)
    np.testing.assert_allclose(w, 1.25, rtol=1e-15)
    # weights use the unbiased score: sigma(l_k) / sum sigma(l_j)
    rng = np.random.default_rng(14)
    logits = rng.standard_normal((20, 16)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, 16).astype(np.float32)
    idx, w = oracle.route_topk(logits, 3, scoring=1, bias=bias)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx, 1).astype(np.float64)))
    np.testing.assert_allclose(w, s / s.sum(1, keepdims=True), rtol=1e-13)


def test_route_argument_errors():
    logits = np.zeros((2, 8), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.route_topk(logits, 9)                       # K > E
    with pytest.raises(oracle.OracleError):
        oracle.route_topk(logits, 2, scoring=1, n_group=3, topk_group=1)   # E % n_group
    with pytest.raises(oracle.OracleError):
        oracle.route_topk(logits, 5, scoring=1, n_group=4, topk_group=2)   # K > kept experts
    with pytest.raises(oracle.OracleError):
        oracle.route_topk(logits, 2, scoring=0, n_group=2, topk_group=1)   # groups need sigmoid
