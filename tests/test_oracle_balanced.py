"""Pins for the oracle's capacity-balanced plan: the hand-derived worked
example, closed-form special cases, and invariants on random inputs."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from balanced_checks import check_balanced_invariants


def test_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "plan_balanced_worked_example.json")) as f:
        case = json.load(f)
    o = oracle.plan_balanced(np.array(case["topk_idx"], np.int32), case["E"], case["R"],
                             case["token_padding"], case["capacity"], case["B"], case["NvS"])
    for k, v in case["expected"].items():
        assert o[k].tolist() == v, k
    check_balanced_invariants(o, case["topk_idx"], case["E"], case["R"], case["token_padding"],
                              case["capacity"], case["B"], case["NvS"])


def test_no_balancing_when_capacity_suffices():
    rng = np.random.default_rng(40)
    topk = workloads.random_topk(rng, 300, 16, 4)
    E, R = 16, 4
    o = oracle.plan_balanced(topk, E, R, 8, 10 ** 6, 2, 4096)
    assert np.all(o["z"] == 0)
    count = np.bincount(topk.ravel(), minlength=E)
    want = np.zeros((R, E), np.int64)
    for e in range(E):
        want[e // (E // R), e] = count[e]
    assert np.array_equal(o["alloc"], want)
    assert np.all(o["experts_to_copy"] == -1) and np.all(o["remote_stats"] == 0)
    # each rank's groups are its own experts only, padded to 8
    for d in range(R):
        local = count[d * 4:(d + 1) * 4]
        padded = np.where(local > 0, -(-local // 8) * 8, 0)
        assert o["rank_cu_seqlens"][d, d * 4:(d + 1) * 4].tolist() == np.cumsum(padded).tolist()
    check_balanced_invariants(o, topk, E, R, 8, 10 ** 6, 2, 4096)


@pytest.mark.parametrize("seed", range(12))
def test_random_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8]))
    E = R * int(rng.integers(1, 6))
    K = int(rng.integers(1, min(E, 6) + 1))
    N = int(rng.integers(1, 400))
    tp = int(rng.choice([1, 2, 4, 16]))
    B = int(rng.integers(0, 4))
    total = N * K
    cap = int(max(1, total // R + rng.integers(-total // (2 * R) - 1, total // (2 * R) + 2)))
    NvS = total + E * tp + 64
    topk = workloads.random_topk(rng, N, E, K, hot=float(rng.choice([0.0, 0.6])))
    o = oracle.plan_balanced(topk, E, R, tp, cap, B, NvS)
    check_balanced_invariants(o, topk, E, R, tp, cap, B, NvS)


def test_capacity_too_small_is_an_error():
    topk = np.zeros((64, 1), np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.plan_balanced(topk, 4, 2, 1, 100, 1, NvS=32)


@pytest.mark.parametrize("E,K,R,tp,cap,B", [(8, 2, 4, 16, 0, 2), (64, 6, 8, 1, 5, 0), (256, 8, 64, 128, 100, 4)])
def test_empty_batch(E, K, R, tp, cap, B):
    # no tokens: nothing to move (z = 0), no rank handles a pair (alloc and
    # its prefix 0), no remote expert has pairs so no redundant expert is
    # chosen (-1), and every group is empty (offsets, ends, padding 0)
    o = oracle.plan_balanced(np.zeros((0, K), np.int32), E, R, tp, cap, B, 64)
    for k in ("z", "alloc", "alloc_cumsum", "remote_stats", "rank_cu_seqlens", "rank_zero_fill", "expert_offsets"):
        assert not o[k].any(), k
    assert o["experts_to_copy"].shape == (R, B) and (o["experts_to_copy"] == -1).all()
    assert o["rank_cu_seqlens"].shape == (R, E + B) and o["dst"].shape == (0, K)
