"""Pins for the oracle's dispatch plan.

- the hand-derived worked example (tests/golden/plan_worked_example.json);
- exhaustive enumeration of every router output for N <= 3 tokens
  (E=4, K=2, distinct experts per token) and random N <= 8 cases, each
  against the counting definition in plan_checks.definition_plan;
- invariants at a medium size, and argument errors.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from plan_checks import check_plan_invariants, definition_plan

KEYS = ["tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "dst", "src_of_slot",
        "is_token_in_rank", "tokens_per_rank", "pairs_per_rank", "rank_prefix",
        "rank_slot_offsets", "dup_groups", "dup_loffs", "dup_counts"]


def _same(p, want):
    for k in KEYS:
        got = np.asarray(p[k]).tolist()
        exp = want[k]
        if k == "dup_groups":
            got = [list(g) for g in got]
        assert got == exp, (k, got, exp)


def test_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "plan_worked_example.json")) as f:
        case = json.load(f)
    topk = np.array(case["topk_idx"], np.int32)
    p = oracle.plan(topk, case["E"], case["R"], case["alignment"])
    _same(p, case["expected"])
    assert p["P"] == 10 and p["P_cap"] == 12


def test_exhaustive_tiny():
    E, K = 4, 2
    pairs = [list(c) for c in itertools.permutations(range(E), K)]   # 12 router outputs
    n_cases = 0
    for N in (1, 2, 3):
        for combo in itertools.product(range(len(pairs)), repeat=N):
            topk = np.array([pairs[i] for i in combo], np.int32)
            for R in (1, 2, 4):
                for a in (1, 2, 4):
                    _same(oracle.plan(topk, E, R, a), definition_plan(topk, E, R, a))
                    n_cases += 1
    assert n_cases == (12 + 144 + 1728) * 9


def test_random_small_against_definition():
    rng = np.random.default_rng(20)
    for trial in range(600):
        R = int(rng.choice([1, 2, 4]))
        E = R * int(rng.integers(1, 4))
        K = int(rng.integers(1, E + 1))
        N = int(rng.integers(1, 9))
        a = int(rng.choice([1, 2, 3, 8]))
        distinct = bool(rng.integers(0, 2))
        topk = workloads.random_topk(rng, N, E, K, distinct=distinct)
        _same(oracle.plan(topk, E, R, a), definition_plan(topk, E, R, a))


@pytest.mark.parametrize("N,E,K,R,a,hot", [(2000, 64, 6, 8, 16, 0.0), (3000, 16, 3, 4, 5, 0.5),
                                            (500, 32, 8, 32, 1, 0.0), (1, 8, 8, 8, 128, 0.0)])
def test_invariants_medium(N, E, K, R, a, hot):
    rng = np.random.default_rng(21)
    topk = workloads.random_topk(rng, N, E, K, hot=hot)
    p = oracle.plan(topk, E, R, a)
    check_plan_invariants(p, topk, E, R, a)


def test_all_pairs_one_expert_and_empty_experts():
    topk = np.zeros((37, 1), np.int32)
    p = oracle.plan(topk, 8, 2, 16)
    assert p["tokens_per_expert"].tolist() == [37] + [0] * 7
    assert p["cu_seqlens"].tolist() == [0] + [48] * 8
    assert p["zero_fill_ranges"].tolist() == [[37, 11]] + [[0, 0]] * 7
    assert p["dst"].ravel().tolist() == list(range(37))
    check_plan_invariants(p, topk, 8, 2, 16)


def test_plan_argument_errors():
    topk = np.zeros((4, 2), np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.plan(topk, 6, 4, 1)           # E % R
    with pytest.raises(oracle.OracleError):
        oracle.plan(topk + 9, 8, 2, 1)       # id out of range
    with pytest.raises(oracle.OracleError):
        oracle.plan(topk, 8, 2, 0)           # alignment


@pytest.mark.parametrize("E,K,R,a", [(8, 2, 2, 8), (256, 8, 64, 128), (4, 1, 1, 1), (6, 3, 3, 5)])
def test_empty_batch(E, K, R, a):
    # no tokens: every count, offset and prefix is zero, no expert is padded
    # (an expert with no pairs pads to zero rows), and all E*(a-1) rows of
    # the capacity are unused; the counting definition agrees
    topk = np.zeros((0, K), np.int32)
    p = oracle.plan(topk, E, R, a)
    assert p["P"] == 0 and p["P_cap"] == E * (a - 1)
    for k in ("tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "pairs_per_rank", "tokens_per_rank",
              "rank_prefix", "rank_slot_offsets", "dup_counts"):
        assert not np.asarray(p[k]).any(), k
    assert p["cu_seqlens"].shape == (E + 1,) and p["rank_prefix"].shape == (R + 1,)
    assert p["src_of_slot"].tolist() == [-1] * (E * (a - 1))
    assert p["dst"].shape == (0, K) and p["is_token_in_rank"].shape == (0, R)
    assert len(p["dup_groups"]) == 0 and len(p["dup_loffs"]) == 0
    _same(p, definition_plan(topk, E, R, a))
