"""Pins for the oracle's grouped-GEMM tile map and rank layout: hand-derived
cases, consistency with the plan's padded offsets, and invariants."""
import numpy as np
import pytest

import oracle
import workloads


def test_tile_map_worked_example():
    # counts [5, 0, 3], tiles of 4: expert 0 -> 2 tiles (rows 0-3, 4; limit 4, 5),
    # expert 1 none, expert 2 -> tile 2 (rows 8-10, limit 11); 3 tiles, 12 rows
    te, tl, sizes = oracle.tile_map([5, 0, 3], 4, 5)
    assert te.tolist() == [0, 0, 2, -1, -1]
    assert tl.tolist() == [4, 5, 11, -1, -1]
    assert sizes.tolist() == [3, 12]


@pytest.mark.parametrize("seed", range(6))
def test_tile_map_matches_plan_offsets(seed):
    rng = np.random.default_rng(70 + seed)
    E, R, K, N = 32, 4, 4, int(rng.integers(1, 2000))
    a = int(rng.choice([1, 8, 128]))
    topk = workloads.random_topk(rng, N, E, K, hot=0.5)
    p = oracle.plan(topk, E, R, a)
    max_tiles = p["P_cap"] // a + 1
    te, tl, sizes = oracle.tile_map(p["tokens_per_expert"], a, max_tiles)
    cu, cnt = p["cu_seqlens"], p["tokens_per_expert"]
    assert sizes.tolist() == [p["P"] // a, p["P"]]
    for t in range(sizes[0]):
        e = te[t]
        assert cu[e] <= t * a < cu[e + 1]                  # the tile lies in its expert's rows
        assert tl[t] == min((t + 1) * a, cu[e] + cnt[e])    # and stops at its real rows
    assert np.all(te[sizes[0]:] == -1)


def test_rank_layout_worked_example():
    itr = np.array([[1, 0], [1, 1], [0, 1], [1, 1], [0, 0]], np.uint8)
    # 2 channels of 3 tokens: rank 0 counts (2, 1) -> prefix (2, 3); rank 1 (2, 1) -> (2, 3)
    cpm, trs = oracle.rank_layout(itr, 2)
    assert cpm.tolist() == [[2, 3], [2, 3]]
    # rank 0 holds tokens 0,1,3 at 0,1,2; rank 1 holds 1,2,3 at 3,4,5
    assert trs.tolist() == [[0, -1], [1, 3], [-1, 4], [2, 5], [-1, -1]]


@pytest.mark.parametrize("seed", range(6))
def test_rank_layout_invariants(seed):
    rng = np.random.default_rng(90 + seed)
    N, R = int(rng.integers(1, 3000)), int(rng.choice([1, 2, 8, 64]))
    C = int(rng.integers(1, 200))
    itr = (rng.random((N, R)) < rng.random()).astype(np.uint8)
    cpm, trs = oracle.rank_layout(itr, C)
    tpr = itr.sum(0)
    assert np.array_equal(cpm[:, -1], tpr) and np.all(np.diff(cpm, axis=1) >= 0)
    prefix = np.concatenate([[0], np.cumsum(tpr)]).astype(np.int64)
    for r in range(R):
        rows = np.nonzero(itr[:, r])[0]
        assert trs[rows, r].tolist() == list(range(prefix[r], prefix[r + 1]))
        assert np.all(trs[itr[:, r] == 0, r] == -1)


def test_rank_layout_empty_batch():
    # no tokens: every channel is empty, so every prefix is zero
    cpm, trs = oracle.rank_layout(np.zeros((0, 4), np.uint8), 3)
    assert cpm.shape == (4, 3) and not cpm.any()
    assert trs.shape == (0, 4)
