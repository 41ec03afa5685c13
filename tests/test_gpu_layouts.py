"""GPU parity of the tile map and the rank layout against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def routed(name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    topk, _ = oracle.route_topk(inp["logits"], w.K, scoring=w.scoring, renormalize=w.renormalize,
                                bias=inp["bias"], n_group=w.n_group, topk_group=w.topk_group,
                                routed_scaling=w.routed_scaling)
    return w, topk


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "large"])
def test_tile_map_and_rank_layout_workloads(m, name):
    w, topk = routed(name)
    p = m.plan(torch.from_numpy(topk).cuda(), w.E, w.R, w.alignment)
    te, tl, sizes = m.tile_map(p)
    want = oracle.plan(topk, w.E, w.R, w.alignment)
    o_te, o_tl, o_sizes = oracle.tile_map(want["tokens_per_expert"], w.alignment, te.numel())
    assert np.array_equal(te.cpu().numpy(), o_te) and np.array_equal(tl.cpu().numpy(), o_tl)
    assert np.array_equal(sizes.cpu().numpy(), o_sizes)
    for C in (1, 7, 48, 304):
        cpm, trs = m.rank_layout(p, C)
        o_cpm, o_trs = oracle.rank_layout(want["is_token_in_rank"], C)
        assert np.array_equal(cpm.cpu().numpy(), o_cpm) and np.array_equal(trs.cpu().numpy(), o_trs), C
    assert m.get_status(p) == 0


@pytest.mark.parametrize("N,E,K,R,a,C", [(1, 4, 2, 2, 1, 3), (5000, 16, 3, 8, 7, 5000), (70000, 8, 2, 8, 64, 1),
                                         (1023, 2, 1, 1, 1, 10), (1025, 64, 8, 64, 128, 33)])
def test_layout_shapes(m, N, E, K, R, a, C):
    rng = np.random.default_rng(N + C)
    topk = workloads.random_topk(rng, N, E, K)
    p = m.plan(torch.from_numpy(topk).cuda(), E, R, a)
    want = oracle.plan(topk, E, R, a)
    te, tl, sizes = m.tile_map(p)
    o = oracle.tile_map(want["tokens_per_expert"], a, te.numel())
    assert np.array_equal(te.cpu().numpy(), o[0]) and np.array_equal(tl.cpu().numpy(), o[1])
    assert np.array_equal(sizes.cpu().numpy(), o[2])
    cpm, trs = m.rank_layout(p, C)
    o_cpm, o_trs = oracle.rank_layout(want["is_token_in_rank"], C)
    assert np.array_equal(cpm.cpu().numpy(), o_cpm) and np.array_equal(trs.cpu().numpy(), o_trs)


def test_rank_layout_workspace_reused_across_sizes_and_calls(m):
    """One workspace, sized for the largest call, serves smaller calls in a
    row (no initialisation between them); a too-small one is refused."""
    from expert_dispatch_planning_gb300 import MoeError
    ws = m.rank_layout_workspace(9000, 64)
    for seed, (N, E, K, R, C) in enumerate([(9000, 256, 8, 64, 76), (300, 8, 2, 4, 7), (9000, 64, 4, 16, 1),
                                            (33, 64, 8, 64, 40)]):
        rng = np.random.default_rng(seed)
        topk = workloads.random_topk(rng, N, E, K)
        p = m.plan(torch.from_numpy(topk).cuda(), E, R, 1)
        want = oracle.plan(topk, E, R, 1)
        cpm, trs = m.rank_layout(p, C, workspace=ws)
        o_cpm, o_trs = oracle.rank_layout(want["is_token_in_rank"], C)
        assert np.array_equal(cpm.cpu().numpy(), o_cpm) and np.array_equal(trs.cpu().numpy(), o_trs), (N, R, C)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(MoeError):
        m.rank_layout(p, 3, workspace=small)
