"""GPU parity of route_plan (routing and the dispatch plan in one call):
identical to route_topk followed by plan, bit for bit, whether it runs as
the fused one-launch kernel or as the two calls; and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from plan_checks import check_plan_invariants
from test_gpu_parity import assert_plan_equal, dev, m, route_kwargs  # noqa: F401  (m: fixture)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def fused_on(monkeypatch):
    monkeypatch.setenv("MOE_ROUTE_PLAN_FUSED", "1")   # the one-launch kernel is opt-in


def oracle_check(topk, w, logits, K, E, R, a, bias=None, **kw):
    o_idx, o_w = oracle.route_topk(logits, K, bias=bias, **kw)
    assert np.array_equal(topk, o_idx), "first mismatch at row %d" % int(np.argwhere((topk != o_idx).any(1))[0][0])
    err = np.abs(w.astype(np.float64) - o_w)
    ok = (err <= 1e-6 * np.abs(o_w)) | ((np.abs(o_w) < 2.0 ** -126) & (err <= 2.0 ** -126))
    assert ok.all(), (err / np.maximum(np.abs(o_w), 1e-300)).max()
    return o_idx


def run_both(m, logits, K, R, a, bias=None, **kw):
    lg = torch.from_numpy(logits).to(dev())
    b = None if bias is None else torch.from_numpy(bias).to(dev())
    E = logits.shape[1]
    idx2, w2 = m.route_topk(lg, K, bias=b, **kw)
    p2 = m.plan(idx2, E, R, a)
    idx1, w1, p1 = m.route_plan(lg, K, R, a, bias=b, **kw)
    assert m.get_status(p1) == 0 and m.get_status(p2) == 0
    assert torch.equal(idx1, idx2)
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))   # bit for bit
    got = p1.to_host()
    assert_plan_equal(got, p2.to_host())
    return idx1.cpu().numpy(), w1.cpu().numpy(), got


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "large"])
def test_route_plan_configs(m, name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    fused = m.route_plan_launches(w.N, w.E, w.K, w.R, w.n_group) == 1
    assert fused == (name in ("tiny", "mixtral"))
    topk, wts, got = run_both(m, inp["logits"], w.K, w.R, w.alignment, bias=inp["bias"], **route_kwargs(w))
    o_idx = oracle_check(topk, wts, inp["logits"], w.K, w.E, w.R, w.alignment, bias=inp["bias"], **route_kwargs(w))
    assert_plan_equal(got, oracle.plan(o_idx, w.E, w.R, w.alignment))


@pytest.mark.parametrize("N,E,K,R,a,scoring,renorm", [      # scoring 0 softmax, 1 sigmoid
    (1, 8, 2, 2, 8, 0, True), (777, 8, 2, 4, 16, 0, False), (1000, 8, 1, 8, 3, 1, True),
    (4097, 4, 4, 2, 5, 1, False), (3000, 8, 8, 4, 1, 0, True), (65536, 8, 2, 8, 16, 0, True),
    (131072, 8, 1, 1, 4, 1, True), (5000, 4, 2, 4, 2, 0, True), (300, 8, 4, 8, 7, 1, True)])
def test_route_plan_fused_shapes(m, N, E, K, R, a, scoring, renorm):
    assert m.route_plan_launches(N, E, K, R) == 1
    rng = np.random.default_rng(N + 7 * E + K)
    logits = (rng.standard_normal((N, E), dtype=np.float32) * 3).astype(np.float32)
    logits[::13, : E // 2] = -0.0        # ties and signed zeros
    logits[5::17] = 0.25
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if scoring == 1 else None
    kw = dict(scoring=scoring, renormalize=renorm, routed_scaling=1.7)
    topk, wts, got = run_both(m, logits, K, R, a, bias=bias, **kw)
    o_idx = oracle_check(topk, wts, logits, K, E, R, a, bias=bias, **kw)
    assert_plan_equal(got, oracle.plan(o_idx, E, R, a))
    if N <= 5000:
        check_plan_invariants(got, o_idx, E, R, a)


def test_route_plan_launch_counts(m, monkeypatch):
    assert m.route_plan_launches(16384, 8, 2, 4) == 1
    assert m.route_plan_launches(16384, 8, 3, 4) == 1 + m.plan_launches(16384, 8, 3, 4)   # K not a power of two
    assert m.route_plan_launches(8192, 128, 8, 8) == 2                                       # E > 8
    assert m.route_plan_launches(4096, 8, 2, 2, n_group=2) == 2                              # group limit
    monkeypatch.setenv("MOE_ROUTE_PLAN_FUSED", "0")                                         # the default
    assert m.route_plan_launches(16384, 8, 2, 4) == 2


def test_route_plan_then_early_permute(m):
    """The benchmark's chain: fused route + plan, then the permute loading x
    early, back to back without synchronisation."""
    w = workloads.get("mixtral")
    inp = workloads.make_inputs(w, seed=3, N=4096)
    lg = torch.from_numpy(inp["logits"]).to(dev())
    x = torch.from_numpy(inp["x_bits"].view(np.int16)).view(torch.bfloat16).to(dev())
    p = m.Plan.allocate(4096, w.E, w.K, w.R, w.alignment)
    perm = torch.full((p.P_cap, w.H), -3.0, dtype=torch.bfloat16, device=dev())
    for _ in range(3):
        idx, wts, _ = m.route_plan(lg, w.K, w.R, w.alignment, out=p, **route_kwargs(w))
        m.permute(x, p, out=perm, early_x=True)
    o_idx, _ = oracle.route_topk(inp["logits"], w.K, **route_kwargs(w))
    want = oracle.plan(o_idx, w.E, w.R, w.alignment)
    fill = np.full((want["P_cap"], w.H), np.frombuffer(np.float32(-3.0).tobytes(), np.uint16)[1], np.uint16)
    o_perm = oracle.permute(inp["x_bits"], want["dst"], want["zero_fill_ranges"], w.K, want["P_cap"], fill=fill)
    assert np.array_equal(perm.view(torch.int16).cpu().numpy().view(np.uint16), o_perm)
    assert m.get_status(p) == 0
