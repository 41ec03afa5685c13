"""GPU parity: every step of the CUDA path against the CPU oracle.

Each stage is fed the same seeded inputs as the oracle (the plan gets the
oracle's routing, the combine the oracle's weights rounded to fp32), so each
comparison isolates one kernel.  Bars: bit-exact for indices, plans and
permuted rows; router weights within 1e-6 relative; the combine bit-exact
(both sides run the same fp32 fused multiply-add sequence; the stated
tolerance 1e-2 absolute is asserted as well).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from plan_checks import check_plan_invariants

pytestmark = pytest.mark.gpu

PLAN_KEYS = ["tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "dst", "src_of_slot",
             "is_token_in_rank", "tokens_per_rank", "pairs_per_rank", "rank_prefix",
             "rank_slot_offsets", "dup_groups", "dup_loffs", "dup_counts"]


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def dev():
    return torch.device("cuda:0")


def to_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_plan_equal(got, want):
    for k in PLAN_KEYS:
        g, w = np.asarray(got[k]), np.asarray(want[k])
        assert g.shape == w.shape and np.array_equal(g, w), "plan field %s differs" % k


def route_both(m, logits, K, bias=None, **kw):
    lg = torch.from_numpy(logits).to(dev())
    b = None if bias is None else torch.from_numpy(bias).to(dev())
    idx, w = m.route_topk(lg, K, bias=b, **kw)
    o_idx, o_w = oracle.route_topk(logits, K, bias=bias, **kw)
    return idx.cpu().numpy(), w.cpu().numpy(), o_idx, o_w


def check_route(m, logits, K, bias=None, **kw):
    idx, w, o_idx, o_w = route_both(m, logits, K, bias, **kw)
    assert np.array_equal(idx, o_idx), "first mismatch at row %d" % int(np.argwhere((idx != o_idx).any(1))[0][0])
    # 1e-6 relative wherever the exact weight is a normal fp32 number; an
    # fp32 output cannot carry relative precision below 2^-126
    err = np.abs(w.astype(np.float64) - o_w)
    ok = (err <= 1e-6 * np.abs(o_w)) | ((np.abs(o_w) < 2.0 ** -126) & (err <= 2.0 ** -126))
    assert ok.all(), (err / np.maximum(np.abs(o_w), 1e-300)).max()
    return o_idx, o_w


def route_kwargs(w):
    return dict(scoring=w.scoring, renormalize=w.renormalize, n_group=w.n_group,
                topk_group=w.topk_group, routed_scaling=w.routed_scaling)


# ---------------------------------------------------------------- router
@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "large"])
def test_route_configs(m, name):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    check_route(m, inp["logits"], w.K, inp["bias"], **route_kwargs(w))


@pytest.mark.parametrize("E,K,scoring,renorm,ng,tg", [
    (3, 2, 0, 1, 1, 1), (5, 5, 0, 0, 1, 1), (8, 1, 0, 1, 1, 1), (13, 4, 1, 1, 1, 1),
    (16, 3, 0, 0, 1, 1), (32, 8, 1, 0, 1, 1), (64, 6, 0, 1, 1, 1), (100, 7, 1, 1, 4, 2),
    (128, 16, 0, 1, 1, 1), (160, 8, 1, 1, 8, 3), (256, 32, 0, 1, 1, 1), (512, 8, 1, 1, 16, 4),
    (1024, 8, 0, 0, 1, 1), (1024, 12, 1, 1, 32, 4), (48, 32, 0, 1, 1, 1), (12, 4, 1, 1, 12, 4)])
def test_route_shapes(m, E, K, scoring, renorm, ng, tg):
    rng = np.random.default_rng(E * 131 + K)
    N = 777
    logits = rng.standard_normal((N, E), dtype=np.float32) * 3
    # force ties and signed zeros on some rows
    logits[::7] = np.round(logits[::7])
    logits[::11, : E // 2] = -0.0
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if scoring == 1 else None
    check_route(m, logits, K, bias, scoring=scoring, renormalize=bool(renorm), n_group=ng,
                topk_group=tg, routed_scaling=1.7)


def test_route_extreme_logits(m):
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((300, 64), dtype=np.float32) * 60   # sigmoid tails, subnormals
    logits[0] = 0.0
    logits[1] = 200.0
    logits[2] = -200.0
    check_route(m, logits, 8, rng.uniform(-0.1, 0.1, 64).astype(np.float32), scoring=1,
                renormalize=True, n_group=8, topk_group=2, routed_scaling=2.5)
    check_route(m, logits / 10, 8, scoring=0, renormalize=False)


# ---------------------------------------------------------------- plan
def plan_both(m, topk, E, R, a, out=None):
    p = m.plan(torch.from_numpy(topk).to(dev()), E, R, a, out=out)
    got = p.to_host()
    assert m.get_status(p) == 0
    want = oracle.plan(topk, E, R, a)
    return p, got, want


@pytest.fixture(params=["small", "medium", "cluster", "grid", "lookback"])
def plan_path(request, monkeypatch):
    """Force one plan path where the sizes allow it (the two-launch look-back
    plan otherwise): small = the E, R <= 32 cluster kernel and medium = the
    32 < E <= 256, R <= 32 one (the defaults where they apply), cluster = the
    general cluster kernel, grid = one launch over all SMs with every tile
    resident, lookback = the two-launch plan."""
    monkeypatch.setenv("MOE_PLAN_PATH", request.param)
    return request.param


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "large"])
def test_plan_configs(m, name, plan_path):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, with_x=False)
    o_idx, _ = oracle.route_topk(inp["logits"], w.K, bias=inp["bias"], **route_kwargs(w))
    _, got, want = plan_both(m, o_idx, w.E, w.R, w.alignment)
    assert_plan_equal(got, want)
    if name != "large":
        check_plan_invariants(got, o_idx, w.E, w.R, w.alignment)


@pytest.mark.parametrize("N,E,K,R,a,mode", [
    (1, 8, 2, 2, 8, "rand"), (1, 256, 8, 64, 128, "rand"), (7, 4, 4, 4, 1, "rand"),
    (333, 16, 1, 1, 4, "rand"), (1000, 8, 8, 8, 3, "rand"), (4097, 64, 3, 16, 16, "rand"),
    (5000, 32, 6, 32, 7, "rand"), (2500, 128, 16, 8, 64, "rand"), (700, 64, 32, 2, 2, "rand"),
    (9000, 8, 2, 4, 16, "hot"), (3000, 1024, 8, 128, 128, "rand"), (2049, 24, 5, 3, 9, "dups"),
    (600, 16, 4, 4, 5, "one"), (12345, 256, 8, 64, 128, "rand"), (20000, 96, 1, 96, 32, "rand"),
    # small and odd E / R: the shared-memory staging of is_token_in_rank must
    # stay 16-byte aligned for every layout
    (1134, 2, 1, 2, 1, "rand"), (777, 6, 2, 3, 5, "rand"), (333, 3, 3, 1, 2, "rand"),
    (2000, 10, 3, 5, 7, "rand"), (9001, 2, 2, 1, 4, "rand"), (40000, 6, 1, 2, 3, "rand"),
    # edges of the one-launch cluster kernels: small-E with 5-bit masks (E = R = 32),
    # K = 1 and the deepest ring (8 steps, 16 tiles); medium-E just above 32
    # experts, at 255 / 256 experts, R = 32, K = 32, alignment 1, one token
    (131072, 32, 1, 32, 4, "rand"), (16384, 32, 2, 32, 16, "hot"), (65536, 8, 1, 8, 2, "rand"),
    (8192, 33, 2, 3, 5, "rand"), (4096, 255, 5, 5, 7, "dups"), (8192, 256, 8, 32, 128, "rand"),
    (2048, 192, 32, 16, 3, "dups"), (100, 40, 7, 8, 1, "one"), (1, 33, 1, 1, 1, "rand")])
def test_plan_shapes(m, N, E, K, R, a, mode, plan_path):
    rng = np.random.default_rng(N + E + K)
    if mode == "one":      # every pair on expert 3: empty experts, one full
        topk = np.full((N, K), 3, np.int32)
        topk[:, 1:] = (3 + np.arange(1, K)) % E
    elif mode == "dups":   # repeated ids inside a token
        topk = rng.integers(0, E, size=(N, K)).astype(np.int32)
    else:
        topk = workloads.random_topk(rng, N, E, K, hot=0.7 if mode == "hot" else 0.0)
    _, got, want = plan_both(m, topk, E, R, a)
    assert_plan_equal(got, want)
    check_plan_invariants(got, topk, E, R, a)


def test_plan_workspace_reuse_across_calls_and_sizes(m, plan_path):
    rng = np.random.default_rng(9)
    E, R, a = 64, 8, 16
    big = m.Plan.allocate(6000, E, 8, R, a)
    ws = big.workspace
    for it in range(6):
        N = [6000, 100, 5999, 1, 3000, 6000][it]
        topk = workloads.random_topk(rng, N, E, 8)
        p = m.Plan.allocate(N, E, 8, R, a)
        p.workspace = ws          # one workspace, calls of different sizes in sequence
        _, got, want = plan_both(m, topk, E, R, a, out=p)
        assert_plan_equal(got, want)


def test_plan_launch_counts(m, monkeypatch):
    assert m.plan_launches(16384, 8, 2, 4) == 1          # small-E cluster kernel
    assert m.plan_launches(8192, 128, 8, 8) == 1         # medium-E cluster kernel
    assert m.plan_launches(65536, 256, 8, 64) == 2       # look-back plan
    monkeypatch.setenv("MOE_PLAN_PATH", "lookback")
    assert m.plan_launches(16384, 8, 2, 4) == 2
    monkeypatch.setenv("MOE_PLAN_PATH", "grid")
    assert m.plan_launches(65536, 256, 8, 64) == 1


def test_plan_bad_expert_id_reports_device_index(m):
    topk = np.zeros((64, 2), np.int32)
    topk[10, 1] = 8
    p = m.plan(torch.from_numpy(topk).to(dev()), 8, 2, 4)
    assert m.get_status(p) == 6


@pytest.mark.parametrize("path", ["grid", "lookback"])     # the paths with a workspace
def test_plan_uninitialised_workspace_reports_error(m, monkeypatch, path):
    monkeypatch.setenv("MOE_PLAN_PATH", path)
    topk = workloads.random_topk(np.random.default_rng(3), 4000, 16, 4)
    t = torch.from_numpy(topk).to(dev())
    p = m.Plan.allocate(4000, 16, 4, 4, 8)
    p.workspace.fill_(0xFF)
    m.plan(t, 16, 4, 8, out=p)
    assert m.get_status(p) == 7
    from expert_dispatch_planning_gb300 import _lib
    _lib.check("init", _lib.load().moe_plan_workspace_init(
        p.workspace.data_ptr(), p.workspace.numel(), torch.cuda.current_stream().cuda_stream))
    m.plan(t, 16, 4, 8, out=p)
    assert m.get_status(p) == 0
    assert_plan_equal(p.to_host(), oracle.plan(topk, 16, 4, 8))


@pytest.mark.parametrize("path", ["grid", "lookback"])     # the paths that wait on other tiles
def test_plan_bounded_wait_reports_timeout_and_recovers(m, monkeypatch, path):
    monkeypatch.setenv("MOE_PLAN_PATH", path)
    N, E, K, R, a = 20000, 64, 8, 8, 16     # several tiles
    topk = workloads.random_topk(np.random.default_rng(4), N, E, K)
    t = torch.from_numpy(topk).to(dev())
    p = m.Plan.allocate(N, E, K, R, a)
    x = torch.zeros((N, 64), dtype=torch.bfloat16, device=dev())
    sentinel = torch.full((p.P_cap, 64), 7.0, dtype=torch.bfloat16, device=dev())
    try:
        m.set_plan_fault(skip_tile=0, timeout_ns=20_000_000)   # tile 0 never publishes
        m.plan(t, E, R, a, out=p)
        m.permute(x, p, out=sentinel)                           # must not move rows by a failed plan
        torch.cuda.synchronize()
    finally:
        m.set_plan_fault(-1, 0)
    assert m.get_status(p) == 5
    assert bool((sentinel == 7.0).all())
    m.plan(t, E, R, a, out=p)                                   # the workspace is usable again
    assert m.get_status(p) == 0
    assert_plan_equal(p.to_host(), oracle.plan(topk, E, R, a))


# ---------------------------------------------------------------- permute / combine
def rows_case(m, name, N=None):
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0, N=N)
    o_idx, o_w = oracle.route_topk(inp["logits"], w.K, bias=inp["bias"], **route_kwargs(w))
    p = m.plan(torch.from_numpy(o_idx).to(dev()), w.E, w.R, w.alignment)
    want = oracle.plan(o_idx, w.E, w.R, w.alignment)
    assert_plan_equal(p.to_host(), want)
    return w, inp, o_idx, o_w, p, want


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3"])
def test_permute_combine_configs(m, name):
    w, inp, o_idx, o_w, p, want = rows_case(m, name)
    x = to_bf16(inp["x_bits"])
    sentinel = torch.full((p.P_cap, w.H), -3.0, dtype=torch.bfloat16, device=dev())
    perm = m.permute(x, p, out=sentinel)
    o_perm = oracle.permute(inp["x_bits"], want["dst"], want["zero_fill_ranges"], w.K, want["P_cap"],
                            fill=np.full((want["P_cap"], w.H), bits(torch.tensor([-3.0], dtype=torch.bfloat16))[0],
                                         np.uint16))
    assert np.array_equal(bits(perm), o_perm)
    # combine over arbitrary expert outputs y with the oracle's weights in fp32
    rng = np.random.default_rng(1)
    y_bits = workloads.make_x_bits(rng, want["P_cap"], w.H)
    w32 = o_w.astype(np.float32)
    out = m.combine(to_bf16(y_bits), torch.from_numpy(w32).to(dev()), p)
    o_out = oracle.combine(y_bits, w32, want["dst"])
    got = bits(out)
    assert np.array_equal(got, o_out)
    diff = np.abs(torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()
                  - torch.from_numpy(o_out.view(np.int16)).view(torch.bfloat16).float().numpy())
    assert diff.max() <= 1e-2
    assert m.get_status(p) == 0


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3"])
def test_permute_early_x_right_after_plan(m, name):
    """MOE_PERMUTE_EARLY_X directly after the plan call, x produced before it:
    the rows loaded while the plan kernel still runs give the same buffer."""
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0)
    o_idx, _ = oracle.route_topk(inp["logits"], w.K, bias=inp["bias"], **route_kwargs(w))
    want = oracle.plan(o_idx, w.E, w.R, w.alignment)
    x = to_bf16(inp["x_bits"])
    idx = torch.from_numpy(o_idx).to(dev())
    p = m.Plan.allocate(w.N, w.E, w.K, w.R, w.alignment)
    perm = torch.full((p.P_cap, w.H), -3.0, dtype=torch.bfloat16, device=dev())
    for _ in range(2):                      # back to back, no synchronisation in between
        m.plan(idx, w.E, w.R, w.alignment, out=p)
        m.permute(x, p, out=perm, early_x=True)
    o_perm = oracle.permute(inp["x_bits"], want["dst"], want["zero_fill_ranges"], w.K, want["P_cap"],
                            fill=np.full((want["P_cap"], w.H), bits(torch.tensor([-3.0], dtype=torch.bfloat16))[0],
                                         np.uint16))
    assert np.array_equal(bits(perm), o_perm)
    assert m.get_status(p) == 0


def test_permute_early_x_after_failed_plan_writes_nothing(m):
    topk = workloads.random_topk(np.random.default_rng(5), 4096, 8, 2)
    topk[100, 1] = 8                                             # expert id out of range
    x = torch.ones((4096, 256), dtype=torch.bfloat16, device=dev())
    idx = torch.from_numpy(topk).to(dev())
    p = m.Plan.allocate(4096, 8, 2, 4, 16)
    sentinel = torch.full((p.P_cap, 256), 7.0, dtype=torch.bfloat16, device=dev())
    m.plan(idx, 8, 4, 16, out=p)
    m.permute(x, p, out=sentinel, early_x=True)
    torch.cuda.synchronize()
    assert m.get_status(p) == 6
    assert bool((sentinel == 7.0).all())


def raw_slots(dst: np.ndarray) -> np.ndarray:
    """Row of each pair in the permuted buffer (dst encodes duplicates as -row-1)."""
    return np.where(dst >= 0, dst, -dst - 1).astype(np.int64)


def oracle_rows_of_tokens(x_bits, dst, K, s0, s1):
    """The oracle's permute restricted to tokens [s0, s1): their K rows each,
    in pair order (local row j = pair s0*K + j), as uint16[(s1-s0)*K, H].

    The pairs' rows are distinct (one pair per non-pad slot), so relabelling
    them 0..n-1 (keeping the duplicate sign encoding) leaves what the oracle
    writes into each row unchanged."""
    d = dst[s0 * K:s1 * K]
    j = np.arange(d.size, dtype=np.int32)
    local = np.where(d >= 0, j, -j - 1).astype(np.int32)
    return oracle.permute(x_bits[s0:s1], local, np.zeros((0, 2), np.int32), K, d.size), local


def row_scale(rows: torch.Tensor) -> torch.Tensor:
    """A per-row factor for stand-in experts (so a token's K rows differ)."""
    return 1.0 + (rows % 7).float() / 8.0


@pytest.mark.parametrize("chunk", [4096])
def test_permute_combine_large_full(m, chunk):
    """The large dedup-heavy workload at full size, in the benchmark's launch
    configuration: every permuted row against the oracle's permute (token
    slices, plus the pad rows), then the combine of per-row scaled rows
    against the oracle's combine for every token, all bit-exact."""
    w, inp, o_idx, o_w, p, want = rows_case(m, "large")
    x = to_bf16(inp["x_bits"])
    P, P_cap, K, H = want["P"], want["P_cap"], w.K, w.H
    perm = torch.empty((P_cap, H), dtype=torch.bfloat16, device=dev())
    perm[P:] = 5.0
    m.permute(x, p, out=perm, early_x=True)     # as the benchmark launches it (the fill above is not x)
    dst = want["dst"].reshape(-1)
    raw = raw_slots(dst)
    raw_t = torch.from_numpy(raw).to(dev())
    for s0 in range(0, w.N, chunk):
        s1 = min(w.N, s0 + chunk)
        o_rows, _ = oracle_rows_of_tokens(inp["x_bits"], dst, K, s0, s1)
        assert np.array_equal(bits(perm.index_select(0, raw_t[s0 * K:s1 * K])), o_rows), "tokens %d.." % s0
    # pad rows: the oracle's permute of no tokens over the zero-fill ranges,
    # relabelled to consecutive rows
    zfr = want["zero_fill_ranges"].reshape(-1, 2)
    pads = np.concatenate([np.arange(st, st + c) for st, c in zfr if c > 0]).astype(np.int64)
    counts = np.array([c for _, c in zfr if c > 0], np.int64)
    local_z = np.stack([np.concatenate([[0], np.cumsum(counts)[:-1]]), counts], 1).astype(np.int32)
    o_pads = oracle.permute(np.zeros((0, H), np.uint16), np.zeros((0, K), np.int32), local_z, K, pads.size,
                            fill=np.full((pads.size, H), 0x7F7F, np.uint16))
    assert np.array_equal(bits(perm.index_select(0, torch.from_numpy(pads).to(dev()))), o_pads)
    assert bool((perm[P:] == 5.0).all())           # rows past the plan are left alone
    # combine: stand-in experts scale each row by row_scale (torch bf16 on both sides)
    y = torch.empty_like(perm)
    for r0 in range(0, P_cap, 1 << 16):
        r1 = min(P_cap, r0 + (1 << 16))
        y[r0:r1] = (perm[r0:r1].float() * row_scale(torch.arange(r0, r1, device=dev()))[:, None]).to(torch.bfloat16)
    del perm
    w32 = o_w.astype(np.float32)
    out = bits(m.combine(y, torch.from_numpy(w32).to(dev()), p))
    assert m.get_status(p) == 0
    for s0 in range(0, w.N, chunk):
        s1 = min(w.N, s0 + chunk)
        o_rows, local = oracle_rows_of_tokens(inp["x_bits"], dst, K, s0, s1)
        o_y = (torch.from_numpy(o_rows.view(np.int16)).view(torch.bfloat16).float()
               * row_scale(torch.from_numpy(raw[s0 * K:s1 * K]))[:, None]).to(torch.bfloat16)
        o_out = oracle.combine(o_y.view(torch.int16).numpy().view(np.uint16), w32[s0:s1], local.reshape(-1, K))
        assert np.array_equal(out[s0:s1], o_out), "combined tokens %d.." % s0


@pytest.mark.parametrize("N,E,K,R,H,a", [(1, 8, 2, 2, 8, 4), (37, 8, 3, 4, 24, 1), (500, 16, 5, 4, 136, 8),
                                          (1000, 64, 7, 8, 72, 16), (300, 32, 16, 8, 512, 3),
                                          (129, 64, 32, 4, 64, 2), (2000, 8, 1, 8, 1024, 64),
                                          (40, 8, 3, 2, 49152, 4)])   # the largest row: 96 KB
def test_permute_combine_shapes(m, N, E, K, R, H, a):
    rng = np.random.default_rng(N * 7 + K)
    topk = workloads.random_topk(rng, N, E, K)
    p = m.plan(torch.from_numpy(topk).to(dev()), E, R, a)
    want = oracle.plan(topk, E, R, a)
    x_bits = workloads.make_x_bits(rng, N, H)
    perm = torch.full((want["P_cap"], H), 9.0, dtype=torch.bfloat16, device=dev())
    m.permute(to_bf16(x_bits), p, out=perm)
    fill = np.full((want["P_cap"], H), bits(torch.tensor([9.0], dtype=torch.bfloat16))[0], np.uint16)
    assert np.array_equal(bits(perm), oracle.permute(x_bits, want["dst"], want["zero_fill_ranges"], K,
                                                     want["P_cap"], fill=fill))
    wts = rng.random((N, K)).astype(np.float32)
    y_bits = workloads.make_x_bits(rng, want["P_cap"], H)
    out = m.combine(to_bf16(y_bits), torch.from_numpy(wts).to(dev()), p)
    assert np.array_equal(bits(out), oracle.combine(y_bits, wts, want["dst"]))
    assert m.get_status(p) == 0


# ---------------------------------------------------------------- end to end
@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "large"])
def test_end_to_end(m, name):
    """GPU chain route -> plan -> permute -> experts -> combine against the
    oracle chain, each side computing its own intermediates from the same
    inputs.  The stand-in experts scale each row by 1 + e/E (bf16, torch on
    both sides) so the combined sums are not exact bf16 ties.  The oracle
    side runs its permute and combine over slices of tokens (each token's
    rows are all a combine reads).  The weights agree within 1e-6, so an
    output may differ by one bf16 rounding step where the fp32 sum falls next
    to a rounding boundary."""
    w = workloads.get(name)
    inp = workloads.make_inputs(w, seed=0)
    lg = torch.from_numpy(inp["logits"]).to(dev())
    b = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev())
    x = to_bf16(inp["x_bits"])
    idx, wts = m.route_topk(lg, w.K, bias=b, **route_kwargs(w))
    p = m.plan(idx, w.E, w.R, w.alignment)
    perm = m.permute(x, p)
    cu = p.cu_seqlens.long()
    y = torch.empty_like(perm)
    for r0 in range(0, p.P_cap, 1 << 16):
        r1 = min(p.P_cap, r0 + (1 << 16))
        row_expert = torch.searchsorted(cu[1:], torch.arange(r0, r1, device=dev()), right=True).clamp(max=w.E - 1)
        y[r0:r1] = (perm[r0:r1].float() * (1.0 + row_expert.float() / w.E)[:, None]).to(torch.bfloat16)
    del perm
    out = bits(m.combine(y, wts, p))
    assert m.get_status(p) == 0
    o_idx, o_w = oracle.route_topk(inp["logits"], w.K, bias=inp["bias"], **route_kwargs(w))
    op = oracle.plan(o_idx, w.E, w.R, w.alignment)
    dst = op["dst"].reshape(-1)
    n_diff = 0
    for s0 in range(0, w.N, 4096):
        s1 = min(w.N, s0 + 4096)
        o_rows, local = oracle_rows_of_tokens(inp["x_bits"], dst, w.K, s0, s1)
        scale = torch.from_numpy(1.0 + o_idx[s0:s1].reshape(-1).astype(np.float32) / w.E)   # each pair's expert
        o_y = (torch.from_numpy(o_rows.view(np.int16)).view(torch.bfloat16).float() * scale[:, None]
               ).to(torch.bfloat16)
        o_out = oracle.combine(o_y.view(torch.int16).numpy().view(np.uint16), o_w[s0:s1].astype(np.float32),
                               local.reshape(-1, w.K))
        g = torch.from_numpy(out[s0:s1].view(np.int16)).view(torch.bfloat16).double().numpy()
        o = torch.from_numpy(o_out.view(np.int16)).view(torch.bfloat16).double().numpy()
        ulp = np.maximum(np.abs(o), 2.0 ** -126) * 2.0 ** -7
        assert np.all(np.abs(g - o) <= np.maximum(1e-2, ulp * 1.0001)), "tokens %d.." % s0
        n_diff += int(np.count_nonzero(g != o))
    assert n_diff < 1e-3 * w.N * w.H


@pytest.mark.parametrize("E,K,R,a", [(8, 2, 2, 8), (256, 8, 64, 128), (4, 1, 1, 1), (6, 3, 3, 5)])
def test_empty_batch(m, E, K, R, a):
    """A batch with no tokens: routing launches nothing, the plan equals the
    oracle's empty plan (every output written over a sentinel), permute and
    combine move no rows and leave the permuted buffer as it was, and the
    plan's tile map, copy, rank layout and balanced plan equal the oracle's
    (all empty or zero)."""
    p = m.Plan.allocate(0, E, K, R, a)
    for k in PLAN_KEYS:
        t = getattr(p, k)
        if t.dtype == torch.int32:
            t.fill_(0x5A5A5A5A)
    logits = torch.empty((0, E), dtype=torch.float32, device=dev())
    idx, wts, p = m.route_plan(logits, K, R, a, out=p)
    assert idx.shape == (0, K) and wts.shape == (0, K)
    assert m.route_plan_launches(0, E, K, R) == 1 == m.plan_launches(0, E, K, R)
    want = oracle.plan(np.zeros((0, K), np.int32), E, R, a)
    assert_plan_equal(p.to_host(), want)

    H = 64
    x = torch.empty((0, H), dtype=torch.bfloat16, device=dev())
    perm = torch.full((p.P_cap, H), 1.5, dtype=torch.bfloat16, device=dev())
    m.permute(x, p, out=perm, early_x=True)
    out = m.combine(perm, wts, p)
    assert out.shape == (0, H)
    assert bool((perm == 1.5).all())
    te, tl, sizes = m.tile_map(p)
    assert sizes.tolist() == [0, 0] and bool((te == -1).all()) and bool((tl == -1).all())
    c = p.clone()
    assert_plan_equal(c.to_host(), want)
    cpm, trs = m.rank_layout(p, 5)
    assert cpm.shape == (R, 5) and not bool(cpm.any()) and trs.shape == (0, R)
    B = 2
    b = m.plan_balanced(idx, p, a, 0, B, 64).to_host()
    o_b = oracle.plan_balanced(np.zeros((0, K), np.int32), E, R, a, 0, B, 64)
    for k, v in o_b.items():
        assert np.array_equal(b[k].reshape(v.shape), v), k
    assert m.get_status(p) == 0 and m.get_status(c) == 0


def test_plan_reuse_and_copy(m):
    """A plan serves several permute/combine calls; a copied plan is identical
    and keeps working after the original's buffers are overwritten."""
    w, inp, o_idx, o_w, p, want = rows_case(m, "qwen3")
    rng = np.random.default_rng(17)
    c = p.clone()
    assert_plan_equal(c.to_host(), want)
    p.dst.fill_(0)          # the copy owns its buffers
    w32 = torch.from_numpy(o_w.astype(np.float32)).to(dev())
    for it in range(2):
        x_bits = workloads.make_x_bits(rng, w.N, w.H)
        perm = m.permute(to_bf16(x_bits), c)
        o_perm = oracle.permute(x_bits, want["dst"], want["zero_fill_ranges"], w.K, want["P_cap"])
        assert np.array_equal(bits(perm)[: want["P"]], o_perm[: want["P"]])
        out = m.combine(perm, w32, c)
        assert np.array_equal(bits(out), oracle.combine(o_perm, o_w.astype(np.float32), want["dst"]))
    assert m.get_status(c) == 0


def test_concurrent_callers_on_separate_streams(m):
    """Host threads calling the library at once (ctypes releases the GIL), each
    on its own stream with its own plan buffers and workspace: every result
    equals the oracle's.  Covers the library's host-side caches (SM count,
    kernel attributes, path choice) under concurrent first use."""
    import threading
    shapes = [(3000, 8, 2, 4, 16), (2000, 128, 8, 8, 128), (20000, 256, 8, 64, 128), (777, 6, 3, 3, 5)]
    errors = []

    def worker(tid):
        try:
            rng = np.random.default_rng(1000 + tid)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for it in range(6):
                    N, E, K, R, a = shapes[(tid + it) % len(shapes)]
                    topk = workloads.random_topk(rng, N, E, K, hot=0.5)
                    p = m.plan(torch.from_numpy(topk).to(dev()), E, R, a)
                    H = 64
                    x_bits = workloads.make_x_bits(rng, N, H)
                    perm = m.permute(to_bf16(x_bits), p)
                    got = p.to_host()
                    want = oracle.plan(topk, E, R, a)
                    assert_plan_equal(got, want)
                    o_perm = oracle.permute(x_bits, want["dst"], want["zero_fill_ranges"], K, want["P_cap"])
                    assert np.array_equal(bits(perm)[: want["P"]], o_perm[: want["P"]])
                    assert m.get_status(p, stream=stream) == 0
        except Exception as e:  # reported on the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
