"""Guard zones around every output: no kernel writes outside its arrays.

compute-sanitizer is not available on the GPUs this library is tested on, so
here every output array (and every caller workspace) is the middle of a
larger device buffer whose 256-byte guard zones before and after hold a byte
pattern.  The calls go through the C ABI with those interior pointers; after
them every guard must still hold the pattern and every interior must equal
the oracle.  Covered: the router (exact and approximate-key kernels), each
plan path, permute, combine, the tile map, the rank layout and the balanced
plan.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

GUARD_BYTES = 256   # keeps every interior 256-byte aligned
PATTERN = 0x5A


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from expert_dispatch_planning_gb300 import _lib
    return _lib


class Guarded:
    """Device arrays, each inside a pattern-filled buffer with guard zones."""

    def __init__(self):
        self.bufs = {}

    def alloc(self, name, n, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        g = GUARD_BYTES // esz
        raw = torch.full(((n + 2 * g) * esz,), PATTERN, dtype=torch.uint8, device="cuda")
        self.bufs[name] = (raw, GUARD_BYTES, n * esz)
        return raw.view(dtype)[g:g + n]

    def check(self):
        torch.cuda.synchronize()
        for name, (raw, off, nb) in self.bufs.items():
            h = raw.cpu().numpy()
            assert (h[:off] == PATTERN).all(), "write before " + name
            assert (h[off + nb:] == PATTERN).all(), "write after " + name


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


PLAN_FIELDS = ["tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "pairs_per_rank", "tokens_per_rank",
               "rank_prefix", "rank_slot_offsets", "is_token_in_rank", "dst", "src_of_slot", "dup_groups",
               "dup_loffs", "dup_counts", "status"]


def guarded_plan(lib, G, topk, E, R, a):
    """moe_plan into guarded outputs and a guarded workspace; returns (arrays, struct)."""
    N, K = topk.shape
    L = lib.load()
    cap = int(L.moe_plan_capacity_rows(N, E, K, a))
    i32, u8 = torch.int32, torch.uint8
    sizes = dict(tokens_per_expert=E, cu_seqlens=E + 1, zero_fill_ranges=2 * E, pairs_per_rank=R,
                 tokens_per_rank=R, rank_prefix=R + 1, rank_slot_offsets=R + 1, is_token_in_rank=N * R,
                 dst=N * K, src_of_slot=cap, dup_groups=3 * N * (K // 2), dup_loffs=N * (K - 1), dup_counts=2,
                 status=4)
    arr = {k: G.alloc(k, sizes[k], u8 if k == "is_token_in_rank" else i32) for k in PLAN_FIELDS}
    arr["status"].zero_()
    st = lib.MoePlanOut(*[arr[k].data_ptr() for k in PLAN_FIELDS])
    ws_bytes = int(L.moe_plan_workspace_size(N, E, K, R))
    ws = G.alloc("workspace", ws_bytes, u8)
    lib.check("moe_plan_workspace_init", L.moe_plan_workspace_init(_p(ws), ws_bytes, _stream()))
    t = torch.from_numpy(topk).cuda()
    lib.check("moe_plan", L.moe_plan(_p(t), N, E, K, R, a, _p(ws), ws_bytes, ctypes.byref(st), _stream()))
    return arr, st


def check_plan(arr, want, K):
    host = {k: v.cpu().numpy() for k, v in arr.items()}
    assert host["status"][0] == 0
    for k in ("tokens_per_expert", "cu_seqlens", "pairs_per_rank", "tokens_per_rank", "rank_prefix",
              "rank_slot_offsets", "src_of_slot", "dup_counts"):
        assert np.array_equal(host[k], np.asarray(want[k]).ravel()), k
    assert np.array_equal(host["zero_fill_ranges"], want["zero_fill_ranges"].ravel())
    assert np.array_equal(host["is_token_in_rank"], want["is_token_in_rank"].ravel())
    assert np.array_equal(host["dst"], want["dst"].ravel())
    g, d = int(want["dup_counts"][0]), int(want["dup_counts"][1])
    assert np.array_equal(host["dup_groups"][: 3 * g], want["dup_groups"].ravel())
    assert np.array_equal(host["dup_loffs"][:d], want["dup_loffs"].ravel())


# the default path of each size class, and the paths MOE_PLAN_PATH can force
@pytest.mark.parametrize("path", ["auto", "small", "medium", "cluster", "grid", "lookback"])
@pytest.mark.parametrize("N,E,K,R,a", [(5000, 8, 2, 4, 16), (3000, 128, 8, 8, 128), (20000, 256, 8, 64, 128),
                                       (777, 6, 3, 3, 5), (1, 1024, 32, 128, 2), (0, 256, 8, 64, 128)])
def test_plan_writes_only_its_arrays(lib, monkeypatch, path, N, E, K, R, a):
    monkeypatch.setenv("MOE_PLAN_PATH", path)
    rng = np.random.default_rng(N + E)
    topk = workloads.random_topk(rng, N, E, K, hot=0.5)
    G = Guarded()
    arr, _ = guarded_plan(lib, G, topk, E, R, a)
    G.check()
    check_plan(arr, oracle.plan(topk, E, R, a), K)


@pytest.mark.parametrize("route_path", ["exact", "fast"])
@pytest.mark.parametrize("N,E,K,scoring,ng,tg", [(3001, 8, 2, 0, 1, 1), (2049, 256, 8, 1, 8, 4),
                                                 (1500, 128, 8, 0, 1, 1), (333, 1024, 32, 0, 1, 1)])
def test_route_writes_only_its_arrays(lib, monkeypatch, route_path, N, E, K, scoring, ng, tg):
    monkeypatch.setenv("MOE_ROUTE_PATH", route_path)
    rng = np.random.default_rng(N * 3 + E)
    logits = rng.standard_normal((N, E), dtype=np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if scoring == 1 else None
    G = Guarded()
    d_logits = G.alloc("logits", N * E, torch.float32)
    d_logits.copy_(torch.from_numpy(logits.ravel()))
    d_bias = None
    if bias is not None:
        d_bias = G.alloc("bias", E, torch.float32)
        d_bias.copy_(torch.from_numpy(bias))
    idx = G.alloc("topk_idx", N * K, torch.int32)
    w = G.alloc("topk_w", N * K, torch.float32)
    L = lib.load()
    lib.check("moe_route_topk", L.moe_route_topk(_p(d_logits), None if d_bias is None else _p(d_bias), N, E, K,
                                                 scoring, 1, ng, tg, 2.5, _p(idx), _p(w), _stream()))
    G.check()
    o_idx, o_w = oracle.route_topk(logits, K, scoring=scoring, renormalize=True, bias=bias, n_group=ng,
                                   topk_group=tg, routed_scaling=2.5)
    assert np.array_equal(idx.cpu().numpy(), o_idx.ravel())
    err = np.abs(w.cpu().numpy().astype(np.float64) - o_w.ravel())
    assert (err <= 1e-6 * np.abs(o_w.ravel()) + 2.0 ** -126).all()


@pytest.mark.parametrize("N,E,K,R,H,a", [(1000, 16, 4, 4, 136, 8), (300, 8, 2, 4, 4096, 16),
                                         (257, 64, 8, 8, 7168, 128), (40, 8, 3, 2, 49152, 4)])
def test_rows_write_only_their_arrays(lib, N, E, K, R, H, a):
    rng = np.random.default_rng(N + H)
    topk = workloads.random_topk(rng, N, E, K)
    G = Guarded()
    arr, st = guarded_plan(lib, G, topk, E, R, a)
    want = oracle.plan(topk, E, R, a)
    cap = want["P_cap"]
    L = lib.load()
    x_bits = workloads.make_x_bits(rng, N, H)
    x = G.alloc("x", N * H, torch.int16)
    x.copy_(torch.from_numpy(x_bits.view(np.int16).ravel()))
    perm = G.alloc("permuted", cap * H, torch.int16)
    lib.check("moe_permute", L.moe_permute(_p(x), N, H, K, E, a, ctypes.byref(st), _p(perm), 0, _stream()))
    wts = rng.random((N, K)).astype(np.float32)
    d_w = G.alloc("topk_w", N * K, torch.float32)
    d_w.copy_(torch.from_numpy(wts.ravel()))
    out = G.alloc("out", N * H, torch.int16)
    lib.check("moe_combine", L.moe_combine(_p(perm), _p(d_w), N, K, H, E, a, ctypes.byref(st), _p(out), _stream()))
    G.check()
    fill = np.full((cap, H), PATTERN * 0x101, np.uint16)   # rows the permute leaves alone keep the pattern
    o_perm = oracle.permute(x_bits, want["dst"], want["zero_fill_ranges"], K, cap, fill=fill)
    assert np.array_equal(perm.cpu().numpy().view(np.uint16).reshape(cap, H), o_perm)
    assert np.array_equal(out.cpu().numpy().view(np.uint16).reshape(N, H), oracle.combine(o_perm, wts, want["dst"]))
    assert int(arr["status"][0]) == 0


@pytest.mark.parametrize("N,E,K,R,a,C", [(5000, 16, 3, 8, 7, 33), (20000, 256, 8, 64, 128, 76), (31, 4, 2, 4, 1, 7)])
def test_layouts_write_only_their_arrays(lib, N, E, K, R, a, C):
    rng = np.random.default_rng(N + C)
    topk = workloads.random_topk(rng, N, E, K)
    G = Guarded()
    arr, st = guarded_plan(lib, G, topk, E, R, a)
    want = oracle.plan(topk, E, R, a)
    L = lib.load()
    max_tiles = max(1, want["P_cap"] // a)
    te = G.alloc("tile_expert", max_tiles, torch.int32)
    tl = G.alloc("tile_row_limit", max_tiles, torch.int32)
    sizes = G.alloc("sizes", 2, torch.int32)
    lib.check("moe_tile_map", L.moe_tile_map(ctypes.byref(st), E, a, _p(te), _p(tl), max_tiles, _p(sizes),
                                             _stream()))
    ws_bytes = int(L.moe_rank_layout_workspace_size(N, R))
    ws = G.alloc("rank_layout_workspace", ws_bytes, torch.uint8)
    cpm = G.alloc("channel_prefix_matrix", R * C, torch.int32)
    trs = G.alloc("token_rank_slot", N * R, torch.int32)
    lib.check("moe_rank_layout", L.moe_rank_layout(ctypes.byref(st), N, R, C, _p(ws), ws_bytes, _p(cpm), _p(trs),
                                                   _stream()))
    G.check()
    o_te, o_tl, o_sizes = oracle.tile_map(want["tokens_per_expert"], a, max_tiles)
    assert np.array_equal(te.cpu().numpy(), o_te) and np.array_equal(tl.cpu().numpy(), o_tl)
    assert np.array_equal(sizes.cpu().numpy(), o_sizes)
    o_cpm, o_trs = oracle.rank_layout(want["is_token_in_rank"], C)
    assert np.array_equal(cpm.cpu().numpy(), o_cpm.ravel()) and np.array_equal(trs.cpu().numpy(), o_trs.ravel())
    assert int(arr["status"][0]) == 0


BALANCED_FIELDS = ["z", "alloc", "alloc_cumsum", "experts_to_copy", "remote_stats", "rank_cu_seqlens",
                   "rank_zero_fill", "expert_offsets", "dst"]


@pytest.mark.parametrize("N,E,K,R,tp,B", [(3000, 64, 6, 8, 16, 4), (20000, 256, 8, 64, 128, 4), (50, 4, 2, 2, 1, 0)])
def test_balanced_writes_only_its_arrays(lib, N, E, K, R, tp, B):
    rng = np.random.default_rng(N + B)
    topk = workloads.random_topk(rng, N, E, K, hot=0.6)
    G = Guarded()
    arr, st = guarded_plan(lib, G, topk, E, R, 1)
    cap = int(N * K / R * 0.9)
    NvS = N * K + (E + B) * tp
    sizes = dict(z=R * R, alloc=R * E, alloc_cumsum=E * R, experts_to_copy=R * max(B, 1), remote_stats=2 * R,
                 rank_cu_seqlens=R * (E + B), rank_zero_fill=2 * R * (E + B), expert_offsets=R * E, dst=N * K)
    b = {k: G.alloc("balanced_" + k, sizes[k], torch.int32) for k in BALANCED_FIELDS}
    bst = lib.MoeBalancedPlanOut(*[b[k].data_ptr() for k in BALANCED_FIELDS])
    L = lib.load()
    t = torch.from_numpy(topk).cuda()
    lib.check("moe_plan_balanced", L.moe_plan_balanced(ctypes.byref(st), _p(t), N, E, K, R, tp, cap, B, NvS,
                                                       ctypes.byref(bst), _stream()))
    G.check()
    want = oracle.plan_balanced(topk, E, R, tp, cap, B, NvS)
    for k in BALANCED_FIELDS:
        got = b[k].cpu().numpy()
        if k == "experts_to_copy":
            got = got[: R * B]
        assert np.array_equal(got, want[k].ravel()), k
    assert int(arr["status"][0]) == 0
