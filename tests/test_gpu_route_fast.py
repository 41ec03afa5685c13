"""The router's approximate-key kernel against the exact one.

Sigmoid scores over groups of 32 experts, and renormalised softmax scores,
at E = 32 G take a kernel that selects by approximate keys (hardware
approximations of the sigmoid; the logit with 5 low bits replaced for
softmax) and proves the selection exact (margins of twice the keys' error
bound at the top-K and topk_group boundaries), falling back to the exact
kernel per token (by default from 16384 tokens on; MOE_ROUTE_PATH=fast
takes it at any size, as these tests do).  Its output must equal the exact kernel's bit
for bit, on ordinary rows and on rows built to fail each check (ties,
near-ties, a group holding most winners, non-finite logits, large biases),
and match the oracle.  The error bound it assumes is re-measured over every
fp32 input.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DELTA_SIGMA = 2.0 ** -20   # the bound the kernel's margins assume


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def test_sigmoid_approximation_within_half_the_assumed_bound(m):
    from expert_dispatch_planning_gb300 import _lib
    out = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    rc = _lib.load().moe_debug_route_sigmoid_error(_lib.ctypes.c_void_p(out.data_ptr()),
                                                   _lib.ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check("moe_debug_route_sigmoid_error", rc)
    err = float(out.item())
    assert 0.0 < err <= DELTA_SIGMA / 2, err


def route(m, logits, K, bias, monkeypatch, path, scoring="sigmoid", **kw):
    # "exact": the exact kernel; otherwise the fast one at any token count
    monkeypatch.setenv("MOE_ROUTE_PATH", "exact" if path == "exact" else "fast")
    lg = torch.from_numpy(logits).cuda()
    b = None if bias is None else torch.from_numpy(bias).cuda()
    idx, w = m.route_topk(lg, K, scoring=scoring, bias=b, **kw)
    torch.cuda.synchronize()
    monkeypatch.delenv("MOE_ROUTE_PATH", raising=False)
    return idx.cpu().numpy(), w.cpu().numpy()


def adversarial_rows(rng, N, E, G):
    """Rows that exercise every check of the fast kernel."""
    x = rng.standard_normal((N, E), dtype=np.float32)
    x[1::9] = np.round(x[1::9])                       # exact ties in keys
    x[2::9, :] = 0.25                                 # a row of equal keys
    x[3::9, : E // G] += 6.0                          # one group holds every winner
    r4 = x[4::9]
    r4[:, 7] = r4[:, 5]                               # duplicate value at a likely boundary
    x[5::9, 3] = np.inf                               # non-finite logits
    x[6::9, 5] = -np.inf
    x[0::97, 11] = np.nan
    x[7::9] *= 40.0                                   # sigmoid tails, tiny scores
    x[8::9] = -200.0 + rng.standard_normal((x[8::9].shape[0], E), dtype=np.float32)
    return x


SHAPES = [  # E, K, n_group, topk_group
    (128, 4, 4, 2), (128, 1, 1, 1), (128, 4, 4, 4),
    (256, 8, 8, 4), (256, 8, 8, 1), (256, 8, 8, 8), (256, 3, 8, 2), (256, 8, 1, 1), (256, 1, 8, 3),
    (512, 8, 16, 4), (512, 5, 1, 1)]


@pytest.mark.parametrize("E,K,ng,tg", SHAPES)
@pytest.mark.parametrize("bias_scale", [None, 0.1, 3.0])
def test_fast_equals_exact(m, monkeypatch, E, K, ng, tg, bias_scale):
    rng = np.random.default_rng(E * 7 + K * 3 + ng + tg)
    G = E // 32
    N = 1001
    x = adversarial_rows(rng, N, E, G)
    bias = None if bias_scale is None else rng.uniform(-bias_scale, bias_scale, E).astype(np.float32)
    kw = dict(renormalize=bool((E + K) % 2 == 0), n_group=ng, topk_group=tg, routed_scaling=2.5)
    fi, fw = route(m, x, K, bias, monkeypatch, "auto", **kw)
    ei, ew = route(m, x, K, bias, monkeypatch, "exact", **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))
    # and the oracle on the finite rows
    fin = np.isfinite(x).all(axis=1)
    o_idx, o_w = oracle.route_topk(x[fin], K, scoring=1, bias=bias, **kw)
    assert np.array_equal(fi[fin], o_idx)
    err = np.abs(fw[fin].astype(np.float64) - o_w)
    ok = (err <= 1e-6 * np.abs(o_w)) | ((np.abs(o_w) < 2.0 ** -126) & (err <= 2.0 ** -126))
    assert ok.all()


@pytest.mark.parametrize("bias_val", [1e25, np.inf, np.nan])
def test_fast_with_unusable_bias_routes_every_token_exactly(m, monkeypatch, bias_val):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((333, 256), dtype=np.float32)
    bias = rng.uniform(-0.1, 0.1, 256).astype(np.float32)
    bias[17] = bias_val
    kw = dict(renormalize=True, n_group=8, topk_group=4, routed_scaling=1.0)
    fi, fw = route(m, x, 8, bias, monkeypatch, "auto", **kw)
    ei, ew = route(m, x, 8, bias, monkeypatch, "exact", **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))


@pytest.mark.parametrize("E,scoring", [(256, "sigmoid"), (128, "softmax")])
def test_fast_every_token_failing_at_full_blocks(m, monkeypatch, E, scoring):
    """Enough tokens that every block of the fast kernel holds the most
    tokens its queue for the exact router takes, all of them failing a check
    (an unusable bias; an infinite logit in every softmax row): the queued
    tokens are routed exactly, identical to the exact kernel."""
    rng = np.random.default_rng(E)
    N = 700_000
    x = rng.standard_normal((N, E), dtype=np.float32)
    if scoring == "sigmoid":
        bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        bias[5] = np.inf
        kw = dict(renormalize=True, n_group=E // 32, topk_group=2, routed_scaling=2.5)
    else:
        bias = None
        x[np.arange(N), rng.integers(0, E, N)] = -np.inf
        kw = dict(renormalize=True, n_group=1, topk_group=1, routed_scaling=1.0)
    fi, fw = route(m, x, 8 if scoring == "softmax" else 4, bias, monkeypatch, "auto", scoring=scoring, **kw)
    ei, ew = route(m, x, 8 if scoring == "softmax" else 4, bias, monkeypatch, "exact", scoring=scoring, **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 17, 4097])
def test_fast_ragged_token_counts(m, monkeypatch, N):
    rng = np.random.default_rng(N)
    x = rng.standard_normal((N, 256), dtype=np.float32)
    bias = rng.uniform(-0.1, 0.1, 256).astype(np.float32)
    kw = dict(renormalize=True, n_group=8, topk_group=4, routed_scaling=2.5)
    fi, fw = route(m, x, 8, bias, monkeypatch, "auto", **kw)
    o_idx, o_w = oracle.route_topk(x, 8, scoring=1, bias=bias, **kw)
    assert np.array_equal(fi, o_idx)
    assert np.all(np.abs(fw - o_w) <= 1e-6 * np.abs(o_w))


def test_fast_near_ties_at_the_boundary(m, monkeypatch):
    """Keys that differ by a few ulps at the 8th/9th place and at the group
    boundary: the checks must send these tokens to the exact kernel."""
    rng = np.random.default_rng(11)
    N, E = 512, 256
    x = rng.standard_normal((N, E), dtype=np.float32) - 3.0
    bias = np.zeros(E, np.float32)
    for s in range(N):
        base = np.float32(1.0 + rng.standard_normal() * 0.1)
        experts = rng.choice(E, 10, replace=False)
        x[s, experts] = base
        steps = rng.integers(0, 4, size=10)
        for e, st in zip(experts, steps):
            v = base
            for _ in range(int(st)):
                v = np.nextafter(v, np.float32(np.inf))
            x[s, e] = v
    kw = dict(renormalize=True, n_group=8, topk_group=4, routed_scaling=1.0)
    fi, fw = route(m, x, 8, bias, monkeypatch, "auto", **kw)
    ei, ew = route(m, x, 8, bias, monkeypatch, "exact", **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))
    o_idx, _ = oracle.route_topk(x, 8, scoring=1, bias=bias, **kw)
    assert np.array_equal(fi, o_idx)


SOFTMAX_SHAPES = [(128, 8), (128, 1), (128, 5), (256, 8), (256, 2), (512, 8), (512, 3)]


@pytest.mark.parametrize("E,K", SOFTMAX_SHAPES)
@pytest.mark.parametrize("scale", [1.0, 1e-3, 300.0])
def test_fast_softmax_equals_exact(m, monkeypatch, E, K, scale):
    rng = np.random.default_rng(E * 13 + K)
    G = E // 32
    x = adversarial_rows(rng, 1001, E, G)
    x[7::9] = x[7::9] * np.float32(scale)
    kw = dict(renormalize=True, n_group=1, topk_group=1, routed_scaling=1.5)
    fi, fw = route(m, x, K, None, monkeypatch, "auto", scoring="softmax", **kw)
    ei, ew = route(m, x, K, None, monkeypatch, "exact", scoring="softmax", **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))
    fin = np.isfinite(x).all(axis=1)
    o_idx, o_w = oracle.route_topk(x[fin], K, scoring=0, **kw)
    assert np.array_equal(fi[fin], o_idx)
    err = np.abs(fw[fin].astype(np.float64) - o_w)
    ok = (err <= 1e-6 * np.abs(o_w)) | ((np.abs(o_w) < 2.0 ** -126) & (err <= 2.0 ** -126))
    assert ok.all()


def test_fast_softmax_near_ties_inside_the_top_k(m, monkeypatch):
    """Winners a few ulps apart (their order decided by the exact keys) and
    logits that differ only in the packed low bits."""
    rng = np.random.default_rng(12)
    N, E = 700, 128
    x = rng.standard_normal((N, E), dtype=np.float32) - 4.0
    for s in range(N):
        base = np.float32(rng.choice([0.5, 1.0, 3.0, -0.75]))
        experts = rng.choice(E, 12, replace=False)
        for i, e in enumerate(experts):
            v = base
            for _ in range(int(rng.integers(0, 40))):
                v = np.nextafter(v, np.float32(np.inf))
            x[s, e] = v
    kw = dict(renormalize=True, n_group=1, topk_group=1, routed_scaling=1.0)
    fi, fw = route(m, x, 8, None, monkeypatch, "auto", scoring="softmax", **kw)
    ei, ew = route(m, x, 8, None, monkeypatch, "exact", scoring="softmax", **kw)
    assert np.array_equal(fi, ei)
    assert np.array_equal(fw.view(np.uint32), ew.view(np.uint32))
    o_idx, _ = oracle.route_topk(x, 8, scoring=0, **kw)
    assert np.array_equal(fi, o_idx)
