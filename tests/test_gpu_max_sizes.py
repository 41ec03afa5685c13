"""Routing, plans and rows at the largest sizes the host accepts.

The oracle cannot plan at these sizes, so the plan checks are properties
that determine the plan at any size, evaluated with torch on the device in
chunks: exact per-expert counts, aligned cu_seqlens, a bijection between
pairs and non-padding slots, ascending flat index within every expert (the
canonical order), the duplicate rule per (token, rank), the rank matrices
and the dedup totals.  The rows: every slot holds its token's row, every
padding row is zero, rows from P on are untouched, and sampled tokens of the
combine equal the oracle's combine of their gathered rows.  Routing is per
token, so sampled rows are compared with the oracle directly.  Inputs are
seeded random values drawn on the device.  Peak device memory: about 55 GB.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def device_topk(N, E, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, E, (N, K), generator=g, device="cuda", dtype=torch.int32)


def raw_of(dst):
    return torch.where(dst < 0, -dst - 1, dst)


def check_plan_properties(p, topk, E, R, a):
    """Returns P.  Every check runs over chunks of pairs, slots or tokens."""
    N, K = topk.shape
    epn = E // R
    flat = topk.reshape(-1)
    NK = flat.numel()
    counts = torch.bincount(flat, minlength=E).to(torch.int32)
    assert torch.equal(p.tokens_per_expert, counts)
    padded = torch.where(counts > 0, (counts + a - 1) // a * a, torch.zeros_like(counts))
    cu = torch.zeros(E + 1, dtype=torch.int64, device="cuda")
    cu[1:] = torch.cumsum(padded.to(torch.int64), 0)
    assert torch.equal(p.cu_seqlens.to(torch.int64), cu)
    P = int(cu[-1])
    zf_start = torch.where(padded > counts, cu[:-1].to(torch.int32) + counts, torch.zeros_like(counts))
    assert torch.equal(p.zero_fill_ranges[:, 0], zf_start)
    assert torch.equal(p.zero_fill_ranges[:, 1], padded - counts)

    dst = p.dst.reshape(-1)
    src = p.src_of_slot
    assert int((src >= 0).sum()) == NK                       # one source per non-padding slot ...
    assert bool((src[P:] == -1).all())
    for f0 in range(0, NK, CHUNK):                           # ... and it is the pair whose slot it is
        f1 = min(NK, f0 + CHUNK)
        raw = raw_of(dst[f0:f1]).to(torch.int64)
        assert torch.equal(src[raw], torch.arange(f0, f1, dtype=torch.int32, device="cuda"))
        e = flat[f0:f1].to(torch.int64)
        assert bool(((raw >= cu[e]) & (raw < cu[e] + counts[e])).all())
    # canonical order: inside every expert's rows the flat index ascends
    for j0 in range(0, P - 1, CHUNK):
        j1 = min(P, j0 + CHUNK + 1)
        s = src[j0:j1]
        real = s >= 0
        e_slot = flat[s.clamp(min=0).to(torch.int64)]
        same = real[:-1] & real[1:] & (e_slot[:-1] == e_slot[1:])
        assert bool((s[1:][same] > s[:-1][same]).all())

    # duplicates (an earlier k of the same token on the same rank), rank
    # matrices and (token, rank) group sizes, over chunks of tokens
    tpr = torch.zeros(R, dtype=torch.int64, device="cuda")
    n_groups = n_dup = 0
    for s0 in range(0, N, CHUNK // K):
        s1 = min(N, s0 + CHUNK // K)
        ranks = (topk[s0:s1] // epn).to(torch.int64)
        dup = torch.zeros_like(ranks, dtype=torch.bool)
        for k in range(1, K):
            dup[:, k] = (ranks[:, :k] == ranks[:, k:k + 1]).any(1)
        assert torch.equal(p.dst[s0:s1] < 0, dup)
        n_dup += int(dup.sum())
        itr = torch.zeros((s1 - s0, R), dtype=torch.uint8, device="cuda").scatter_(1, ranks, 1)
        assert torch.equal(p.is_token_in_rank[s0:s1], itr)
        tpr += itr.sum(0, dtype=torch.int64)
        per = torch.zeros((s1 - s0, R), dtype=torch.int32, device="cuda").scatter_add_(
            1, ranks, torch.ones_like(ranks, dtype=torch.int32))
        n_groups += int((per >= 2).sum())
    assert torch.equal(p.tokens_per_rank.to(torch.int64), tpr)
    assert torch.equal(p.pairs_per_rank.to(torch.int64), counts.to(torch.int64).reshape(R, epn).sum(1))
    rp = torch.zeros(R + 1, dtype=torch.int64, device="cuda")
    rp[1:] = torch.cumsum(tpr, 0)
    assert torch.equal(p.rank_prefix.to(torch.int64), rp)
    assert torch.equal(p.rank_slot_offsets.to(torch.int64), cu[torch.arange(R + 1, device="cuda") * epn])
    # dedup totals; every duplicate's slot listed once in dup_loffs
    assert p.dup_counts.tolist() == [n_groups, n_dup]
    assert int(p.dup_groups[:n_groups, 2].sum(dtype=torch.int64)) == n_dup
    dups = raw_of(dst[dst < 0])
    assert torch.equal(torch.sort(p.dup_loffs[:n_dup])[0], torch.sort(dups)[0])
    return P


def test_plan_at_the_pair_limit(m):
    """N*K = 2^30 - 64 (the host accepts N*K < 2^30): the two-launch
    look-back plan over 131072 tiles, slots near 2^30."""
    K, E, R, a = 8, 256, 8, 128
    N = ((1 << 30) - 64) // K
    assert m.plan_launches(N, E, K, R) == 2
    topk = device_topk(N, E, K, seed=3)
    p = m.plan(topk, E, R, a)
    assert m.get_status(p) == 0
    P = check_plan_properties(p, topk, E, R, a)
    assert P >= N * K


def test_rows_with_a_permuted_buffer_above_2_30_rows(m):
    """Alignment 2^20 over 1024 experts: about 2^30 rows of 16 bytes (row
    offsets beyond 2^31 elements), almost all of them padding that the
    permute zeroes; the combine gathers from the far end of the buffer."""
    N, E, K, R, a, H = 4096, 1024, 2, 8, 1 << 20, 8
    topk = device_topk(N, E, K, seed=4)
    p = m.plan(topk, E, R, a)
    assert m.get_status(p) == 0
    P = check_plan_properties(p, topk, E, R, a)
    assert P > (1 << 29) and P * H > (1 << 31) and p.P_cap < (1 << 31)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    perm = torch.full((p.P_cap, H), 3.0, dtype=torch.bfloat16, device="cuda")
    m.permute(x, p, out=perm)
    raw = raw_of(p.dst).reshape(-1).to(torch.int64)
    xi, pi = x.view(torch.int16), perm.view(torch.int16)
    rows = xi.repeat_interleave(K, 0)
    assert torch.equal(pi[raw], rows)
    # every other row below P is padding (+0.0); rows from P on are untouched
    pi[raw] = 0
    for c0 in range(0, P, CHUNK):
        assert int(torch.count_nonzero(pi[c0:min(P, c0 + CHUNK)])) == 0
    three = int(torch.tensor([3.0], dtype=torch.bfloat16).view(torch.int16).item())
    assert bool((pi[P:] == three).all())
    pi[raw] = rows

    w = torch.rand((N, K), generator=g, device="cuda")
    out = m.combine(perm, w, p)
    assert m.get_status(p) == 0
    # sampled tokens against the oracle: their rows gathered, slots renumbered
    tok = np.random.default_rng(6).choice(N, 256, replace=False)
    t = torch.from_numpy(tok).cuda()
    y_small = pi[raw.reshape(N, K)[t].reshape(-1)].cpu().numpy().view(np.uint16)
    d_small = np.arange(256 * K, dtype=np.int32).reshape(256, K)
    want = oracle.combine(y_small, w[t].cpu().numpy(), d_small)
    assert np.array_equal(out.view(torch.int16)[t].cpu().numpy().view(np.uint16), want)


@pytest.mark.parametrize("N,E,K,scoring,ng,tg,path", [
    ((1 << 30) - 7, 8, 2, 0, 1, 1, "auto"),       # N*K just under 2^31; logits 34 GB
    ((1 << 24) + 5, 256, 8, 1, 8, 4, "auto"),     # N*E above 2^32 elements; the approximate-key kernel
    ((1 << 24) + 5, 256, 8, 1, 8, 4, "exact")])
def test_route_at_the_limits(m, monkeypatch, N, E, K, scoring, ng, tg, path):
    """Routing is per token, so sampled rows (and the last ones) are compared
    with the oracle exactly: indices bit for bit, weights within 1e-6."""
    monkeypatch.setenv("MOE_ROUTE_PATH", path)
    g = torch.Generator(device="cuda")
    g.manual_seed(N % 1000)
    logits = torch.randn((N, E), generator=g, device="cuda")
    bias = None
    if scoring == 1:
        bias = torch.from_numpy(np.random.default_rng(7).uniform(-0.1, 0.1, E).astype(np.float32)).cuda()
    idx, w = m.route_topk(logits, K, scoring=scoring, renormalize=True, bias=bias, n_group=ng, topk_group=tg,
                          routed_scaling=2.5)
    rows = np.concatenate([np.random.default_rng(8).choice(N, 4096, replace=False), np.arange(N - 64, N)])
    t = torch.from_numpy(rows).cuda()
    o_idx, o_w = oracle.route_topk(logits[t].cpu().numpy(), K, scoring=scoring, renormalize=True,
                                   bias=None if bias is None else bias.cpu().numpy(), n_group=ng, topk_group=tg,
                                   routed_scaling=2.5)
    assert np.array_equal(idx[t].cpu().numpy(), o_idx)
    err = np.abs(w[t].cpu().numpy().astype(np.float64) - o_w)
    assert (err <= 1e-6 * np.abs(o_w) + 2.0 ** -126).all()
