"""Definition-level checks of a dispatch plan, shared by the oracle pins and
the GPU parity tests.

``definition_plan`` restates each plan output as a counting definition
(O((N*K)^2) on purpose: slot(f) counts earlier pairs of the same expert;
a pair is a duplicate when an earlier k of its token hit the same rank),
independent of the oracle's running counters.  ``check_plan_invariants``
tests properties that hold at any size.
"""
import numpy as np


def definition_plan(topk, E, R, a):
    topk = np.asarray(topk)
    N, K = topk.shape
    epn = E // R
    flat = topk.reshape(-1).tolist()
    NK = len(flat)
    count = [sum(1 for v in flat if v == e) for e in range(E)]
    padded = [(-(-c // a)) * a if c > 0 else 0 for c in count]
    cu = [sum(padded[:e]) for e in range(E + 1)]
    zfr = [[cu[e] + count[e], padded[e] - count[e]] if padded[e] > count[e] else [0, 0]
           for e in range(E)]
    raw = [cu[flat[f]] + sum(1 for g in range(f) if flat[g] == flat[f]) for f in range(NK)]
    dup = []
    for f in range(NK):
        s, k = divmod(f, K)
        r = flat[f] // epn
        dup.append(any(flat[s * K + j] // epn == r for j in range(k)))
    dst = [-raw[f] - 1 if dup[f] else raw[f] for f in range(NK)]
    cap = NK + E * (a - 1)
    src = [-1] * cap
    for f in range(NK):
        src[raw[f]] = f
    itr = [[int(any(flat[s * K + k] // epn == r for k in range(K))) for r in range(R)]
           for s in range(N)]
    tpr = [sum(itr[s][r] for s in range(N)) for r in range(R)]
    ppr = [sum(count[r * epn:(r + 1) * epn]) for r in range(R)]
    rank_prefix = [sum(tpr[:r]) for r in range(R + 1)]
    rso = [cu[r * epn] for r in range(R + 1)]
    groups, loffs = [], []
    for s in range(N):
        for k in range(K):
            f = s * K + k
            if dup[f]:
                continue
            r = flat[f] // epn
            later = [s * K + j for j in range(k + 1, K) if flat[s * K + j] // epn == r]
            if later:
                groups.append([raw[f], len(loffs), len(later)])
                loffs.extend(raw[g] for g in later)
    return dict(
        tokens_per_expert=count, cu_seqlens=cu, zero_fill_ranges=zfr,
        dst=np.array(dst).reshape(N, K).tolist(), src_of_slot=src,
        is_token_in_rank=itr, tokens_per_rank=tpr, pairs_per_rank=ppr,
        rank_prefix=rank_prefix, rank_slot_offsets=rso,
        dup_groups=groups, dup_loffs=loffs, dup_counts=[len(groups), len(loffs)])


def check_plan_invariants(p, topk, E, R, a):
    """Properties any correct plan satisfies (works at full size)."""
    topk = np.asarray(topk, dtype=np.int64)
    N, K = topk.shape
    epn = E // R
    counts = np.asarray(p["tokens_per_expert"], np.int64)
    cu = np.asarray(p["cu_seqlens"], np.int64)
    assert counts.sum() == N * K
    assert np.array_equal(counts, np.bincount(topk.ravel(), minlength=E))
    steps = np.diff(cu)
    assert cu[0] == 0 and np.all(steps >= counts) and np.all(steps % a == 0)
    assert np.all((steps == 0) == (counts == 0)) and np.all(steps - counts < a)
    dst = np.asarray(p["dst"], np.int64).reshape(N, K)
    raw = np.where(dst >= 0, dst, -dst - 1)
    # each pair's slot lies inside its expert's row range
    e = topk
    assert np.all(raw >= cu[e]) and np.all(raw < cu[e] + counts[e])
    # slots are unique, ascending in f within each expert
    flat_raw = raw.ravel()
    assert np.unique(flat_raw).size == flat_raw.size
    order = np.lexsort((np.arange(N * K), topk.ravel()))
    rs = flat_raw[order]
    same = topk.ravel()[order][1:] == topk.ravel()[order][:-1]
    assert np.all(rs[1:][same] == rs[:-1][same] + 1)
    # src_of_slot is the inverse map; every other row -1
    src = np.asarray(p["src_of_slot"], np.int64)
    assert src.size >= N * K + E * (a - 1)
    assert np.array_equal(src[flat_raw], np.arange(N * K))
    mask = np.ones(src.size, bool)
    mask[flat_raw] = False
    assert np.all(src[mask] == -1)
    # zero-fill ranges cover exactly the padding rows of each expert
    z = np.asarray(p["zero_fill_ranges"], np.int64).reshape(E, 2)
    pad = steps - counts
    assert np.all(z[:, 1] == pad)
    assert np.all(z[pad > 0, 0] == cu[:-1][pad > 0] + counts[pad > 0])
    assert np.all(z[pad == 0] == 0)
    # duplicates: negative exactly when an earlier k of the token hit the rank
    rank = topk // epn
    earlier = np.zeros((N, K), bool)
    for k in range(1, K):
        earlier[:, k] = np.any(rank[:, :k] == rank[:, k:k + 1], axis=1)
    assert np.array_equal(dst < 0, earlier)
    itr = np.asarray(p["is_token_in_rank"], np.int64).reshape(N, R)
    want_itr = np.zeros((N, R), np.int64)
    np.put_along_axis(want_itr, rank, 1, axis=1)
    assert np.array_equal(itr, want_itr)
    tpr = np.asarray(p["tokens_per_rank"], np.int64)
    assert np.array_equal(tpr, itr.sum(0))
    assert np.array_equal(np.asarray(p["rank_prefix"], np.int64), np.concatenate([[0], np.cumsum(tpr)]))
    assert np.array_equal(np.asarray(p["pairs_per_rank"], np.int64), counts.reshape(R, epn).sum(1))
    assert np.array_equal(np.asarray(p["rank_slot_offsets"], np.int64), cu[::epn])
    # dedup structures: every duplicate slot appears once, in the group whose
    # primary is its token's primary on the same rank
    dc = np.asarray(p["dup_counts"], np.int64)
    groups = np.asarray(p["dup_groups"], np.int64).reshape(-1, 3)[: dc[0]]
    loffs = np.asarray(p["dup_loffs"], np.int64)[: dc[1]]
    n_dup = int((dst < 0).sum())
    assert dc[1] == n_dup and loffs.size == n_dup
    assert np.array_equal(np.sort(loffs), np.sort(raw[dst < 0]))
    slot_owner = {}
    for s in range(N):
        for k in range(K):
            slot_owner[int(raw[s, k])] = (s, k)
    prim_of = {}
    for s in range(N):
        for k in range(K):
            if dst[s, k] >= 0:
                prim_of[(s, int(rank[s, k]))] = int(raw[s, k])
    assert groups.shape[0] == sum(1 for (s, r) in prim_of if (rank[s] == r).sum() >= 2)
    nxt = 0
    last_key = None
    for g in range(groups.shape[0]):
        prim, begin, cnt = (int(v) for v in groups[g])
        s, k = slot_owner[prim]
        assert dst[s, k] >= 0
        assert (s, k) > last_key if last_key else True
        last_key = (s, k)
        assert begin == nxt and cnt >= 1
        nxt += cnt
        ks = []
        for j in range(begin, begin + cnt):
            s2, k2 = slot_owner[int(loffs[j])]
            assert s2 == s and rank[s2, k2] == rank[s, k] and dst[s2, k2] < 0
            ks.append(k2)
        assert ks == sorted(ks) and ks[0] > k
    assert nxt == n_dup
