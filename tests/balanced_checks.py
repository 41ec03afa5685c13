"""Properties of a capacity-balanced plan (MoonEP's rank-0 planning in its
single-source form) that hold at any size; shared by the oracle pins and the
GPU parity tests."""
import numpy as np


def check_balanced_invariants(o, topk, E, R, tp, cap, B, NvS):
    topk = np.asarray(topk, np.int64)
    N, K = topk.shape
    epn = E // R
    count = np.bincount(topk.ravel(), minlength=E)
    owner = np.arange(E) // epn
    z = np.asarray(o["z"], np.int64)
    alloc = np.asarray(o["alloc"], np.int64)
    # balancing leaves no rank above CAP while another is below it
    group = count.reshape(R, epn).sum(1)
    bal = group - cap - z.sum(1) + z.sum(0)
    assert not (np.any(bal > 0) and np.any(bal < 0))
    assert np.all(np.diag(z) == 0) and np.all(z >= 0)
    # allocations: every pair somewhere, moved only along z, within the quota
    assert np.all(alloc >= 0) and np.array_equal(alloc.sum(0), count)
    for o_r in range(R):
        for r in range(R):
            if r == o_r:
                continue
            moved = alloc[r, o_r * epn:(o_r + 1) * epn].sum()
            assert moved <= z[o_r, r]
    assert np.array_equal(np.asarray(o["alloc_cumsum"], np.int64), np.cumsum(alloc, 0).T)
    # redundant experts: remote, distinct, by count (ties to the larger index)
    etc = np.asarray(o["experts_to_copy"], np.int64).reshape(R, B)
    stats = np.asarray(o["remote_stats"], np.int64)
    picks_per_owner = np.zeros(R, np.int64)
    for d in range(R):
        remote = np.where(owner == d, 0, alloc[d])
        assert stats[d, 0] == (remote > 0).sum()
        real = [int(e) for e in etc[d] if e >= 0]
        assert etc[d].tolist() == real + [-1] * (B - len(real))
        assert len(set(real)) == len(real) and all(owner[e] != d and alloc[d, e] > 0 for e in real)
        order = sorted(range(E), key=lambda e: (-remote[e], -e))
        assert real == [e for e in order[:B] if remote[e] > 0]
        for e in real:
            picks_per_owner[owner[e]] += 1
    assert np.array_equal(stats[:, 1], picks_per_owner)
    # per-rank groups
    cu = np.asarray(o["rank_cu_seqlens"], np.int64).reshape(R, E + B)
    zf = np.asarray(o["rank_zero_fill"], np.int64).reshape(R, E + B, 2)
    eo = np.asarray(o["expert_offsets"], np.int64).reshape(R, E)
    for d in range(R):
        picked = set(int(e) for e in etc[d] if e >= 0)
        cnt = [0 if g in picked else alloc[d, g] for g in range(E)]
        cnt += [alloc[d, etc[d, s]] if etc[d, s] >= 0 else 0 for s in range(B)]
        start = np.concatenate([[0], cu[d, :-1]])
        padded = cu[d] - start
        assert np.all(padded >= 0) and np.all(padded % tp == 0) and cu[d, -1] <= NvS
        for g in range(E + B):
            c = cnt[g]
            assert (padded[g] == 0) == (c == 0) and padded[g] - c < tp
            if padded[g] > c and c > 0:
                assert zf[d, g].tolist() == [start[g] + c, padded[g] - c]
            else:
                assert zf[d, g].tolist() == [0, 0]
            if c > 0:
                e = g if g < E else int(etc[d, g - E])
                assert eo[d, e] == start[g]
    # dst: rank-strided rows, each in its expert's group on its rank, unique,
    # ascending flat order within (expert, rank), counts equal to alloc
    dst = np.asarray(o["dst"], np.int64).reshape(N, K)
    raw = np.where(dst >= 0, dst, -dst - 1)
    rank = raw // NvS
    loff = raw % NvS
    assert np.unique(raw).size == raw.size
    got = np.zeros((R, E), np.int64)
    last = {}
    for f in range(N * K):
        s, k = divmod(f, K)
        e, r, l = int(topk[s, k]), int(rank[s, k]), int(loff[s, k])
        assert eo[r, e] <= l < eo[r, e] + alloc[r, e]
        assert last.get((e, r), -1) < l
        last[(e, r)] = l
        got[r, e] += 1
    assert np.array_equal(got, alloc)
    earlier = np.zeros((N, K), bool)
    for k in range(1, K):
        earlier[:, k] = np.any(rank[:, :k] == rank[:, k:k + 1], axis=1)
    assert np.array_equal(dst < 0, earlier)
