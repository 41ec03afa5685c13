"""Pins for the oracle's row movement: permute and weighted combine.

Permute: the gather-back identity, zero padding rows, untouched capacity
rows.  Combine: one-hot weights reproduce rows exactly, zero weights give
+0, and on random inputs the fp32-accumulated, bf16-rounded result lies
within the rounding bound of the exact (fp64) weighted sum.
"""
import numpy as np
import torch

import oracle
import workloads


def bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _plan_case(seed, N=300, E=16, K=4, R=4, a=8, H=40):
    rng = np.random.default_rng(seed)
    topk = workloads.random_topk(rng, N, E, K)
    p = oracle.plan(topk, E, R, a)
    x = workloads.make_x_bits(rng, N, H)
    return rng, topk, p, x


def test_permute_gather_identity_and_padding():
    rng, topk, p, x = _plan_case(30)
    N, K = topk.shape
    H = x.shape[1]
    sentinel = np.full((p["P_cap"], H), 0xBEEF, np.uint16)
    out = oracle.permute(x, p["dst"], p["zero_fill_ranges"], K, p["P_cap"], fill=sentinel)
    raw = np.abs(p["dst"].astype(np.int64) + (p["dst"] < 0)).ravel()   # -raw-1 -> raw
    assert np.array_equal(out[raw], np.repeat(x, K, axis=0))
    pad_rows = [r for e in range(p["zero_fill_ranges"].shape[0])
                for r in range(p["zero_fill_ranges"][e, 0],
                               p["zero_fill_ranges"][e, 0] + p["zero_fill_ranges"][e, 1])]
    assert np.all(out[pad_rows] == 0)
    written = np.zeros(p["P_cap"], bool)
    written[raw] = True
    written[pad_rows] = True
    assert np.all(written[: p["P"]])          # every row below P is defined
    assert np.all(out[p["P"]:] == 0xBEEF)      # capacity rows untouched
    # src_of_slot gathers the permuted rows back
    src = p["src_of_slot"]
    rows = np.nonzero(src >= 0)[0]
    assert np.array_equal(out[rows], x[src[rows] // K])


def test_combine_one_hot_and_zero_weights():
    rng, topk, p, x = _plan_case(31)
    N, K = topk.shape
    y = oracle.permute(x, p["dst"], p["zero_fill_ranges"], K, p["P_cap"])
    for k in range(K):
        w = np.zeros((N, K), np.float32)
        w[:, k] = 1.0
        assert np.array_equal(oracle.combine(y, w, p["dst"]), x)
    out = oracle.combine(y, np.zeros((N, K), np.float32), p["dst"])
    assert np.all(out == 0)


def test_combine_within_rounding_bound_of_exact_sum():
    rng, topk, p, x = _plan_case(32, N=400, K=8, E=32, R=8, H=64)
    N, K = topk.shape
    H = x.shape[1]
    y = workloads.make_x_bits(rng, p["P_cap"], H)        # arbitrary expert outputs
    w = (rng.random((N, K)) * 2.5 / K).astype(np.float32)
    out = bf16_to_f64(oracle.combine(y, w, p["dst"]))
    raw = np.where(p["dst"] >= 0, p["dst"], -p["dst"] - 1).astype(np.int64)
    yv = bf16_to_f64(y)[raw]                              # [N,K,H]
    terms = w.astype(np.float64)[:, :, None] * yv
    exact = terms.sum(1)
    # K fused multiply-adds in fp32: each rounds once (<= 2^-24 of the
    # running magnitude, itself <= sum |terms|); then one bf16 rounding
    # (<= 2^-8 relative: half an ulp of an 8-bit significand).
    acc_err = K * 2.0 ** -24 * np.abs(terms).sum(1)
    bound = acc_err + 2.0 ** -8 * (np.abs(exact) + acc_err) + 1e-30
    assert np.all(np.abs(out - exact) <= bound)
    # and the k-order matters only through rounding: a permuted k order
    # stays within twice the bound
    perm = rng.permutation(K)
    out2 = bf16_to_f64(oracle.combine(y, w[:, perm], p["dst"][:, perm]))
    assert np.all(np.abs(out2 - exact) <= 2 * bound)


def test_combine_rows_matches_full_combine():
    rng, topk, p, x = _plan_case(33)
    N, K = topk.shape
    y = oracle.permute(x, p["dst"], p["zero_fill_ranges"], K, p["P_cap"])
    w = rng.random((N, K)).astype(np.float32)
    full = oracle.combine(y, w, p["dst"])
    toks = rng.choice(N, 25, replace=False)
    assert np.array_equal(oracle.combine_rows(y, w, p["dst"], toks), full[toks])
