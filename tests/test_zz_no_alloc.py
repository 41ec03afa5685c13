"""moe_plan_no_alloc against the oracle and against moe_plan, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory (a host framework owns every buffer, or cudaMalloc's device-wide
synchronisation is not acceptable): its scratch is a fixed array inside the
library.  Its plan must equal the oracle's plan and the one moe_plan builds
with a caller workspace, on consecutive calls of different sizes and plan
paths that all share that array.  This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

FIELDS = ["tokens_per_expert", "cu_seqlens", "zero_fill_ranges", "pairs_per_rank", "tokens_per_rank",
          "rank_prefix", "rank_slot_offsets", "is_token_in_rank", "dst", "src_of_slot", "dup_counts"]


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import expert_dispatch_planning_gb300 as mod
    mod.load()
    return mod


def _call_no_alloc(m, topk, p):
    from expert_dispatch_planning_gb300 import _lib
    N, K = topk.shape
    rc = _lib.load().moe_plan_no_alloc(
        ctypes.c_void_p(topk.data_ptr()), N, p.E, K, p.R, p.alignment, ctypes.byref(p.c_struct),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check("moe_plan_no_alloc", rc)


def _same(a, b):
    ha, hb = a.to_host(), b.to_host()
    for k in FIELDS + ["dup_groups", "dup_loffs"]:
        assert np.array_equal(np.asarray(ha[k]), np.asarray(hb[k])), k


def _same_as_oracle(p, topk, E, R, a):
    got, want = p.to_host(), oracle.plan(topk, E, R, a)
    for k in FIELDS + ["dup_groups", "dup_loffs"]:
        assert np.array_equal(np.asarray(got[k]), np.asarray(want[k])), k


def _check(m, w_or_shape, rng, path=None, monkeypatch=None):
    N, E, K, R, a = w_or_shape
    if path is not None:
        monkeypatch.setenv("MOE_PLAN_PATH", path)
    topk_np = workloads.random_topk(rng, N, E, K)
    topk = torch.from_numpy(topk_np).to("cuda")
    ref = m.plan(topk, E, R, a)
    got = m.Plan.allocate(N, E, K, R, a)
    _call_no_alloc(m, topk, got)
    assert m.get_status(got) == 0 and m.get_status(ref) == 0
    _same_as_oracle(got, topk_np, E, R, a)
    _same(got, ref)
    if path is not None:
        monkeypatch.delenv("MOE_PLAN_PATH")


def _shape(name):
    w = workloads.get(name)
    return (w.N, w.E, w.K, w.R, w.alignment)


@pytest.mark.parametrize("name", ["qwen3", "large"])
def test_no_alloc_matches_oracle_and_workspace_plan_on_consecutive_calls(m, name):
    rng = np.random.default_rng(11)
    for _ in range(2):
        _check(m, _shape(name), rng)


def test_no_alloc_across_sizes_and_paths_sharing_the_array(m, monkeypatch):
    """One process, one shared array: the large look-back plan, smaller plans
    on the look-back and grid paths (the array's flags and counters left by
    a bigger call), then the large plan again."""
    rng = np.random.default_rng(12)
    large = _shape("large")
    _check(m, large, rng)
    _check(m, (20000, 64, 8, 8, 16), rng, "lookback", monkeypatch)
    _check(m, (4096, 256, 8, 64, 128), rng, "grid", monkeypatch)
    _check(m, (777, 16, 3, 4, 8), rng, "lookback", monkeypatch)
    _check(m, (8192, 128, 8, 8, 128), rng)          # the medium-E cluster kernel (no scratch)
    _check(m, large, rng)


def test_no_alloc_rejects_sizes_beyond_its_scratch(m):
    from expert_dispatch_planning_gb300 import _lib
    lib = _lib.load()
    N, E, K, R = 1 << 20, 1024, 8, 128        # workspace far above 1 MiB
    assert lib.moe_plan_workspace_size(N, E, K, R) > (1 << 20)
    p = m.Plan.allocate(8, E, K, R, 1)        # never written: the size check fails first
    rc = lib.moe_plan_no_alloc(ctypes.c_void_p(16), N, E, K, R, 1, ctypes.byref(p.c_struct),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.MOE_ERR_CAPACITY
