"""moe_plan_no_alloc against moe_plan, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory (a host framework owns every buffer, or cudaMalloc's device-wide
synchronisation is not acceptable): its scratch is a fixed array inside the
library.  Its plan must equal the one moe_plan builds with a caller
workspace, on consecutive calls that share that array.  This file is
collected last so that a stop-at-first-failure run has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("name", ["qwen3", "large"])
def test_no_alloc_matches_workspace_plan_on_consecutive_calls(m, name):
    w = workloads.get(name)
    rng = np.random.default_rng(11)
    for call in range(2):
        topk = torch.from_numpy(workloads.random_topk(rng, w.N, w.E, w.K)).to("cuda")
        ref = m.plan(topk, w.E, w.R, w.alignment)
        got = m.Plan.allocate(w.N, w.E, w.K, w.R, w.alignment)
        _call_no_alloc(m, topk, got)
        assert m.get_status(got) == 0 and m.get_status(ref) == 0
        _same(got, ref)


def test_no_alloc_rejects_sizes_beyond_its_scratch(m):
    from expert_dispatch_planning_gb300 import _lib
    lib = _lib.load()
    N, E, K, R = 1 << 20, 1024, 8, 128        # workspace far above 1 MiB
    assert lib.moe_plan_workspace_size(N, E, K, R) > (1 << 20)
    p = m.Plan.allocate(8, E, K, R, 1)        # never written: the size check fails first
    rc = lib.moe_plan_no_alloc(ctypes.c_void_p(16), N, E, K, R, 1, ctypes.byref(p.c_struct),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.MOE_ERR_CAPACITY
