"""moe_plan_noalloc, the route-metadata call for callers that cannot allocate device memory.

Such callers -- a runtime that forbids cudaMalloc on its execution path, or a plugin host
that hands an operator only its inputs and outputs -- get no workspace to pass to moe_plan.
moe_plan_noalloc keeps its scratch in a fixed device array inside the library instead. These
tests call it through the C ABI and require the same plan as moe_plan (counts and offsets
bit-exact, each expert's rows the same set of (token, slot) identities), on two calls in a
row so that the second call cannot lean on anything the first one left in the shared array.
"""
import numpy as np
import pytest
import torch

from gpu_util import lib
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    return lib()


def _plan_with_workspace(moe, ids, d, E, rows=None, expect_error=0):
    """moe_plan's outputs; E and rows count the shared experts and their slots when d has any."""
    rows = ids.numel() if rows is None else rows
    ws = moe.alloc_workspace(d, "a16w16", DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_src = torch.empty(max(rows, 1), dtype=torch.int32, device=DEV)
    moe.moe_plan(ids, d, ws, counts, offsets, row_src)
    assert moe.moe_check_device_error(ws) == expect_error
    return counts.cpu().numpy(), offsets.cpu().numpy(), row_src.cpu().numpy()


def _plan_without_workspace(moe, ids, d, E, rows=None):
    rows = ids.numel() if rows is None else rows
    # poison the outputs so that anything the call leaves unwritten shows up
    counts = torch.full((E,), -5, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -5, dtype=torch.int32, device=DEV)
    row_src = torch.full((max(rows, 1),), -5, dtype=torch.int32, device=DEV)
    moe.moe_plan_noalloc(ids, d, counts, offsets, row_src)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), row_src.cpu().numpy()


def _same_plan(a, b, E):
    ca, oa, ra = a
    cb, ob, rb = b
    assert ca.tolist() == cb.tolist()
    assert oa.tolist() == ob.tolist()
    for e in range(E):
        lo, hi = oa[e], oa[e + 1]
        assert sorted(ra[lo:hi].tolist()) == sorted(rb[lo:hi].tolist()), f"expert {e}"


def test_noalloc_plan_matches_workspace_plan_twice(moe):
    cases = [Workload("first", "a8w4_fp8_fp4", 8192, 128, 128, 256, 8, 41, 0.0, zipf_s=1.2, zipf_empty=16),
             Workload("second", "a16w16", 300, 128, 128, 6, 2, 42, 0.0)]
    for wl in cases:  # two calls in a row with different routing
        ids = make_inputs(wl, device=DEV)["topk_ids"]
        if wl.name == "second":
            ids = ids.clone()
            ids[::5, 1] = -1  # masked routes
        d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
        _same_plan(_plan_without_workspace(moe, ids, d, wl.E), _plan_with_workspace(moe, ids, d, wl.E), wl.E)


def test_noalloc_plan_rejects_sizes_beyond_its_array(moe):
    d = moe.dims(65537, 128, 128, 8, 1)  # T*K above the 65536 routes the array holds
    ids = torch.zeros((65537, 1), dtype=torch.int32, device=DEV)
    out = torch.zeros(65537, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_plan_noalloc(ids, d, out[:8], out[:9], out)
    assert err.value.status == 1  # MOE_ERR_INVALID_ARG, nothing launched
    d = moe.dims(4, 128, 128, 2000, 1)  # more experts than the array holds
    with pytest.raises(moe.MoeError):
        moe.moe_plan_noalloc(ids[:4], d, out[:2000], out[:2001], out[:4])


def test_noalloc_plan_with_shared_experts_and_the_largest_expert_count(moe):
    """Shared experts add one slot per token each (T*(K+S) routes, E+S experts); the second case
    fills the 1024 experts the array holds, where the scan and the per-expert histograms are largest."""
    for T, E, K, S, seed in ((300, 6, 2, 1, 43), (64, 1022, 4, 2, 44)):
        wl = Workload("shared", "a16w16", T, 128, 128, E, K, seed, 0.0)
        ids = make_inputs(wl, device=DEV)["topk_ids"]
        d = moe.dims(T, 128, 128, E, K, S)
        a = _plan_without_workspace(moe, ids, d, E + S, T * (K + S))
        b = _plan_with_workspace(moe, ids, d, E + S, T * (K + S))
        _same_plan(a, b, E + S)
        assert a[0][E:].tolist() == [T] * S  # every token reaches every shared expert


def test_noalloc_plan_skips_bad_ids_like_masked_routes(moe):
    """An id outside [-1, E) is skipped (this call has no error word to report it): the plan equals
    moe_plan's plan of the same routing with that id masked, and moe_plan reports the bad route."""
    wl = Workload("bad", "a16w16", 200, 128, 128, 8, 2, 45, 0.0)
    ids = make_inputs(wl, device=DEV)["topk_ids"].clone()
    ids[7, 1] = 8
    ids[100, 0] = 1 << 20
    masked = ids.clone()
    masked[7, 1] = -1
    masked[100, 0] = -1
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    _same_plan(_plan_without_workspace(moe, ids, d, wl.E), _plan_with_workspace(moe, masked, d, wl.E), wl.E)
    _same_plan(_plan_with_workspace(moe, ids, d, wl.E, expect_error=moe.MOE_ERR_BAD_ROUTE),
               _plan_with_workspace(moe, masked, d, wl.E), wl.E)


def test_noalloc_plan_takes_the_same_dims_as_moe_plan(moe):
    """Shapes moe_plan rejects are rejected here too, before anything is launched; so are shared-expert
    slots that take T*(K+S) past the array although T*K fits."""
    ids = torch.zeros((30000, 2), dtype=torch.int32, device=DEV)
    out = torch.zeros(90000, dtype=torch.int32, device=DEV)
    for d in (moe.dims(4, 100, 128, 8, 2), moe.dims(4, 128, 128, 2, 3), moe.dims(4, 128, 128, 8, 2, 31)):
        with pytest.raises(moe.MoeError) as err:
            moe.moe_plan_noalloc(ids[:4], d, out[:40], out[:41], out[:200])
        assert err.value.status == 1
        assert moe.moe_workspace_bytes(d, "a16w16") == 0  # moe_plan's own dims check fails too
    d = moe.dims(30000, 128, 128, 8, 2, 1)  # T*K = 60000 fits, T*(K+S) = 90000 does not
    with pytest.raises(moe.MoeError) as err:
        moe.moe_plan_noalloc(ids, d, out[:9], out[:10], out)
    assert err.value.status == 1
