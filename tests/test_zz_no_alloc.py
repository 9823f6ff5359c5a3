"""moe_bucket_noalloc against moe_pre_dispatch (GB300 only).

moe_bucket_noalloc serves callers that cannot allocate device memory where they
route tokens (runtimes that plan all device buffers ahead of time, threads that
cannot afford cudaMalloc's device-wide synchronisation): its scratch is a static
array inside the library.  Here two calls in a row, with different routings, must
give exactly the counts and assignment rows that moe_pre_dispatch stores in a
workspace, and the ones the oracle's bucketing defines (integer outputs:
bit-exact).  This file sorts last so that a run
stopping at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_scaled_fp4_pre_gb300 as mx  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _existing_path(dims, ws, ids, tw):
    T = ids.shape[0]
    x = torch.zeros((T, dims.hidden), dtype=torch.bfloat16, device="cuda")
    # moe_bucket_noalloc lays rows out in 128-row tiles; pre_dispatch then must too
    mx.moe_workspace_set_tiles(ws, mx.MOE_TILES_WIDE)
    mx.moe_pre_dispatch(dims, x, _dev(ids), _dev(tw), T, ws)
    d = mx.moe_read_dispatch(dims, ws, T)
    return d["counts"], d["assign_slot"]


def _noalloc_path(dims, ids, tw):
    T, k = ids.shape
    counts = torch.full((dims.num_experts,), -7, dtype=torch.int32, device="cuda")
    slots = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    mx.moe_bucket_noalloc(dims, _dev(ids), _dev(tw), T, counts, slots)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), slots.cpu().numpy()


def _oracle_path(ids, E, tile_rows=128):
    """Counts and assignment rows from the oracle's bucketing: within an expert the
    oracle's (token, k index) order, each expert's rows starting at the sum of the
    earlier experts' counts rounded up to 128-row tiles; -1 for ids outside [0, E)."""
    T, k = ids.shape
    counts, offsets, st, sj, bad = oracle.bucket(ids, E)
    slots = np.full(T * k, -1, np.int64)
    seg = 0
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for i in range(lo, hi):
            slots[int(st[i]) * k + int(sj[i])] = seg + (i - lo)
        seg += -(-int(counts[e]) // tile_rows) * tile_rows
    return counts, slots, bad


def test_noalloc_bucketing_matches_pre_dispatch_on_two_calls():
    dims = mx.make_dims(256, 128, 32, 4, 2048)
    ws = torch.empty(mx.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    mx.moe_workspace_init(dims, ws)
    # call 1: skewed routing, 2048 tokens x 4 = 8192 assignments (the limit), several
    # 128-row tiles for the popular experts
    w1 = synth.Workload("nz1", T=2048, H=256, I=128, E=32, k=4, routing="zipf")
    ids1, tw1 = synth.routing(w1, seed=3)
    # call 2: fewer tokens, uniform routing and two ids outside [0, E), so that rows
    # left over from call 1 would show if the scratch leaked into the result
    w2 = synth.Workload("nz2", T=300, H=256, I=128, E=32, k=4)
    ids2, tw2 = synth.routing(w2, seed=4)
    ids2[5, 1] = -1
    ids2[17, 3] = 32
    for ids, tw in ((ids1, tw1), (ids2, tw2)):
        got_counts, got_slots = _noalloc_path(dims, ids, tw)
        ref_counts, ref_slots = _existing_path(dims, ws, ids, tw)
        assert np.array_equal(got_counts, ref_counts)
        assert np.array_equal(got_slots, ref_slots)
        o_counts, o_slots, o_bad = _oracle_path(ids, dims.num_experts)
        assert np.array_equal(got_counts, o_counts)
        assert np.array_equal(got_slots, o_slots)
        # skipped ids show as -1 rows and as counts summing short of T * k
        assert int(got_counts.sum()) == ids.size - o_bad
    assert (got_slots == -1).sum() == 2


def test_noalloc_rejects_sizes_beyond_its_limits():
    small = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(mx.MoeError) as ei:      # 2049 * 4 > 8192 assignments
        mx.moe_bucket_noalloc(mx.make_dims(256, 128, 32, 4, 4096), small, small, 2049, small, small)
    assert ei.value.status == mx.MOE_ERR_INVALID_ARG
    assert "8192" in mx.moe_last_error()
    with pytest.raises(mx.MoeError) as ei:      # more than 256 experts
        mx.moe_bucket_noalloc(mx.make_dims(256, 128, 512, 4, 16), small, small, 1, small, small)
    assert ei.value.status == mx.MOE_ERR_INVALID_ARG
    assert "256" in mx.moe_last_error()
