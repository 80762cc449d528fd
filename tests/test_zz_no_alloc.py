"""gp_boundary_demand_noalloc against gp_boundary_demand, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory at call time (for example a server that reserves all GPU memory at
start-up so that no request later fails on an out-of-memory error or stalls
on cudaMalloc's implicit synchronisation).  It keeps every temporary in one
static device array.  Here its results must equal the allocating entry
point's on two calls in a row (the D_p tolerance of the other tests is +-1 at
ties with p; the two calls run the same kernels, so they agree exactly), and
a call that needs more scratch than the array holds must be refused with a
clear error.  This file is collected last so that a failure here does not
stop the other tests from running first.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_step_gb300 as gp
import synth

import harness as hz

pytestmark = pytest.mark.gpu


def _run(name):
    kw = {"variant": "compress"} if name == "tiny" else {}
    w = synth.make_workload(name, device="cuda", **kw)
    if name == "llama8b_single":
        for t in range(32):
            w.history.append(synth.query_step(w, [t < 24]))
    run = hz.EngineRun(w, max_slots=16)
    run.feed_history()
    return w, run


@pytest.mark.parametrize("name", ["tiny", "llama8b_single"])
def test_noalloc_matches_allocating_entry_point_twice(name):
    w, run = _run(name)
    try:
        q = w.history[-1]
        ref = gp.gp_boundary_demand(run.ctx, run.reqs, q)
        kref = gp.gp_debug_demand_k(run.ctx, 0, run.units)
        for call in range(2):
            k = np.full((1, run.units, 2), -1, dtype=np.int32)
            got = gp.gp_boundary_demand_noalloc(run.ctx, run.reqs, q, k)
            torch.cuda.synchronize()
            assert np.abs(k[0].astype(np.int64) - kref).max() <= 1, f"call {call}"
            assert np.array_equal(k[0], kref), f"call {call}: per-unit D_p differ"
            assert got[0].sum_k_short == ref[0].sum_k_short, f"call {call}"
            assert got[0].sum_k_long == ref[0].sum_k_long, f"call {call}"
            assert got[0].num_candidates == ref[0].num_candidates
            assert got[0].delta == ref[0].delta
    finally:
        run.close()


def test_noalloc_refuses_calls_beyond_its_scratch():
    w, run = _run("llama8b_single")
    try:
        pages = run.reqs[0].pages
        reqs = [run.reqs[0]]
        for _ in range(7):   # 8 requests x 32 pages x 256 units: > 64 MiB of importance and a-values
            slot = gp.gp_slot_acquire(run.ctx)
            reqs.append(gp.Request(slot, pages, run.reqs[0].pos, run.cfg.max_pages_per_req))
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_boundary_demand_noalloc(run.ctx, reqs, torch.zeros(
                w.shape.num_layers, len(reqs), w.shape.num_q_heads, w.shape.head_dim,
                dtype=torch.bfloat16, device="cuda"))
        assert ei.value.status == gp.GP_ERR_INVALID
        assert "static scratch" in str(ei.value)
        # the refused call left the engine usable
        got = gp.gp_boundary_demand_noalloc(run.ctx, [run.reqs[0]], w.history[-1])
        ref = gp.gp_boundary_demand(run.ctx, [run.reqs[0]], w.history[-1])
        assert (got[0].sum_k_short, got[0].sum_k_long) == (ref[0].sum_k_short, ref[0].sum_k_long)
    finally:
        run.close()
