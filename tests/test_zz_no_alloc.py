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
from synth.workloads import ModelShape

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


def _compare(run, reqs, q, tag):
    """gp_boundary_demand_noalloc against gp_boundary_demand on the same requests."""
    ref = gp.gp_boundary_demand(run.ctx, reqs, q)
    kref = [gp.gp_debug_demand_k(run.ctx, i, run.units) for i in range(len(reqs))]
    for call in range(2):
        k = np.full((len(reqs), run.units, 2), -1, dtype=np.int32)
        got = gp.gp_boundary_demand_noalloc(run.ctx, reqs, q, k)
        for i in range(len(reqs)):
            assert np.array_equal(k[i], kref[i]), f"{tag} call {call} request {i}: per-unit D_p differ"
            assert (got[i].sum_k_short, got[i].sum_k_long) == (ref[i].sum_k_short, ref[i].sum_k_long)
            assert got[i].num_candidates == ref[i].num_candidates and got[i].delta == ref[i].delta


def test_noalloc_several_requests_both_scans_odd_layout():
    """Several requests of mixed lengths in one call, on the tensor-core and
    the CUDA-core scan, with an odd number of (layer, KV head) units and an
    odd recent window, so that no request's regions start on a 16-byte
    boundary unless the entry point aligns them; and no device memory is
    allocated by repeated calls."""
    shape = ModelShape(3, 2, 1, 128, "bf16", "bf16", 5.0e5)      # 3 units, G = 2
    w = synth.make_workload("custom", device="cuda", shape=shape, sizes=[2, 17, 40, 3], seed_xor=5)
    run = hz.EngineRun(w, recent_window=3)
    try:
        run.feed_history()
        q = w.history[-1]
        for kind, tag in ((gp.GP_SCAN_AUTO, "tensor core"), (gp.GP_SCAN_CUDA_CORE, "CUDA core")):
            gp.gp_set_scan_kernel(run.ctx, kind)
            _compare(run, run.reqs, q, tag)
        gp.gp_set_scan_kernel(run.ctx, gp.GP_SCAN_AUTO)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(5):
            gp.gp_boundary_demand_noalloc(run.ctx, run.reqs, q)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    finally:
        run.close()


def test_noalloc_call_drops_the_demand_record_of_its_slots():
    """After a no-allocation call, Compress & Hold of the same request needs a
    new gp_boundary_demand: the cached importance predates the queries just
    scored."""
    w, run = _run("tiny")
    try:
        q = w.history[-1]
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        gp.gp_boundary_demand_noalloc(run.ctx, run.reqs, q)
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(run.ctx, run.reqs)
        assert ei.value.status == gp.GP_ERR_STATE
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        gp.gp_compress_hold(run.ctx, run.reqs)
        gp.gp_synchronize(run.ctx)
    finally:
        run.close()
