"""Asynchronous compaction on a side stream (App. E.3), through the C ABI.

Two engines over identical synthetic caches run the same boundary event:
one compacts on its own stream, the other on a side stream while summary
updates of the next decode steps are issued on the engine stream.  After
gp_wait_compaction the K/V caches, the block tables, the page pool, the
keep masks and a following demand call must be identical.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_step_gb300 as gp
import synth
from synth.workloads import ModelShape

import harness as hz

pytestmark = pytest.mark.gpu

SHAPE = ModelShape(2, 8, 2, 128, "bf16", "bf16", 5.0e5)


def _engine(side):
    w = synth.make_workload("custom", device="cuda", shape=SHAPE, sizes=[5, 33, 64, 2], seed_xor=31)
    run = hz.EngineRun(w)
    if side is not None:
        gp.gp_set_compaction_stream(run.ctx, side)
    run.feed_history()
    return w, run


@pytest.mark.parametrize("call", ["compress_hold", "shrink", "compress_fill"])
def test_side_stream_compaction_matches_engine_stream(call):
    side = torch.cuda.Stream()
    (wa, ra), (wb, rb) = _engine(None), _engine(side)
    try:
        q = wa.history[-1]
        assert torch.equal(q, wb.history[-1])
        reqs_a = [r for r in ra.reqs if r.num_pages >= 3]
        reqs_b = [r for r in rb.reqs if r.num_pages >= 3]
        da = gp.gp_boundary_demand(ra.ctx, reqs_a, q)
        db = gp.gp_boundary_demand(rb.ctx, reqs_b, q)
        assert [(x.sum_k_short, x.sum_k_long) for x in da] == [(x.sum_k_short, x.sum_k_long) for x in db]
        fn = getattr(gp, "gp_" + call)
        fn(ra.ctx, reqs_a)
        fn(rb.ctx, reqs_b)
        # decode steps of the side-stream engine go on while its compaction runs
        for t in range(4):
            qn = synth.query_step(wb, [True] * wb.n)
            rb.update(qn, False)
            ra.update(qn.clone(), False)
        gp.gp_wait_compaction(rb.ctx, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.equal(wa.k_cache, wb.k_cache) and torch.equal(wa.v_cache, wb.v_cache)
        assert [r.pages for r in reqs_a] == [r.pages for r in reqs_b]
        for pg in range(wa.num_pages):
            assert gp.gp_page_refcount(ra.ctx, pg) == gp.gp_page_refcount(rb.ctx, pg)
        for i, r in enumerate(reqs_a):
            P = len(r.pages) + (1 if call == "shrink" else 0)
            ma = gp.gp_debug_keep_mask(ra.ctx, i, ra.units, P)
            mb = gp.gp_debug_keep_mask(rb.ctx, i, rb.units, P)
            assert np.array_equal(ma, mb)
        assert gp.gp_stats(ra.ctx)["moved_rows"] == gp.gp_stats(rb.ctx)["moved_rows"] > 0
        # the next demand call waits for the side stream by itself
        q2 = synth.query_step(wa, [False] * wa.n)
        d2a = gp.gp_boundary_demand(ra.ctx, reqs_a, q2)
        d2b = gp.gp_boundary_demand(rb.ctx, reqs_b, q2)
        assert [(x.sum_k_short, x.sum_k_long) for x in d2a] == [(x.sum_k_short, x.sum_k_long) for x in d2b]
    finally:
        ra.close()
        rb.close()
