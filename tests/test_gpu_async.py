"""Asynchronous compaction on a side stream (App. E.3), through the C ABI.

Also decode attention issued while the compaction is pending: over requests
it does not touch (no wait) and over compacted ones (a wait on it).

Two engines over identical synthetic caches run the same boundary event:
one compacts on its own stream, the other on a side stream while summary
updates of the next decode steps are issued on the engine stream.  After
gp_wait_compaction the K/V caches, the block tables, the page pool, the
keep masks and a following demand call must be identical.  A side-stream
compaction of two requests sharing a prefix is also checked against the
oracle (copy-on-write plans, keep masks, gathered bytes).
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


def test_side_stream_compaction_with_a_shared_prefix_matches_oracle():
    """Both holders of a shared two-page prefix compressed in one side-stream
    call, against the oracle: copy-on-write plans taken with the refcounts at
    the start of the call (App. E.2; every co-sharer of the call copies, and
    the originals are freed once both dropped them), the Eq. 10 keep masks,
    and the K/V bytes of the oracle's gather under the new tables."""
    import oracle.growpage as og
    w = synth.make_workload("custom", device="cuda", shape=SHAPE, sizes=[4, 3], seed_xor=41)
    t0, t1 = w.block_tables
    w.block_tables[1] = [t0[0], t0[1]] + t1
    w.positions[1] = len(w.block_tables[1]) * 256
    cfg = hz.engine_config(w)
    ctx = gp.gp_create(cfg, w.k_cache, w.v_cache, None)
    side = torch.cuda.Stream()
    try:
        for _ in range(w.num_pages):
            gp.gp_page_alloc(ctx)
        used = set(t0) | set(w.block_tables[1])
        for pg in range(w.num_pages):
            if pg not in used:
                gp.gp_page_unref(ctx, pg)
        gp.gp_page_ref(ctx, t0[0])
        gp.gp_page_ref(ctx, t0[1])
        reqs = [gp.Request(gp.gp_slot_acquire(ctx), w.block_tables[r], w.positions[r], cfg.max_pages_per_req)
                for r in range(2)]
        slots = torch.tensor([q.slot for q in reqs], dtype=torch.int32, device="cuda")
        first, nfirst = torch.ones(2, dtype=torch.uint8, device="cuda"), torch.zeros(2, dtype=torch.uint8, device="cuda")
        for t, q in enumerate(w.history):
            gp.gp_update_summaries(ctx, 2, slots, q.contiguous(), first if t == 0 else nfirst)
        gp.gp_set_compaction_stream(ctx, side)
        q = w.history[-1]
        sh = w.shape
        units = sh.num_layers * sh.num_kv_heads
        # the oracle's selection inputs, from the keys before the compaction
        oracle_units = []
        for r, req in enumerate(reqs):
            s, l = hz.oracle_summaries(w.history, r)
            qt = og.summary_queries(s, l, q[:, r].double().cpu().numpy(), req.pos, sh.rope_theta)
            oracle_units.append([hz.oracle_unit_dev(qt, w.k_cache, req.pages, u // sh.num_kv_heads,
                                                    u % sh.num_kv_heads, sh.group) for u in range(units)])
        pool = og.PagePool(w.num_pages, [gp.gp_page_refcount(ctx, pg) for pg in range(w.num_pages)])
        old = [list(r.pages) for r in reqs]
        plans = [og.cow_plan(t, pool) for t in old]          # refcounts as at the start of the call
        for _, replaced in plans:
            og.release_replaced(replaced, pool)
        pre_k, pre_v = w.k_cache.double().cpu().numpy(), w.v_cache.double().cpu().numpy()
        gp.gp_boundary_demand(ctx, reqs, q)
        gp.gp_compress_hold(ctx, reqs)
        for t in range(3):                                   # decode steps while the side stream compacts
            gp.gp_update_summaries(ctx, 2, slots, synth.query_step(w, [True, False]), nfirst)
        gp.gp_wait_compaction(ctx, torch.cuda.current_stream())
        gp.gp_synchronize(ctx)
        torch.cuda.synchronize()
        assert [r.pages for r in reqs] == [p for p, _ in plans]
        assert [gp.gp_page_refcount(ctx, pg) for pg in range(w.num_pages)] == pool.refcount
        assert gp.gp_page_refcount(ctx, t0[0]) == 0 and gp.gp_page_refcount(ctx, t0[1]) == 0
        ek, ev = pre_k, pre_v
        for r, req in enumerate(reqs):
            P = req.num_pages
            keep = gp.unpack_mask(gp.gp_debug_keep_mask(ctx, r, units, P), P * 256)
            for u in range(units):
                ok, _, msg = hz.topk_ok(keep[u], oracle_units[r][u].s, P)
                assert ok, f"request {r} unit {u}: {msg}"
            ek, ev = og.compress_cache(ek, ev, old[r], req.pages,
                                       keep.reshape(sh.num_layers, sh.num_kv_heads, -1), 256)
        got_k, got_v = w.k_cache.double().cpu().numpy(), w.v_cache.double().cpu().numpy()
        for req in reqs:
            n_live = (req.num_pages - 1) * 256
            for layer in range(sh.num_layers):
                for h in range(sh.num_kv_heads):
                    for exp, got in ((ek, got_k), (ev, got_v)):
                        assert np.array_equal(og.gather_logical(exp, req.pages, layer, h)[:n_live],
                                              og.gather_logical(got, req.pages, layer, h)[:n_live])
    finally:
        gp.gp_destroy(ctx)


def test_decode_attention_beside_a_side_stream_compaction():
    """App. E.3: while a Compress & Hold runs on the side stream, decode
    attention over a request it does not touch runs without waiting for it,
    and attention over a compacted request waits for it (its pages overlap);
    both give exactly the outputs of the engine that compacted on its own
    stream (the tensor-core attention kernel, summaries updated in passing)."""
    side = torch.cuda.Stream()
    (wa, ra), (wb, rb) = _engine(None), _engine(side)
    try:
        sh = wa.shape
        q = wa.history[-1]
        comp_a = [r for r in ra.reqs if r.num_pages >= 3]
        comp_b = [r for r in rb.reqs if r.num_pages >= 3]
        idle_a = [r for r in ra.reqs if r.num_pages < 3]
        idle_b = [r for r in rb.reqs if r.num_pages < 3]
        assert comp_a and idle_a
        gp.gp_boundary_demand(ra.ctx, comp_a, q)
        gp.gp_boundary_demand(rb.ctx, comp_b, q)
        gp.gp_compress_hold(ra.ctx, comp_a)
        gp.gp_compress_hold(rb.ctx, comp_b)   # on the side stream
        qa = torch.randn(len(ra.reqs), sh.num_q_heads, sh.head_dim, generator=torch.Generator().manual_seed(9))
        qa = qa.to(torch.bfloat16).cuda()
        outs = []
        for run, idle, comp in ((ra, idle_a, comp_a), (rb, idle_b, comp_b)):
            o_idle = torch.empty(len(idle), sh.num_q_heads, sh.head_dim, device="cuda")
            o_comp = torch.empty(len(comp), sh.num_q_heads, sh.head_dim, device="cuda")
            nf_i = torch.zeros(len(idle), dtype=torch.uint8, device="cuda")
            nf_c = torch.zeros(len(comp), dtype=torch.uint8, device="cuda")
            for layer in range(sh.num_layers):
                # the untouched requests first: no wait for the side stream
                gp.gp_decode_attention(run.ctx, layer, idle, [x.num_pages * 256 for x in idle],
                                       qa[:len(idle)].contiguous(), nf_i, o_idle)
                gp.gp_decode_attention(run.ctx, layer, comp, [x.num_pages * 256 for x in comp],
                                       qa[len(idle):len(idle) + len(comp)].contiguous(), nf_c, o_comp)
            gp.gp_synchronize(run.ctx)
            torch.cuda.synchronize()
            outs.append((o_idle.cpu(), o_comp.cpu()))
        assert torch.equal(outs[0][0], outs[1][0]), "attention beside the compaction differs"
        assert torch.equal(outs[0][1], outs[1][1]), "attention after the compaction differs"
        for x, y in zip(ra.reqs, rb.reqs):
            sa = gp.gp_read_summaries(ra.ctx, x.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            sb = gp.gp_read_summaries(rb.ctx, y.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            assert np.array_equal(sa, sb)
    finally:
        ra.close()
        rb.close()
