"""GPU parity of Shrink (App. H.1, Eq. 13) through the C ABI.

Shrink runs the Eq. 10 selection with K_t = (P-2) b - R, compacts two
pages' worth of history into logical slots [0, (P-2) b) and returns the
emptied last page to the pool.  Against the fp64 oracle, for every
(layer, KV head): the keep masks (identical except within the top-k
tolerance), the compacted K/V bytes for the GPU's own index set (exact),
the shortened block table and the pool; with a prefix shared by two
requests, the copy-on-write pages as the oracle plans them.
"""

import numpy as np
import pytest
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth
from synth.workloads import ModelShape

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256
SHAPE = ModelShape(2, 8, 2, 128, "bf16", "bf16", 5.0e5)


def _oracle_request(w, r):
    s, l = hz.oracle_summaries(w.history, r)
    qc = w.history[-1][:, r].double().cpu().numpy()
    return og.summary_queries(s, l, qc, w.positions[r], w.shape.rope_theta)


@pytest.mark.parametrize("shared", [False, True])
def test_shrink_matches_oracle(shared):
    sizes = [3, 5, 33, 129]
    w = synth.make_workload("custom", device="cuda", shape=SHAPE, sizes=sizes, seed_xor=21)
    run = hz.EngineRun(w, policy=gp.GP_POLICY_SHRINK)
    try:
        if shared:
            # request 1 takes a reference to request 0's first two pages (a shared prefix)
            pre = run.reqs[0].pages[:2]
            for pg in pre:
                gp.gp_page_ref(run.ctx, pg)
            old1 = run.reqs[1].pages
            for pg in old1[:2]:
                gp.gp_page_unref(run.ctx, pg)
            run.reqs[1] = gp.Request(run.reqs[1].slot, pre + old1[2:], run.reqs[1].pos, run.cfg.max_pages_per_req)
        run.feed_history()
        q = w.history[-1]
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        sh = w.shape
        units = run.units
        # the oracle's page pool from the engine's state before the call
        pool = og.PagePool(w.num_pages)
        for pg in range(w.num_pages):
            pool.refcount[pg] = gp.gp_page_refcount(run.ctx, pg)
        before = [list(x.pages) for x in run.reqs]
        snap, oracle_units = {}, {}
        for r, req in enumerate(run.reqs):
            qt = _oracle_request(w, r)
            for idx in range(units):
                layer, h = divmod(idx, sh.num_kv_heads)
                oracle_units[(r, idx)] = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group)
                snap[(r, idx)] = (hz.unit_keys_dev(w.k_cache, req.pages, layer, h),
                                  hz.unit_keys_dev(w.v_cache, req.pages, layer, h))
        gp.gp_shrink(run.ctx, run.reqs)
        torch.cuda.synchronize()
        # one call plans every request's copy-on-write first (lowest free
        # pages, request order), then drops the replaced references, then
        # returns each request's emptied last page
        plans = [og.cow_plan(before[r], pool) for r in range(len(run.reqs))]
        for _, replaced in plans:
            og.release_replaced(replaced, pool)
        for r, req in enumerate(run.reqs):
            P = len(before[r])
            expect = og.shrink_release(plans[r][0], pool)
            assert req.pages == expect, f"request {r}: block table {req.pages} vs oracle {expect}"
            masks = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, r, units, P), P * PAGE)
            for idx in range(units):
                u = oracle_units[(r, idx)]
                ok, _, msg = hz.topk_ok(masks[idx], u.s, P, drop=2)
                assert ok, f"request {r} (P={P}) unit {idx}: {msg}"
                layer, h = divmod(idx, sh.num_kv_heads)
                kept = np.nonzero(masks[idx])[0]
                n_live = (P - 2) * PAGE
                kp, vp = snap[(r, idx)]
                assert np.array_equal(hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:n_live], kp[kept])
                assert np.array_equal(hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:n_live], vp[kept])
        for pg in range(w.num_pages):
            assert gp.gp_page_refcount(run.ctx, pg) == pool.refcount[pg], f"page {pg}"
        if shared:
            assert gp.gp_stats(run.ctx)["cow_pages"] >= 2
    finally:
        run.close()


def test_shrink_needs_three_pages():
    w = synth.make_workload("custom", device="cuda", shape=SHAPE, sizes=[2], seed_xor=22)
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_shrink(run.ctx, run.reqs)
        assert ei.value.status == gp.GP_ERR_INVALID
        assert run.reqs[0].num_pages == 2
    finally:
        run.close()


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("select_mode", ["speculative", "in_compaction"])
def test_hole_fill_matches_oracle(shared, select_mode):
    """gp_compress_fill: the Eq. 10 selection of Compress & Hold, then the
    order-destroying hole fill: bytes exactly as the oracle's hole fill of
    the GPU's own keep masks, copy-on-write as planned by the oracle.  With
    the selection speculative (its own launch after the demand call) and
    inside the compaction launch."""
    sizes = [2, 5, 33]
    w = synth.make_workload("custom", device="cuda", shape=SHAPE, sizes=sizes, seed_xor=23)
    run = hz.EngineRun(w)
    gp.gp_set_selection_mode(run.ctx, gp.GP_SELECT_SPECULATIVE if select_mode == "speculative"
                             else gp.GP_SELECT_IN_COMPACTION)
    try:
        if shared:
            pre = run.reqs[0].pages[:2]
            for pg in pre:
                gp.gp_page_ref(run.ctx, pg)
            old1 = run.reqs[1].pages
            for pg in old1[:2]:
                gp.gp_page_unref(run.ctx, pg)
            run.reqs[1] = gp.Request(run.reqs[1].slot, pre + old1[2:], run.reqs[1].pos, run.cfg.max_pages_per_req)
        run.feed_history()
        gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
        sh = w.shape
        units = run.units
        pool = og.PagePool(w.num_pages)
        for pg in range(w.num_pages):
            pool.refcount[pg] = gp.gp_page_refcount(run.ctx, pg)
        before = [list(x.pages) for x in run.reqs]
        snap, oracle_units = {}, {}
        for r, req in enumerate(run.reqs):
            qt = _oracle_request(w, r)
            for idx in range(units):
                layer, h = divmod(idx, sh.num_kv_heads)
                oracle_units[(r, idx)] = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group)
                snap[(r, idx)] = (hz.unit_keys_dev(w.k_cache, req.pages, layer, h),
                                  hz.unit_keys_dev(w.v_cache, req.pages, layer, h))
        moved0 = gp.gp_stats(run.ctx)["moved_rows"]
        gp.gp_compress_fill(run.ctx, run.reqs)
        torch.cuda.synchronize()
        plans = [og.cow_plan(before[r], pool) for r in range(len(run.reqs))]
        for _, replaced in plans:
            og.release_replaced(replaced, pool)
        fillers = 0
        for r, req in enumerate(run.reqs):
            P = len(before[r])
            assert req.pages == plans[r][0]
            masks = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, r, units, P), P * PAGE)
            for idx in range(units):
                ok, _, msg = hz.topk_ok(masks[idx], oracle_units[(r, idx)].s, P)
                assert ok, f"request {r} (P={P}) unit {idx}: {msg}"
                layer, h = divmod(idx, sh.num_kv_heads)
                kp, vp = snap[(r, idx)]
                n_live = (P - 1) * PAGE
                assert np.array_equal(hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:n_live],
                                      og.hole_fill_unit(kp, masks[idx], P, PAGE))
                assert np.array_equal(hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:n_live],
                                      og.hole_fill_unit(vp, masks[idx], P, PAGE))
                fillers += int(masks[idx][n_live:P * PAGE].sum())
        for pg in range(w.num_pages):
            assert gp.gp_page_refcount(run.ctx, pg) == pool.refcount[pg]
        if not shared:
            # without copy-on-write only the last page's kept rows move
            assert gp.gp_stats(run.ctx)["moved_rows"] - moved0 == fillers
    finally:
        run.close()
