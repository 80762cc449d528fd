"""Failure handling of the engine on the GPU, without faulting it.

* A bounded wait that gives up (GrowPage's Compress & Hold, Sec. 3.3 and
  App. E.2, runs its copies through bounded waits).  The compaction's copy
  waits get a limit of zero clock cycles through the test hook, so every CTA
  with rows to move gives up at its first chunk, whether or not the copy has
  landed.
  Each CTA then waits, with the full limit, for the copies it already issued
  and returns; gp_synchronize reports GP_ERR_TIMEOUT and clears it.  The
  context stays usable: with the default limit back and the cache restored, a
  new demand call and Compress & Hold match the oracle.
* A compaction launch that fails after the copy-on-write pages were taken
  (App. E.2), injected on the host: gp_compress_hold returns GP_ERR_CUDA and
  leaves the block table, every refcount, the free pool and the K/V bytes as
  they were.  The same call then succeeds and matches the oracle's
  copy-on-write plan and gather.
"""

import numpy as np
import pytest
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256


def _oracle_units(w, run, q):
    """Oracle demand and importance of every unit of request 0 over the cache
    as it is now (call before the compaction rewrites it)."""
    req = run.reqs[0]
    sh = w.shape
    s, l = hz.oracle_summaries(w.history, 0)
    qt = og.summary_queries(s, l, q[:, 0].double().cpu().numpy(), req.pos, sh.rope_theta)
    pages = hz.cache_f64(w.k_cache, req.pages)
    return {layer * sh.num_kv_heads + h: hz.oracle_unit(qt, pages, req.pages, layer, h, sh.group)
            for layer in range(sh.num_layers) for h in range(sh.num_kv_heads)}


def _check_compaction(w, run, units, pre_k, pre_v, old_table):
    """Keep masks against Eq. 10 and the moved rows against the oracle's gather."""
    req = run.reqs[0]
    sh = w.shape
    P = req.num_pages
    keep = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, 0, run.units, P), P * PAGE)
    masks = np.zeros((sh.num_layers, sh.num_kv_heads, P * PAGE), bool)
    for idx, u in units.items():
        ok, _, msg = hz.topk_ok(keep[idx], u.s, P)
        assert ok, f"unit {idx}: {msg}"
        masks[idx // sh.num_kv_heads, idx % sh.num_kv_heads] = keep[idx]
    torch.cuda.synchronize()
    ek, ev = og.compress_cache(pre_k.double().cpu().numpy(), pre_v.double().cpu().numpy(), old_table,
                               req.pages, masks, PAGE)
    got_k = w.k_cache.double().cpu().numpy()
    got_v = w.v_cache.double().cpu().numpy()
    n_live = (P - 1) * PAGE
    for layer in range(sh.num_layers):
        for h in range(sh.num_kv_heads):
            for exp, got in ((ek, got_k), (ev, got_v)):
                e = og.gather_logical(exp, req.pages, layer, h)[:n_live]
                g = og.gather_logical(got, req.pages, layer, h)[:n_live]
                assert np.array_equal(e, g), f"unit ({layer}, {h}): bytes differ"


def test_compaction_wait_timeout_is_reported_and_the_context_recovers():
    w = synth.make_workload("tiny", device="cuda", variant="compress")
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        q = w.history[-1]
        pre_k, pre_v = w.k_cache.clone(), w.v_cache.clone()
        old = list(run.reqs[0].pages)
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        gp.gp_debug_set_wait_limit(run.ctx, gp.GP_KERNEL_COMPRESS, 0)
        gp.gp_compress_hold(run.ctx, run.reqs)          # asynchronous: returns before the kernel ends
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_synchronize(run.ctx)                  # returns: every CTA gave up, drained and left
        assert ei.value.status == gp.GP_ERR_TIMEOUT, str(ei.value)
        gp.gp_synchronize(run.ctx)                      # the error word was cleared
        # the call's host state was committed (no page is shared, so the table
        # keeps its pages); restore the bytes and run the event again
        assert run.reqs[0].pages == old
        gp.gp_debug_set_wait_limit(run.ctx, gp.GP_KERNEL_COMPRESS, -1)
        w.k_cache.copy_(pre_k)
        w.v_cache.copy_(pre_v)
        torch.cuda.synchronize()
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        units = _oracle_units(w, run, q)
        gp.gp_compress_hold(run.ctx, run.reqs)
        gp.gp_synchronize(run.ctx)
        _check_compaction(w, run, units, pre_k, pre_v, old)
    finally:
        run.close()


def test_failed_compaction_launch_rolls_back_copy_on_write():
    w = synth.make_workload("tiny", device="cuda", variant="compress")
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        q = w.history[-1]
        req = run.reqs[0]
        shared = req.pages[1]
        gp.gp_page_ref(run.ctx, shared)                 # a second holder: copy-on-write at compaction
        gp.gp_boundary_demand(run.ctx, run.reqs, q)
        units = _oracle_units(w, run, q)
        pre_k, pre_v = w.k_cache.clone(), w.v_cache.clone()
        old = list(req.pages)
        rc = [gp.gp_page_refcount(run.ctx, p) for p in range(w.num_pages)]
        free = gp.gp_free_page_count(run.ctx)
        gp.gp_debug_fail_next_launch(run.ctx, gp.GP_KERNEL_COMPRESS)
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(run.ctx, run.reqs)
        assert ei.value.status == gp.GP_ERR_CUDA and "injected" in str(ei.value)
        gp.gp_synchronize(run.ctx)
        assert req.pages == old and req.num_pages == len(old)
        assert [gp.gp_page_refcount(run.ctx, p) for p in range(w.num_pages)] == rc
        assert gp.gp_free_page_count(run.ctx) == free
        assert torch.equal(w.k_cache, pre_k) and torch.equal(w.v_cache, pre_v)
        # the same call now succeeds, with the oracle's copy-on-write plan and gather
        pool = og.PagePool(w.num_pages, list(rc))
        plan, replaced = og.cow_plan(old, pool)
        assert replaced == [shared]
        gp.gp_compress_hold(run.ctx, run.reqs)
        gp.gp_synchronize(run.ctx)
        assert req.pages == plan
        og.release_replaced(replaced, pool)
        assert [gp.gp_page_refcount(run.ctx, p) for p in range(w.num_pages)] == pool.refcount
        _check_compaction(w, run, units, pre_k, pre_v, old)
        # the shared page itself was never written
        assert torch.equal(w.k_cache[:, shared], pre_k[:, shared])
        assert torch.equal(w.v_cache[:, shared], pre_v[:, shared])
    finally:
        run.close()
