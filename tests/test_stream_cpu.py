"""CPU tests of the continuous-batching stream's recipe and of its lifecycle
bookkeeping on a host-only engine context (no GPU: only the page pool and
slot calls run).  The GPU stream itself is tests/test_gpu_stream.py."""

import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth
from synth.stream import ContinuousBatch
from synth.workloads import ModelShape, event_counts, private_pages

SMALL = ModelShape(2, 4, 2, 64, "bf16", "bf16", 1.0e4)


def _small(**kw):
    args = dict(shape=SMALL, seats=16, group=8, prefix_pages=2, spare_pages=24, max_pages=24)
    args.update(kw)
    return synth.make_workload("stream256", device="cpu", **args)


def test_recipe_lengths_and_events():
    g = torch.Generator().manual_seed(3)
    pages = private_pages(g, 20000)
    assert min(pages) == 2 and max(pages) == 64          # 512 .. 16384 tokens in 256-token pages
    med = sorted(pages)[len(pages) // 2]
    assert med == 8                                       # median 2048 tokens
    ev = event_counts(g, 200000, 12.0)
    assert min(ev) >= 1 and abs(sum(ev) / len(ev) - 12.0) < 0.2


def test_recipe_prefix_groups_share_pages():
    w = _small()
    pre = w.extra["prefixes"]
    assert len(pre) == 2 and all(len(p) == 2 for p in pre)
    for s, table in enumerate(w.block_tables):
        assert table[:2] == pre[s // 8]
        assert len(table) >= 4
    priv = [pg for t in w.block_tables for pg in t[2:]]
    assert len(priv) == len(set(priv))                    # private pages are distinct
    assert w.num_pages == 4 + len(priv) + 24
    w2 = _small()
    assert w2.block_tables == w.block_tables              # seeded
    assert torch.equal(w2.k_cache, w.k_cache)


def _host_stream():
    w = _small()
    cfg = gp.gp_config_default(num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=64, max_slots=16,
                               num_pages=w.num_pages, max_pages_per_req=24)
    ctx = gp.gp_create(cfg)
    return w, ctx, ContinuousBatch(gp, ctx, w, 24)


def test_initial_pool_mirrors_the_tables():
    w, ctx, drv = _host_stream()
    try:
        for pg in range(w.num_pages):
            n = sum(t.count(pg) for t in w.block_tables)
            assert gp.gp_page_refcount(ctx, pg) == n
        assert gp.gp_page_refcount(ctx, w.extra["prefixes"][0][0]) == 8
        assert gp.gp_free_page_count(ctx) == 24
    finally:
        gp.gp_destroy(ctx)


def test_release_and_admission_follow_the_oracle_pool():
    w, ctx, drv = _host_stream()
    try:
        pool = og.PagePool(w.num_pages)
        for t in w.block_tables:
            for pg in t:
                pool.refcount[pg] += 1
        # release two members of group 0: their private pages return, the prefix stays shared
        from synth.stream import StepLog
        for s in (1, 2):
            for pg in drv.seats[s].req.pages:
                pool.unref(pg)
            drv._release(s)
        log = StepLog(step=0)
        drv._admit(1, 0, log)
        assert len(log.admitted) == 1
        s, table = log.admitted[0]
        assert table[:2] == w.extra["prefixes"][0]        # the live prefix is shared
        for pg in table:
            if pool.refcount[pg] > 0:
                pool.ref(pg)
            else:
                assert pool.alloc() == pg                 # lowest free page first
        for pg in range(w.num_pages):
            assert gp.gp_page_refcount(ctx, pg) == pool.refcount[pg]
        # the whole group leaves: the next member of the group writes a fresh prefix
        for s2 in range(8):
            if drv.seats[s2].req is not None:
                drv._release(s2)
        log = StepLog(step=1)
        drv._admit(0, 1, log)
        table = log.admitted[0][1]
        assert all(gp.gp_page_refcount(ctx, pg) == 1 for pg in table)
        assert drv.prefix[0] == table[:2]
    finally:
        gp.gp_destroy(ctx)
