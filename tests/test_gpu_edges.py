"""GPU parity on edge cases of the GrowPage boundary engine, through the C ABI.

Small model shapes (2 layers, 2 KV heads) that reach every kernel variant:
bf16 caches with head_dim 64 / 128 and GQA group 2 / 4 (the tensor-core scan
and, when forced, the CUDA-core scan), an fp32 cache (CUDA-core only), and
requests of 1, 2, 5, 33, 64, 65, 128, 129, 160, 161 and 256 pages (one to
26 tensor-core parts per unit, every cluster shape of the CUDA-core scan, the
largest block table).  Against the fp64 oracle: D_p within the tie
tolerance, the demand distributions within 1e-4, the importance, the
decision (forced Grow at P = 1), the Eq. 10 keep masks and the compacted
bytes.  Also: copy-on-write of a shared prefix, GP_ERR_NO_PAGES leaving
everything unchanged, GP_ERR_STATE without a demand call, and caller masks
of the wrong size being refused.
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
SIZES = [1, 2, 5, 33, 64, 65, 128, 129, 160, 161, 256]
SHAPES = {
    "bf16_g4_d128": ModelShape(2, 8, 2, 128, "bf16", "bf16", 5.0e5),
    "bf16_g2_d128": ModelShape(2, 4, 2, 128, "bf16", "bf16", 5.0e5),
    "bf16_g4_d64": ModelShape(2, 8, 2, 64, "bf16", "bf16", 1.0e4),
    "bf16_g2_d64": ModelShape(2, 4, 2, 64, "bf16", "bf16", 1.0e4),
    "f32_g4_d128": ModelShape(2, 8, 2, 128, "f32", "f32", 5.0e5),
}


def _workload(shape, sizes, seed_xor=0):
    return synth.make_workload("custom", device="cuda", shape=shape, sizes=sizes, seed_xor=seed_xor)


def _oracle_request(w, r):
    s, l = hz.oracle_summaries(w.history, r)
    qc = w.history[-1][:, r].double().cpu().numpy()
    return og.summary_queries(s, l, qc, w.positions[r], w.shape.rope_theta)


def _check_units(run, w, r, qt, check_probs=True):
    """Compare request r's demand results with the oracle; return oracle units."""
    sh = w.shape
    req = run.reqs[r]
    P = req.num_pages
    ndem, ncmp = (P - 1) * PAGE, P * PAGE - 16
    ks = gp.gp_debug_demand_k(run.ctx, r, run.units)
    probs = gp.gp_debug_probs(run.ctx, r, run.units, ndem) if (check_probs and ndem) else None
    scores = gp.gp_debug_scores(run.ctx, r, run.units, ncmp)
    res, ties = {}, 0
    for layer in range(sh.num_layers):
        for h in range(sh.num_kv_heads):
            idx = layer * sh.num_kv_heads + h
            u = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group)
            res[idx] = u
            if ndem == 0:
                assert ks[idx, 0] == 0 and ks[idx, 1] == 0
            else:
                for x in range(2):
                    ok, msg = hz.dp_ok(int(ks[idx, x]), u.a_dem[x], 0.99)
                    assert ok, f"P={P} unit {idx} x {x}: {msg}"
                    ties += int(ks[idx, x] != u.k[x])
            if probs is not None:
                err = np.abs(probs[idx].astype(np.float64) - u.a_dem).max()
                assert err <= hz.PROB_ABS, f"P={P} unit {idx}: probability error {err}"
            sg = np.exp2(scores[idx].astype(np.float64))
            big = u.s > 1e-30
            rel = np.abs(sg[big] - u.s[big]) / u.s[big]
            assert rel.max() < 2e-5, f"P={P} unit {idx}: importance relative error {rel.max()}"
    return res, ties, ks


@pytest.mark.parametrize("shape_name", list(SHAPES))
def test_demand_decide_compress_all_sizes(shape_name):
    shape = SHAPES[shape_name]
    w = _workload(shape, SIZES)
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        q = w.history[-1]
        kinds = [gp.GP_SCAN_AUTO] + ([gp.GP_SCAN_CUDA_CORE] if shape.kv_dtype == "bf16" else [])
        if shape.kv_dtype != "bf16":
            with pytest.raises(gp.GrowPageError) as ei:
                gp.gp_set_scan_kernel(run.ctx, gp.GP_SCAN_TENSOR_CORE)
            assert ei.value.status == gp.GP_ERR_UNSUPPORTED
        qts = [_oracle_request(w, r) for r in range(w.n)]
        per_kind = {}
        for kind in kinds:
            gp.gp_set_scan_kernel(run.ctx, kind)
            dem = gp.gp_boundary_demand(run.ctx, run.reqs, q)
            out = []
            for r in range(w.n):
                res, ties, ks = _check_units(run, w, r, qts[r], check_probs=(kind == gp.GP_SCAN_AUTO))
                assert dem[r].sum_k_short == int(ks[:, 0].sum())
                assert dem[r].sum_k_long == int(ks[:, 1].sum())
                out.append((res, ties, ks))
            per_kind[kind] = out
        # bf16: the tensor-core scan serves every size up to the 256-page
        # block-table limit (161 and 256 pages included) -- forcing it must not
        # be refused, and it is the scan AUTO ran
        if shape.kv_dtype == "bf16":
            gp.gp_set_scan_kernel(run.ctx, gp.GP_SCAN_TENSOR_CORE)
            gp.gp_boundary_demand(run.ctx, run.reqs, q)
            for r in range(w.n):
                assert np.array_equal(gp.gp_debug_demand_k(run.ctx, r, run.units), per_kind[gp.GP_SCAN_AUTO][r][2]), \
                    f"request {r} (P={run.reqs[r].num_pages}): forced tensor-core scan differs from AUTO"
        # the two scans agree exactly where no oracle tie decides
        if len(per_kind) == 2:
            for r in range(w.n):
                a, b = per_kind[gp.GP_SCAN_AUTO][r], per_kind[gp.GP_SCAN_CUDA_CORE][r]
                if a[1] == 0 and b[1] == 0:
                    assert np.array_equal(a[2], b[2]), f"request {r}: scans disagree"
        # decision on the last demand call (CUDA core for bf16 shapes, else auto)
        gp.gp_set_scan_kernel(run.ctx, gp.GP_SCAN_AUTO)
        dem = gp.gp_boundary_demand(run.ctx, run.reqs, q)
        acts = gp.gp_decide(run.ctx, run.reqs, dem)
        free = gp.gp_free_page_count(run.ctx)
        granted = 0
        ks_last = [gp.gp_debug_demand_k(run.ctx, r, run.units) for r in range(w.n)]
        for r in range(w.n):
            res, _, _ = per_kind[gp.GP_SCAN_AUTO][r]
            P = run.reqs[r].num_pages
            kk = np.array([res[i].k for i in range(run.units)])
            for idx in range(run.units):
                for x in range(2):
                    if P > 1:
                        ok, msg = hz.dp_ok(int(ks_last[r][idx, x]), res[idx].a_dem[x], 0.99)
                        assert ok, f"P={P} unit {idx} x {x}: {msg}"
            ok, msg = hz.decision_ok(acts[r], kk, ks_last[r], P, free - granted)
            assert ok, f"request {r} (P={P}): {msg}"
            if acts[r].kind == gp.GP_ACT_GROW and not acts[r].forced:
                granted += 1
            if P == 1:
                assert acts[r].kind == gp.GP_ACT_GROW and acts[r].forced
        # Compress & Hold on every request with two or more pages
        sel = [r for r in range(w.n) if run.reqs[r].num_pages >= 2]
        reqs = [run.reqs[r] for r in sel]
        pre = {}
        for r in sel:
            for layer in range(shape.num_layers):
                for h in range(shape.num_kv_heads):
                    pre[(r, layer, h)] = (hz.unit_keys_dev(w.k_cache, run.reqs[r].pages, layer, h),
                                          hz.unit_keys_dev(w.v_cache, run.reqs[r].pages, layer, h))
        old_tables = {r: list(run.reqs[r].pages) for r in sel}
        # demand for exactly these requests (Compress & Hold uses its scores)
        gp.gp_boundary_demand(run.ctx, reqs, q[:, sel].contiguous())
        gp.gp_compress_hold(run.ctx, reqs)
        torch.cuda.synchronize()
        for j, r in enumerate(sel):
            P = run.reqs[r].num_pages
            assert run.reqs[r].pages == old_tables[r] and P == len(old_tables[r])
            masks = gp.gp_debug_keep_mask(run.ctx, j, run.units, P)
            keep = gp.unpack_mask(masks, P * PAGE)
            res = per_kind[gp.GP_SCAN_AUTO][r][0]
            for layer in range(shape.num_layers):
                for h in range(shape.num_kv_heads):
                    idx = layer * shape.num_kv_heads + h
                    ok, _, msg = hz.topk_ok(keep[idx], res[idx].s, P)
                    assert ok, f"P={P} unit {idx}: {msg}"
                    kpre, vpre = pre[(r, layer, h)]
                    kept = np.nonzero(keep[idx])[0]
                    n_live = (P - 1) * PAGE
                    kpost = hz.unit_keys_dev(w.k_cache, run.reqs[r].pages, layer, h)[:n_live]
                    vpost = hz.unit_keys_dev(w.v_cache, run.reqs[r].pages, layer, h)[:n_live]
                    assert np.array_equal(kpost, kpre[kept]), f"P={P} unit {idx}: K bytes"
                    assert np.array_equal(vpost, vpre[kept]), f"P={P} unit {idx}: V bytes"
    finally:
        run.close()


def _two_sharing(num_spare):
    """Two 4-page requests sharing their first two pages, plus spare pages."""
    shape = SHAPES["bf16_g4_d128"]
    w = _workload(shape, [4, 2], seed_xor=7)
    # request 1 = request 0's first two pages + its own two pages
    t0, t1 = w.block_tables
    w.block_tables[1] = [t0[0], t0[1]] + t1
    w.positions[1] = 4 * PAGE
    cfg = hz.engine_config(w, num_pages=w.num_pages)
    ctx = gp.gp_create(cfg, w.k_cache, w.v_cache, None)
    for _ in range(w.num_pages):
        gp.gp_page_alloc(ctx)
    used = set(t0) | set(w.block_tables[1])
    for pg in range(w.num_pages):
        if pg not in used:
            gp.gp_page_unref(ctx, pg)
    gp.gp_page_ref(ctx, t0[0])
    gp.gp_page_ref(ctx, t0[1])
    # keep only num_spare free pages
    held = []
    while gp.gp_free_page_count(ctx) > num_spare:
        held.append(gp.gp_page_alloc(ctx))
    reqs = [gp.Request(gp.gp_slot_acquire(ctx), w.block_tables[r], w.positions[r], cfg.max_pages_per_req)
            for r in range(2)]
    slots = torch.tensor([q.slot for q in reqs], dtype=torch.int32, device="cuda")
    first = torch.ones(2, dtype=torch.uint8, device="cuda")
    nfirst = torch.zeros(2, dtype=torch.uint8, device="cuda")
    for t, q in enumerate(w.history):
        gp.gp_update_summaries(ctx, 2, slots, q.contiguous(), first if t == 0 else nfirst)
    return w, ctx, reqs


def test_copy_on_write_of_a_shared_prefix():
    w, ctx, reqs = _two_sharing(num_spare=4)
    try:
        q = w.history[-1]
        a = reqs[0]
        shared = a.pages[:2]
        other_before = {pg: (w.k_cache[:, pg].clone(), w.v_cache[:, pg].clone()) for pg in reqs[1].pages}
        free_before = gp.gp_free_page_count(ctx)
        pool = og.PagePool(w.num_pages)
        pool.refcount = [gp.gp_page_refcount(ctx, pg) for pg in range(w.num_pages)]
        plan, replaced = og.cow_plan(list(a.pages), pool)
        assert sorted(replaced) == sorted(shared)
        pre = [(hz.unit_keys_dev(w.k_cache, a.pages, layer, h), hz.unit_keys_dev(w.v_cache, a.pages, layer, h))
               for layer in range(w.shape.num_layers) for h in range(w.shape.num_kv_heads)]
        gp.gp_boundary_demand(ctx, [a], q[:, :1].contiguous())
        gp.gp_compress_hold(ctx, [a])
        torch.cuda.synchronize()
        assert a.pages == plan, (a.pages, plan)
        for pg in shared:
            assert gp.gp_page_refcount(ctx, pg) == 1          # request 1's reference remains
        for pg in a.pages[:2]:
            assert gp.gp_page_refcount(ctx, pg) == 1
        assert gp.gp_free_page_count(ctx) == free_before - 2
        for pg, (kb, vb) in other_before.items():             # the sharer's bytes are untouched
            assert torch.equal(w.k_cache[:, pg], kb) and torch.equal(w.v_cache[:, pg], vb)
        units = w.shape.num_layers * w.shape.num_kv_heads
        keep = gp.unpack_mask(gp.gp_debug_keep_mask(ctx, 0, units, 4), 4 * PAGE)
        for u, (kp, vp) in enumerate(pre):
            layer, h = divmod(u, w.shape.num_kv_heads)
            kept = np.nonzero(keep[u])[0]
            n_live = 3 * PAGE
            assert np.array_equal(hz.unit_keys_dev(w.k_cache, a.pages, layer, h)[:n_live], kp[kept])
            assert np.array_equal(hz.unit_keys_dev(w.v_cache, a.pages, layer, h)[:n_live], vp[kept])
        st = gp.gp_stats(ctx)
        assert st["cow_pages"] == 2
    finally:
        gp.gp_destroy(ctx)


def test_no_pages_for_copy_on_write_changes_nothing():
    w, ctx, reqs = _two_sharing(num_spare=1)
    try:
        q = w.history[-1]
        a = reqs[0]
        table = list(a.pages)
        rc = [gp.gp_page_refcount(ctx, pg) for pg in range(w.num_pages)]
        kb, vb = w.k_cache.clone(), w.v_cache.clone()
        gp.gp_boundary_demand(ctx, [a], q[:, :1].contiguous())
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(ctx, [a])
        assert ei.value.status == gp.GP_ERR_NO_PAGES
        torch.cuda.synchronize()
        assert a.pages == table
        assert [gp.gp_page_refcount(ctx, pg) for pg in range(w.num_pages)] == rc
        assert torch.equal(w.k_cache, kb) and torch.equal(w.v_cache, vb)
    finally:
        gp.gp_destroy(ctx)


def test_compress_without_demand_is_a_state_error():
    w = _workload(SHAPES["bf16_g4_d128"], [3, 4], seed_xor=3)
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(run.ctx, [run.reqs[0]])
        assert ei.value.status == gp.GP_ERR_STATE
        # a demand call for the other request does not cover this one
        gp.gp_boundary_demand(run.ctx, [run.reqs[1]], w.history[-1][:, 1:].contiguous())
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(run.ctx, [run.reqs[0]])
        assert ei.value.status == gp.GP_ERR_STATE
        # after Grow the old demand no longer matches the request
        gp.gp_boundary_demand(run.ctx, [run.reqs[0]], w.history[-1][:, :1].contiguous())
        gp.gp_grow_page(run.ctx, run.reqs[0])
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_compress_hold(run.ctx, [run.reqs[0]])
        assert ei.value.status == gp.GP_ERR_STATE
    finally:
        run.close()


def test_caller_masks_of_the_wrong_size_are_refused():
    shape = SHAPES["bf16_g4_d128"]
    w = _workload(shape, [3], seed_xor=5)
    run = hz.EngineRun(w)
    try:
        req = run.reqs[0]
        P = req.num_pages
        units = run.units
        rng = np.random.default_rng(0)
        keep = np.zeros((units, P * PAGE), bool)
        for u in range(units):
            keep[u, rng.choice(P * PAGE, (P - 1) * PAGE, replace=False)] = True
        keep[1, np.nonzero(keep[1])[0][0]] = False          # one slot short in unit 1
        kb = w.k_cache.clone()
        words = torch.as_tensor(gp.pack_mask(keep).view(np.int32), device="cuda")
        gp.gp_compact_kv(run.ctx, [req], words)
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_debug_keep_mask(run.ctx, 0, units, P)       # synchronises, reports the count
        assert ei.value.status == gp.GP_ERR_INVALID
        # unit 1 was not moved; the others were compacted
        layer, h = divmod(1, shape.num_kv_heads)
        assert torch.equal(w.k_cache[layer, req.pages, h], kb[layer, req.pages, h])
        kept = np.nonzero(keep[0])[0]
        pre0 = kb[0, req.pages, 0].reshape(P * PAGE, -1)[torch.as_tensor(kept, device="cuda")]
        post0 = w.k_cache[0, req.pages, 0].reshape(P * PAGE, -1)[: (P - 1) * PAGE]
        assert torch.equal(pre0, post0)
    finally:
        run.close()
