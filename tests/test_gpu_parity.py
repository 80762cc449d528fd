"""GPU parity of the C-ABI engine against the fp64 oracle (GrowPage boundary
engine).  Element-by-element on seeded synthetic inputs:

  * summaries (Eq. 6 + first-step init)      -- 1e-12 relative to the row RMS
  * a^S, a^L over C_t (softmax + GQA mean)   -- 1e-4 absolute
  * importance max(a^S, a^L) (Eq. 9)         -- 1e-4 absolute (and used for top-k)
  * D_p per (layer, KV head) (Eqs. 2, 7)     -- +-1 only at oracle ties with p (1e-6)
  * decision (Eq. 8, Sec. 4.2)               -- exact
  * keep masks (Eq. 10 + window)             -- exact up to 1e-5 score ties
  * compaction for a given index set         -- bit-exact bytes, tables exact
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


def _oracle_event(w, run, req_idx=0, q_cur=None, units_filter=None):
    """Oracle for one request at a boundary: summaries, qt, per-unit results."""
    req = run.reqs[req_idx]
    s, l = hz.oracle_summaries(w.history, req_idx)
    if q_cur is None:
        q_cur = w.history[-1]
    qc = q_cur[:, req_idx].double().cpu().numpy()
    qt = og.summary_queries(s, l, qc, req.pos, w.shape.rope_theta)
    pages = hz.cache_f64(w.k_cache, req.pages)
    G = w.shape.group
    res = {}
    for layer in range(w.shape.num_layers):
        for h in range(w.shape.num_kv_heads):
            idx = layer * w.shape.num_kv_heads + h
            if units_filter is not None and idx not in units_filter:
                continue
            res[idx] = hz.oracle_unit(qt, pages, req.pages, layer, h, G)
    return s, l, res


def _check_demand(run, req_idx, res, probs=None, scores=None):
    ks = gp.gp_debug_demand_k(run.ctx, req_idx, run.units)
    ties = 0
    for idx, u in res.items():
        for x in range(2):
            ok, msg = hz.dp_ok(int(ks[idx, x]), u.a_dem[x], 0.99)
            assert ok, f"unit {idx} x {x}: {msg}"
            ties += int(ks[idx, x] != u.k[x])
        if probs is not None:
            err = np.abs(probs[idx].astype(np.float64) - u.a_dem).max()
            assert err <= hz.PROB_ABS, f"unit {idx}: prob err {err}"
        if scores is not None:
            sg = np.exp2(scores[idx].astype(np.float64))
            err = np.abs(sg - u.s).max()
            assert err <= hz.PROB_ABS, f"unit {idx}: importance err {err}"
            # relative accuracy where it matters for ranking
            big = u.s > 1e-30
            rel = np.abs(sg[big] - u.s[big]) / u.s[big]
            assert rel.max() < 2e-5, f"unit {idx}: importance rel err {rel.max()}"
    return ks, ties


def _gathered_ok(pre_k, pre_v, post_k, post_v, old_table, new_table, keep, L, hkv):
    """Post-compaction caches hold pre[kept slots] in order (bit-exact)."""
    P = len(old_table)
    n = P * PAGE
    dev = post_k.device
    old_t = torch.as_tensor(old_table, device=dev)
    new_t = torch.as_tensor(new_table, device=dev)
    keep_t = torch.as_tensor(keep, device=dev)
    for layer in range(L):
        for h in range(hkv):
            u = layer * hkv + h
            idx = torch.nonzero(keep_t[u, :n]).flatten()
            for pre, post in ((pre_k, post_k), (pre_v, post_v)):
                src = pre[layer, old_t, h].reshape(n, -1)[idx]
                dst = post[layer, new_t, h].reshape(n, -1)[: (P - 1) * PAGE]
                ity = torch.int16 if src.element_size() == 2 else torch.int32
                if not torch.equal(src.view(ity), dst.view(ity)):
                    return False, (layer, h)
    return True, None


@pytest.mark.parametrize("variant", ["grow", "compress"])
def test_tiny_boundary_event(variant):
    w = synth.make_workload("tiny", device="cuda", variant=variant)
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        req = run.reqs[0]
        P = req.num_pages
        sh = w.shape
        s, l, res = _oracle_event(w, run)
        gs = gp.gp_read_summaries(run.ctx, req.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
        assert hz.summaries_ok(gs[:, 0], s) <= hz.SUMMARY_REL
        assert hz.summaries_ok(gs[:, 1], l) <= hz.SUMMARY_REL
        dem = gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
        probs = gp.gp_debug_probs(run.ctx, 0, run.units, (P - 1) * PAGE)
        scores = gp.gp_debug_scores(run.ctx, 0, run.units, P * PAGE - 16)
        ks, _ = _check_demand(run, 0, res, probs, scores)
        kk = np.array([res[i].k for i in range(run.units)])
        assert dem[0].sum_k_short == ks[:, 0].sum() and dem[0].sum_k_long == ks[:, 1].sum()
        delta = og.demand_trend(kk[:, 0], kk[:, 1], (P - 1) * PAGE)
        ref = og.decide(delta, P, gp.gp_free_page_count(run.ctx), 0, 0.0)
        act = gp.gp_decide(run.ctx, run.reqs, dem)[0]
        assert act.kind == ref.kind == (og.GROW if variant == "grow" else og.COMPRESS)
        if act.kind == gp.GP_ACT_COMPRESS:
            pre_k, pre_v = w.k_cache.clone(), w.v_cache.clone()
            old = req.pages
            gp.gp_compress_hold(run.ctx, run.reqs)
            masks = gp.gp_debug_keep_mask(run.ctx, 0, run.units, P)
            keep = gp.unpack_mask(masks, P * PAGE)
            for idx, u in res.items():
                ok, nd, msg = hz.topk_ok(keep[idx], u.s, P)
                assert ok, f"unit {idx}: {msg}"
            torch.cuda.synchronize()
            ok, where = _gathered_ok(pre_k, pre_v, w.k_cache, w.v_cache, old, req.pages, keep,
                                     sh.num_layers, sh.num_kv_heads)
            assert ok, where
            assert req.pages == old and req.num_pages == P
        else:
            gp.gp_grow_page(run.ctx, req)
            assert req.num_pages == P + 1
    finally:
        run.close()


def test_tiny_compaction_with_oracle_masks_is_bit_exact():
    w = synth.make_workload("tiny", device="cuda", variant="compress")
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        req = run.reqs[0]
        P = req.num_pages
        sh = w.shape
        _, _, res = _oracle_event(w, run)
        keep = np.zeros((run.units, P * PAGE), bool)
        for idx, u in res.items():
            keep[idx] = og.select_retained(u.s, P, PAGE, 16, 64)
        kd = torch.as_tensor(gp.pack_mask(keep).view(np.int32), device="cuda")
        pre_k = w.k_cache.double().cpu().numpy()
        pre_v = w.v_cache.double().cpu().numpy()
        old = req.pages
        gp.gp_compact_kv(run.ctx, run.reqs, kd)
        torch.cuda.synchronize()
        masks = keep.reshape(sh.num_layers, sh.num_kv_heads, -1)
        ek, ev = og.compress_cache(pre_k, pre_v, old, req.pages, masks, PAGE)
        got_k = w.k_cache.double().cpu().numpy()
        got_v = w.v_cache.double().cpu().numpy()
        n_live = (P - 1) * PAGE
        for layer in range(sh.num_layers):
            for h in range(sh.num_kv_heads):
                for exp, got in ((ek, got_k), (ev, got_v)):
                    e = og.gather_logical(exp, req.pages, layer, h)[:n_live]
                    g = og.gather_logical(got, req.pages, layer, h)[:n_live]
                    assert np.array_equal(e, g)
        st = gp.gp_stats(run.ctx)
        assert st["moved_rows"] > 0
    finally:
        run.close()


def test_llama_single_boundary_event():
    """Config 2 shape (32L, 32q/8kv, d128, bf16, 32 pages): one full event."""
    w = synth.make_workload("llama8b_single", device="cuda")
    run = hz.EngineRun(w)
    try:
        # a short history: 48 concentrated steps then 16 diffuse ones
        for t in range(64):
            w.history.append(synth.query_step(w, [t < 48]))
        run.feed_history()
        req = run.reqs[0]
        P = req.num_pages
        sh = w.shape
        s, l, res = _oracle_event(w, run)
        gs = gp.gp_read_summaries(run.ctx, req.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
        assert hz.summaries_ok(gs[:, 0], s) <= hz.SUMMARY_REL
        assert hz.summaries_ok(gs[:, 1], l) <= hz.SUMMARY_REL
        dem = gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
        probs = gp.gp_debug_probs(run.ctx, 0, run.units, (P - 1) * PAGE)
        scores = gp.gp_debug_scores(run.ctx, 0, run.units, P * PAGE - 16)
        ks, ties = _check_demand(run, 0, res, probs, scores)
        kk = np.array([res[i].k for i in range(run.units)])
        act = gp.gp_decide(run.ctx, run.reqs, dem)[0]
        ok, msg = hz.decision_ok(act, kk, ks, P, gp.gp_free_page_count(run.ctx))
        assert ok, msg
        # Compress & Hold regardless of the decision, to check selection + bytes
        pre_k, pre_v = w.k_cache.clone(), w.v_cache.clone()
        old = req.pages
        gp.gp_compress_hold(run.ctx, run.reqs)
        masks = gp.gp_debug_keep_mask(run.ctx, 0, run.units, P)
        keep = gp.unpack_mask(masks, P * PAGE)
        ndiff = 0
        for idx, u in res.items():
            ok, nd, msg = hz.topk_ok(keep[idx], u.s, P)
            assert ok, f"unit {idx}: {msg}"
            ndiff += nd
        torch.cuda.synchronize()
        ok, where = _gathered_ok(pre_k, pre_v, w.k_cache, w.v_cache, old, req.pages, keep,
                                 sh.num_layers, sh.num_kv_heads)
        assert ok, where
    finally:
        run.close()
