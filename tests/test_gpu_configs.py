"""GPU parity at the full sizes of the batch configurations, through the C ABI.

* 64 requests of 4..128 pages (Llama-8B-like shape, shuffled shared pool,
  about 142 GB of K/V) and 16 requests of 128 pages (Qwen3-8B-like shape,
  36 layers, QK-normed, 30 % concentrated units, about 77 GB), all at a
  boundary in one gp_boundary_demand call -- the launch configuration of a
  real batch.
* The oracle computes sampled outputs one by one: D_p, the demand
  distributions and the importance of a few (layer, KV head) units of
  requests spread over every cluster shape; the decision of one whole small
  request; then Compress & Hold of every request (the paper's forced
  variant), with the keep masks and the gathered K/V bytes of the sampled
  units checked against the oracle's selection and gather.
"""

import gc

import numpy as np
import pytest
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256


def _sample_requests(w, count=6):
    sizes = [len(t) for t in w.block_tables]
    order = sorted(range(w.n), key=lambda r: sizes[r])
    picks = {order[0], order[-1]}
    for lo, hi in ((2, 32), (33, 64), (65, 127)):
        inside = [r for r in order if lo <= sizes[r] <= hi]
        if inside:
            picks.add(inside[len(inside) // 2])
    for r in order[:: max(1, w.n // 3)]:
        if len(picks) >= count:
            break
        picks.add(r)
    return sorted(picks)


def _sample_units(units, seed):
    rng = np.random.default_rng(seed)
    extra = rng.choice(np.arange(1, units - 1), 2, replace=False).tolist()
    return sorted({0, units - 1, *extra})


@pytest.fixture(scope="module", params=["batch64", "qwen3_8b"])
def loaded(request):
    name = request.param
    w = synth.make_workload(name, device="cuda")
    run = hz.EngineRun(w)
    run.feed_history()
    yield name, w, run
    run.close()
    del run, w
    gc.collect()
    torch.cuda.empty_cache()


def test_batch_demand_decide_compress_sampled(loaded):
    name, w, run = loaded
    sh = w.shape
    q = w.history[-1]
    dem = gp.gp_boundary_demand(run.ctx, run.reqs, q)
    picks = _sample_requests(w)
    checked = {}
    for r in picks:
        req = run.reqs[r]
        P = req.num_pages
        s, l = hz.oracle_summaries(w.history, r)
        qt = og.summary_queries(s, l, q[:, r].double().cpu().numpy(), req.pos, sh.rope_theta)
        ks = gp.gp_debug_demand_k(run.ctx, r, run.units)
        assert dem[r].sum_k_short == int(ks[:, 0].sum()) and dem[r].sum_k_long == int(ks[:, 1].sum())
        probs = gp.gp_debug_probs(run.ctx, r, run.units, (P - 1) * PAGE)
        scores = gp.gp_debug_scores(run.ctx, r, run.units, P * PAGE - 16)
        for idx in _sample_units(run.units, seed=r):
            layer, h = divmod(idx, sh.num_kv_heads)
            u = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group)
            for x in range(2):
                ok, msg = hz.dp_ok(int(ks[idx, x]), u.a_dem[x], 0.99)
                assert ok, f"{name} request {r} (P={P}) unit {idx} x {x}: {msg}"
            err = np.abs(probs[idx].astype(np.float64) - u.a_dem).max()
            assert err <= hz.PROB_ABS, f"{name} request {r} unit {idx}: probability error {err}"
            sg = np.exp2(scores[idx].astype(np.float64))
            big = u.s > 1e-30
            rel = np.abs(sg[big] - u.s[big]) / u.s[big]
            assert rel.max() < 2e-5, f"{name} request {r} unit {idx}: importance error {rel.max()}"
            checked[(r, idx)] = u
    # the decision of the smallest request, from every one of its units
    r0 = min(range(w.n), key=lambda r: run.reqs[r].num_pages)
    req = run.reqs[r0]
    P = req.num_pages
    s, l = hz.oracle_summaries(w.history, r0)
    qt = og.summary_queries(s, l, q[:, r0].double().cpu().numpy(), req.pos, sh.rope_theta)
    ks = gp.gp_debug_demand_k(run.ctx, r0, run.units)
    kk, ties = np.zeros((run.units, 2), np.int64), 0
    for idx in range(run.units):
        layer, h = divmod(idx, sh.num_kv_heads)
        u = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group)
        kk[idx] = u.k
        for x in range(2):
            ok, msg = hz.dp_ok(int(ks[idx, x]), u.a_dem[x], 0.99)
            assert ok, f"{name} request {r0} unit {idx} x {x}: {msg}"
            ties += int(ks[idx, x] != u.k[x])
    acts = gp.gp_decide(run.ctx, run.reqs, dem)
    if ties == 0:
        delta = og.demand_trend(kk[:, 0], kk[:, 1], (P - 1) * PAGE)
        # the free pool is ample for this request, so only Delta decides
        assert (acts[r0].kind == gp.GP_ACT_GROW) == (delta > 0.0) or acts[r0].fallback
    # Compress & Hold of every request (the forced-compress run)
    pre = {}
    for (r, idx), u in checked.items():
        layer, h = divmod(idx, sh.num_kv_heads)
        pre[(r, idx)] = (hz.unit_keys_dev(w.k_cache, run.reqs[r].pages, layer, h),
                         hz.unit_keys_dev(w.v_cache, run.reqs[r].pages, layer, h))
    tables = [list(x.pages) for x in run.reqs]
    gp.gp_compress_hold(run.ctx, run.reqs)
    torch.cuda.synchronize()
    assert [list(x.pages) for x in run.reqs] == tables       # no page is shared: no copy-on-write
    masks_by_req = {}
    for (r, idx), u in checked.items():
        req = run.reqs[r]
        P = req.num_pages
        if r not in masks_by_req:
            masks_by_req[r] = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, r, run.units, P), P * PAGE)
        keep = masks_by_req[r][idx]
        ok, _, msg = hz.topk_ok(keep, u.s, P)
        assert ok, f"{name} request {r} (P={P}) unit {idx}: {msg}"
        layer, h = divmod(idx, sh.num_kv_heads)
        kept = np.nonzero(keep)[0]
        n_live = (P - 1) * PAGE
        kp, vp = pre[(r, idx)]
        assert np.array_equal(hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:n_live], kp[kept])
        assert np.array_equal(hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:n_live], vp[kept])
