"""GPU parity at the full sizes of the batch configurations, through the C ABI.

* 64 requests of 4..128 pages (Llama-8B-like shape, shuffled shared pool,
  about 142 GB of K/V) and 16 requests of 128 pages (Qwen3-8B-like shape,
  36 layers, QK-normed, 30 % concentrated units, about 77 GB), all at a
  boundary in one gp_boundary_demand call -- the launch configuration of a
  real batch.
* The oracle checks D_p of every (layer, KV head) unit of every request
  (Eqs. 2, 7; the tie rule) and the decision of every request (Eq. 8 and the
  rule after it, with the tie window), on a thread pool over the host cores.
  The demand distributions and the importance are compared element by
  element on a sample of units of every request; then Compress & Hold of
  every request (the paper's forced variant), with the keep masks (Eq. 10)
  and the gathered K/V bytes of one whole request per page-count band and of
  the sampled units of the others.
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
BANDS = ((2, 32), (33, 64), (65, 127), (128, 256))


def _whole_requests(w):
    """One request per page-count band (the middle one of the band)."""
    sizes = [len(t) for t in w.block_tables]
    picks = []
    for lo, hi in BANDS:
        inside = sorted((r for r in range(w.n) if lo <= sizes[r] <= hi), key=lambda r: sizes[r])
        if inside:
            picks.append(inside[len(inside) // 2])
    return picks


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


def test_batch_every_unit_and_decision_then_compress(loaded):
    name, w, run = loaded
    sh = w.shape
    q = w.history[-1]
    dem = gp.gp_boundary_demand(run.ctx, run.reqs, q)
    acts = gp.gp_decide(run.ctx, run.reqs, dem)
    free = gp.gp_free_page_count(run.ctx)
    whole = _whole_requests(w)
    granted = 0
    checked = {}            # (r, unit) -> oracle importance over C_cmp
    for r in range(w.n):
        req = run.reqs[r]
        P = req.num_pages
        s, l = hz.oracle_summaries(w.history, r)
        qt = og.summary_queries(s, l, q[:, r].double().cpu().numpy(), req.pos, sh.rope_theta)
        ks = gp.gp_debug_demand_k(run.ctx, r, run.units)
        assert dem[r].sum_k_short == int(ks[:, 0].sum()) and dem[r].sum_k_long == int(ks[:, 1].sum())
        sample = _sample_units(run.units, seed=r)
        keep_ids = range(run.units) if r in whole else sample
        k_or, fails, kept = hz.request_dp_check(w, req, qt, ks, keep=keep_ids)
        assert not fails, f"{name} request {r} (P={P}): {len(fails)} units, e.g. {fails[:3]}"
        ok, msg = hz.decision_ok(acts[r], k_or, ks, P, free - granted)
        assert ok, f"{name} request {r} (P={P}): {msg}"
        if acts[r].kind == gp.GP_ACT_GROW and not acts[r].forced:
            granted += 1
        probs = gp.gp_debug_probs(run.ctx, r, run.units, (P - 1) * PAGE)
        scores = gp.gp_debug_scores(run.ctx, r, run.units, P * PAGE - 16)
        for idx in sample:
            u = kept[idx]
            err = np.abs(probs[idx].astype(np.float64) - u.a_dem).max()
            assert err <= hz.PROB_ABS, f"{name} request {r} unit {idx}: probability error {err}"
            sg = np.exp2(scores[idx].astype(np.float64))
            big = u.s > 1e-30
            rel = np.abs(sg[big] - u.s[big]) / u.s[big]
            assert rel.max() < 2e-5, f"{name} request {r} unit {idx}: importance error {rel.max()}"
        for idx, u in kept.items():
            checked[(r, idx)] = u.s
        del kept, probs, scores
    # Compress & Hold of every request (the forced-compress run).  Snapshot the
    # checked units' K/V (bf16 bit patterns) first.
    pre = {}
    for (r, idx) in checked:
        layer, h = divmod(idx, sh.num_kv_heads)
        pre[(r, idx)] = (_unit_bits(w.k_cache, run.reqs[r].pages, layer, h),
                         _unit_bits(w.v_cache, run.reqs[r].pages, layer, h))
    tables = [list(x.pages) for x in run.reqs]
    gp.gp_compress_hold(run.ctx, run.reqs)
    torch.cuda.synchronize()
    assert [list(x.pages) for x in run.reqs] == tables       # no page is shared: no copy-on-write
    masks_by_req = {}
    for r in sorted({r for r, _ in checked}):
        P = run.reqs[r].num_pages
        masks_by_req[r] = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, r, run.units, P), P * PAGE)

    def one(key):
        r, idx = key
        req = run.reqs[r]
        P = req.num_pages
        keep = masks_by_req[r][idx]
        ok, _, msg = hz.topk_ok(keep, checked[key], P)
        if not ok:
            return f"request {r} (P={P}) unit {idx}: {msg}"
        layer, h = divmod(idx, sh.num_kv_heads)
        n_live = (P - 1) * PAGE
        kp, vp = pre[key]
        if not np.array_equal(_unit_bits(w.k_cache, req.pages, layer, h)[:n_live], og.compact_unit(kp, keep)):
            return f"request {r} unit {idx}: K bytes differ from the oracle's gather"
        if not np.array_equal(_unit_bits(w.v_cache, req.pages, layer, h)[:n_live], og.compact_unit(vp, keep)):
            return f"request {r} unit {idx}: V bytes differ from the oracle's gather"
        return None

    bad = [m for m in hz.oracle_pool().map(one, sorted(checked)) if m]
    assert not bad, f"{name}: {len(bad)} units, e.g. {bad[:3]}"


def _unit_bits(cache, table, layer, h):
    """Raw bit patterns of one unit's rows in logical order (host)."""
    idx = torch.as_tensor(list(table), device=cache.device, dtype=torch.long)
    sub = cache[layer].index_select(0, idx)[:, h]
    view = torch.int16 if sub.dtype == torch.bfloat16 else torch.int32
    return sub.contiguous().view(view).cpu().numpy().reshape(len(table) * PAGE, -1)
