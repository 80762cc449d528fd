"""The entropy metric of the dual-timescale ablation (GrowPage Sec. 5.3,
Table 2) through the C ABI, against the fp64 oracle.

With demand_metric = ENTROPY the engine reports, per (layer, KV head) and
summary, the effective support size exp(H(a^x)) of the demand distribution
over C_t, sums them per request, and decides on
Delta = (sum E^S - sum E^L) / (|C_t| L Hkv).

Tolerance of exp(H): 1e-4 relative.  The GPU's a-values carry a relative
error of about 1e-6 (fp32 exponentials and sums of up to 41k terms); H
moves by at most that times (H + 1), and H <= ln 41k < 11, so exp(H) moves
by about 1.2e-5 relative; the fp32 terms a ln a add about 1e-7.  The
decision must equal the oracle's unless the oracle's Delta is within 2e-4
relative of the support sizes of tau (the bound the 1e-4 tolerance allows).
"""

import numpy as np
import pytest

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth
from synth.workloads import ModelShape

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256
EFF_REL = 1e-4


def _oracle_support(w, run, r):
    """exp(H(a^x)) per unit from the oracle's own demand distributions."""
    req = run.reqs[r]
    s, l = hz.oracle_summaries(w.history, r)
    qc = w.history[-1][:, r].double().cpu().numpy()
    qt = og.summary_queries(s, l, qc, req.pos, w.shape.rope_theta)
    G, hkv = w.shape.group, w.shape.num_kv_heads
    eff = np.zeros((run.units, 2))
    for layer in range(w.shape.num_layers):
        for h in range(hkv):
            u = hz.oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, G)
            for x in range(2):
                eff[layer * hkv + h, x] = og.entropy_support(u.a_dem[x])
    return eff


def _check_event(w, run):
    dem = gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
    free = gp.gp_free_page_count(run.ctx)
    acts = gp.gp_decide(run.ctx, run.reqs, dem)
    granted, decided = 0, 0
    for r, req in enumerate(run.reqs):
        P = req.num_pages
        cand = (P - 1) * PAGE
        got = gp.gp_debug_entropy(run.ctx, r, run.units)
        ref = _oracle_support(w, run, r)
        rel = np.abs(got - ref) / ref
        assert rel.max() <= EFF_REL, f"request {r}: exp(H) rel err {rel.max()} at {np.unravel_index(rel.argmax(), rel.shape)}"
        # the request sums and Delta are formed from the per-unit values
        assert dem[r].eff_short == pytest.approx(got[:, 0].sum(), rel=1e-12)
        assert dem[r].eff_long == pytest.approx(got[:, 1].sum(), rel=1e-12)
        delta_ref = og.demand_trend(ref[:, 0], ref[:, 1], cand)
        margin = 2 * EFF_REL * (ref.sum() / (cand * run.units))
        assert abs(dem[r].delta - delta_ref) <= margin
        if abs(delta_ref) > margin:
            want = og.decide(delta_ref, P, free - granted, 0, 0.0)
            assert acts[r].kind == want.kind and bool(acts[r].fallback) == want.fallback, (r, delta_ref)
            decided += 1
        granted += int(acts[r].kind == gp.GP_ACT_GROW and not acts[r].forced)
    return dem, acts, decided


@pytest.mark.parametrize("variant", ["grow", "compress"])
def test_entropy_metric_tiny(variant):
    """fp32 caches: the CUDA-core scan's a-values."""
    w = synth.make_workload("tiny", device="cuda", variant=variant)
    run = hz.EngineRun(w, demand_metric=gp.GP_METRIC_ENTROPY)
    base = hz.EngineRun(synth.make_workload("tiny", device="cuda", variant=variant))
    try:
        run.feed_history()
        base.feed_history()
        dem, _, decided = _check_event(w, run)
        assert decided == 1
        # the D_p side is untouched by the metric; TOP_P reports no support sizes
        ref = gp.gp_boundary_demand(base.ctx, base.reqs, base.w.history[-1])
        assert (dem[0].sum_k_short, dem[0].sum_k_long) == (ref[0].sum_k_short, ref[0].sum_k_long)
        assert ref[0].eff_short == 0.0 and ref[0].eff_long == 0.0
        with pytest.raises(gp.GrowPageError):
            gp.gp_debug_entropy(base.ctx, 0, base.units)
    finally:
        run.close()
        base.close()


def test_entropy_metric_bf16_batch():
    """bf16 caches: the tensor-core scan (P <= 160) and the CUDA-core scan
    (P > 160) in one call, ragged request sizes."""
    sh = ModelShape(2, 8, 2, 128, "bf16", "bf16", 5.0e5)
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=[2, 9, 33, 161], seed_xor=51)
    run = hz.EngineRun(w, demand_metric=gp.GP_METRIC_ENTROPY)
    try:
        run.feed_history()
        _check_event(w, run)
    finally:
        run.close()


def test_noalloc_refuses_the_entropy_metric():
    w = synth.make_workload("tiny", device="cuda", variant="grow")
    run = hz.EngineRun(w, demand_metric=gp.GP_METRIC_ENTROPY)
    try:
        run.feed_history()
        with pytest.raises(gp.GrowPageError):
            gp.gp_boundary_demand_noalloc(run.ctx, run.reqs, w.history[-1])
    finally:
        run.close()
