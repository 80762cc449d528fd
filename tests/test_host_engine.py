"""CPU tests of the C-ABI library: it loads, exports every declared symbol,
its structs match the header, and the host-side logic (page pool with
refcounts, slots, decision, Grow) behaves as the oracle's model says.
No compute call touches a GPU here: the contexts are host-only."""

import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "growpage.h")


@pytest.fixture(scope="module")
def lib():
    return gp.load()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:gp_status|const char\*)\s+(gp_\w+)\s*\(", txt, re.M)))


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", gp.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(gp_\w+)", out))
    missing = [d for d in declared if d not in exported]
    assert not missing, missing
    assert set(declared) == set(gp.EXPORTS)
    for name in declared:
        getattr(lib, name)


def test_struct_layout_matches_header():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "growpage.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(gp_config), offsetof(gp_config, beta_s),
         offsetof(gp_config, rope_theta), sizeof(gp_request), offsetof(gp_request, pos),
         sizeof(gp_demand), sizeof(gp_action), sizeof(gp_stats_t), offsetof(gp_config, shrink_threshold),
         offsetof(gp_config, random_seed), offsetof(gp_stats_t, shrink), offsetof(gp_config, demand_metric),
         offsetof(gp_demand, eff_long));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        vals = list(map(int, subprocess.run([exe], capture_output=True, text=True,
                                            check=True).stdout.split()))
    import ctypes as C
    ref = [C.sizeof(gp.GpConfig), gp.GpConfig.beta_s.offset, gp.GpConfig.rope_theta.offset,
           C.sizeof(gp.GpRequest), gp.GpRequest.pos.offset, C.sizeof(gp.GpDemand),
           C.sizeof(gp.GpAction), C.sizeof(gp.GpStats), gp.GpConfig.shrink_threshold.offset,
           gp.GpConfig.random_seed.offset, gp.GpStats.shrink.offset, gp.GpConfig.demand_metric.offset,
           gp.GpDemand.eff_long.offset]
    assert vals == ref


def _host_ctx(num_pages=16, **over):
    cfg = gp.gp_config_default(num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
                               max_slots=8, num_pages=num_pages, max_pages_per_req=8)
    for k, v in over.items():
        setattr(cfg, k, v)
    return gp.gp_create(cfg)


def test_config_validation():
    bad = [dict(head_dim=96), dict(page_size=128), dict(num_q_heads=6), dict(p=1.0),
           dict(beta_s=1.0), dict(max_pages_per_req=300), dict(recent_window=256),
           dict(num_q_heads=16)]
    for over in bad:
        with pytest.raises(gp.GrowPageError):
            _host_ctx(**over)


def test_page_pool_matches_oracle_model():
    ctx = _host_ctx(12)
    model = og.PagePool(12)
    rng = np.random.default_rng(0)
    owned = []
    try:
        for step in range(400):
            op = rng.integers(3)
            if op == 0:
                if model.free_count() == 0:
                    with pytest.raises(gp.GrowPageError) as ei:
                        gp.gp_page_alloc(ctx)
                    assert ei.value.status == gp.GP_ERR_NO_PAGES
                else:
                    a = gp.gp_page_alloc(ctx)
                    assert a == model.alloc()          # lowest free id first
                    owned.append(a)
            elif op == 1 and owned:
                p = owned[rng.integers(len(owned))]
                gp.gp_page_ref(ctx, p)
                model.ref(p)
                owned.append(p)
            elif op == 2 and owned:
                p = owned.pop(rng.integers(len(owned)))
                gp.gp_page_unref(ctx, p)
                model.unref(p)
            assert gp.gp_free_page_count(ctx) == model.free_count()
            for p in range(12):
                assert gp.gp_page_refcount(ctx, p) == model.refcount[p]
            # conservation: references held == sum of refcounts
            assert sum(model.refcount) == len(owned)
        with pytest.raises(gp.GrowPageError):
            gp.gp_page_unref(ctx, 11 if model.refcount[11] == 0 else -1)
    finally:
        gp.gp_destroy(ctx)


def test_slots_lowest_first_and_release():
    ctx = _host_ctx()
    try:
        got = [gp.gp_slot_acquire(ctx) for _ in range(8)]
        assert got == list(range(8))
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_slot_acquire(ctx)
        assert ei.value.status == gp.GP_ERR_NO_SLOTS
        gp.gp_slot_release(ctx, 3)
        with pytest.raises(gp.GrowPageError):
            gp.gp_slot_release(ctx, 3)
        assert gp.gp_slot_acquire(ctx) == 3
    finally:
        gp.gp_destroy(ctx)


def _demand(sk, sl, P, units=4):
    d = gp.GpDemand()
    d.sum_k_short, d.sum_k_long = sk, sl
    d.num_candidates = (P - 1) * 256
    d.num_units = units
    d.delta = (sk - sl) / (d.num_candidates * units) if P > 1 else 0.0
    return d


def test_decide_matches_oracle_rules():
    rng = np.random.default_rng(1)
    for trial in range(200):
        free = int(rng.integers(0, 4))
        reserve = int(rng.integers(0, 2))
        tau = float(rng.choice([0.0, 0.001, -0.001]))
        policy = int(rng.integers(2))
        ctx = _host_ctx(num_pages=8, reserve_pages=reserve, tau=tau, policy=policy)
        try:
            for _ in range(8 - free):
                gp.gp_page_alloc(ctx)
            n = int(rng.integers(1, 5))
            reqs, dem, ref = [], [], []
            granted = 0
            for r in range(n):
                P = int(rng.integers(1, 5))
                sk, sl = int(rng.integers(0, 2000)), int(rng.integers(0, 2000))
                if trial % 7 == 0:
                    sl = sk                       # Delta = 0 compresses
                reqs.append(gp.Request(r, [0] * P, 0, 8))
                d = _demand(sk, sl, P)
                dem.append(d)
                a = og.decide(d.delta, P, free - granted, reserve, tau,
                              policy="growpage" if policy == 0 else "fixed")
                if a.kind == og.GROW and not a.forced:
                    granted += 1
                ref.append(a)
            acts = gp.gp_decide(ctx, reqs, dem)
            for a, b in zip(acts, ref):
                assert (a.kind, bool(a.fallback), bool(a.forced)) == (b.kind, b.fallback, b.forced)
        finally:
            gp.gp_destroy(ctx)


def test_grow_appends_lowest_free_and_never_touches_prefix():
    ctx = _host_ctx(num_pages=6)
    try:
        pages = [gp.gp_page_alloc(ctx) for _ in range(3)]   # 0,1,2
        gp.gp_page_ref(ctx, 0)                              # shared prefix page
        slot = gp.gp_slot_acquire(ctx)
        req = gp.Request(slot, pages, 768, 4)
        gp.gp_grow_page(ctx, req)
        assert req.pages == [0, 1, 2, 3]
        assert gp.gp_page_refcount(ctx, 0) == 2 and gp.gp_page_refcount(ctx, 3) == 1
        with pytest.raises(gp.GrowPageError):               # block table full
            gp.gp_grow_page(ctx, req)
        assert req.num_pages == 4
        req2 = gp.Request(slot, [gp.gp_page_alloc(ctx)], 0, 4)   # page 4
        gp.gp_grow_page(ctx, req2)                          # takes page 5
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_grow_page(ctx, req2)
        assert ei.value.status == gp.GP_ERR_NO_PAGES and req2.pages == [4, 5]
        # the C side enforces max_pages_per_req
        ctx2 = _host_ctx(num_pages=16, max_pages_per_req=2)
        try:
            r3 = gp.Request(0, [gp.gp_page_alloc(ctx2), gp.gp_page_alloc(ctx2)], 0, 8)
            with pytest.raises(gp.GrowPageError) as ei:
                gp.gp_grow_page(ctx2, r3)
            assert ei.value.status == gp.GP_ERR_INVALID and r3.num_pages == 2
        finally:
            gp.gp_destroy(ctx2)
    finally:
        gp.gp_destroy(ctx)


def test_host_only_context_refuses_device_calls():
    ctx = _host_ctx()
    try:
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_update_summaries(ctx, 1, 0, 0, 0)
        assert ei.value.status == gp.GP_ERR_STATE
        with pytest.raises(gp.GrowPageError) as ei:
            gp.gp_boundary_demand(ctx, [gp.Request(0, [0], 0, 8)], 0)
        assert ei.value.status == gp.GP_ERR_STATE
        # every other call that touches the device is refused the same way, before any work
        req = [gp.Request(0, [0, 1], 256, 8)]
        calls = [
            lambda: gp.gp_boundary_demand_noalloc(ctx, req, 0),
            lambda: gp.gp_compress_hold(ctx, req),
            lambda: gp.gp_shrink(ctx, req),
            lambda: gp.gp_compress_fill(ctx, req),
            lambda: gp.gp_decode_attention(ctx, 0, req, [256], 0, 0, 0),
            lambda: gp.gp_set_compaction_stream(ctx, None),
            lambda: gp.gp_wait_compaction(ctx, None),
            lambda: gp.gp_debug_probs(ctx, 0, 4, 256),
            lambda: gp.gp_read_summaries(ctx, 0, 2, 4, 64),
        ]
        for i, call in enumerate(calls):
            with pytest.raises(gp.GrowPageError) as ei:
                call()
            assert ei.value.status == gp.GP_ERR_STATE, i
        assert req[0].pages == [0, 1] and req[0].num_pages == 2   # tables untouched
    finally:
        gp.gp_destroy(ctx)


@pytest.mark.parametrize("n", [1, 5, 20])
def test_request_marshalling_matches_the_c_struct(n):
    """The binding packs gp_request fields with struct; read back through the
    ctypes field descriptors they are the requests' own values, and
    num_pages written by the C side comes back to each request (both
    read-back paths: up to 8 requests and more)."""
    import ctypes as C
    from paged_kv_cache_step_gb300 import binding as bd
    rng = np.random.default_rng(n)
    reqs = [gp.Request(int(rng.integers(0, 512)), list(rng.integers(0, 1000, int(rng.integers(1, 9)))),
                       int(rng.integers(0, 1 << 40)), 16) for _ in range(n)]
    arr = bd._marshal(reqs)
    for i, r in enumerate(reqs):
        assert arr[i].slot == r.slot and arr[i].num_pages == r.num_pages and arr[i].pos == r.pos
        assert C.cast(arr[i].block_table, C.c_void_p).value == r.table.ctypes.data
        assert arr[i].block_table[r.num_pages - 1] == r.pages[-1]
    for i in range(n):
        arr[i].num_pages = i + 1
    bd._unmarshal(arr, reqs)
    assert [r.num_pages for r in reqs] == list(range(1, n + 1))


def test_mask_pack_roundtrip():
    rng = np.random.default_rng(2)
    keep = rng.random((3, 512)) < 0.5
    assert np.array_equal(gp.unpack_mask(gp.pack_mask(keep), 512), keep)


POLICIES = {"growpage": gp.GP_POLICY_GROWPAGE, "fixed": gp.GP_POLICY_FIXED, "random": gp.GP_POLICY_RANDOM,
            "inverse": gp.GP_POLICY_INVERSE, "shrink": gp.GP_POLICY_SHRINK}


@pytest.mark.parametrize("policy", sorted(POLICIES))
def test_decide_policies_match_oracle(policy):
    """Every policy of App. H.1 against the oracle's rules, over random sums,
    sizes and pool states; the random policy's draws follow the decision
    counter, so the oracle replays them from its own generator."""
    rng = np.random.default_rng(11)
    ctx = _host_ctx(num_pages=64, policy=POLICIES[policy], random_seed=5)
    try:
        units, k = 8, 0
        for trial in range(60):
            n = int(rng.integers(1, 9))
            reqs, dem = [], []
            for i in range(n):
                P = int(rng.integers(1, 9))
                reqs.append(gp.Request(i, list(range(P)), P * 256, 8))
                cand = (P - 1) * 256
                d = gp.GpDemand()
                d.num_candidates, d.num_units = cand, units
                # Delta spread over the zones of Eq. 13 (and exactly 0)
                delta = float(rng.choice([0.0, -0.005, 0.02, -0.02, rng.normal(0, 0.01)]))
                base = int(rng.integers(0, cand * units + 1)) if cand else 0
                d.sum_k_long = base
                d.sum_k_short = base + int(round(delta * cand * units))
                d.delta = 0.0
                dem.append(d)
            free = gp.gp_free_page_count(ctx)
            acts = gp.gp_decide(ctx, reqs, dem)
            granted = 0
            for r, (q, d, a) in enumerate(zip(reqs, dem, acts)):
                P = q.num_pages
                delta = (d.sum_k_short - d.sum_k_long) / (d.num_candidates * d.num_units) if P > 1 else 0.0
                ref = og.decide(delta, P, free - granted, 0, 0.0, policy=policy, draw=og.policy_draw(5, k))
                k += 1
                assert (a.kind, bool(a.fallback), bool(a.forced)) == (ref.kind, ref.fallback, ref.forced), \
                    (policy, trial, r, P, delta)
                granted += int(a.kind == gp.GP_ACT_GROW and not a.forced)
        st = gp.gp_stats(ctx)
        assert st["grow"] + st["compress"] + st["shrink"] == k
        if policy == "shrink":
            assert st["shrink"] > 0
        if policy == "random":
            assert 0.55 < st["compress"] / max(1, k - st["forced_grow"]) < 0.85
    finally:
        gp.gp_destroy(ctx)


def test_policy_config_validation():
    for bad in (dict(policy=9), dict(random_compress=1.5), dict(shrink_floor_pages=1),
                dict(shrink_threshold=float("nan")), dict(demand_metric=2), dict(demand_metric=-1)):
        with pytest.raises(gp.GrowPageError):
            _host_ctx(**bad)


@pytest.mark.parametrize("policy", ["growpage", "inverse", "shrink"])
def test_decide_entropy_metric_matches_oracle(policy):
    """Under the entropy metric (Sec. 5.3 ablation) Delta comes from the
    effective support sizes exp(H(a^x)) summed over the units, compared with
    tau in double; the D_p sums are ignored.  Against the oracle's rules."""
    rng = np.random.default_rng(12)
    for tau in (0.0, 0.01):
        ctx = _host_ctx(num_pages=64, policy=POLICIES[policy], demand_metric=gp.GP_METRIC_ENTROPY, tau=tau)
        try:
            units = 8
            for trial in range(40):
                n = int(rng.integers(1, 6))
                reqs, dem = [], []
                for i in range(n):
                    P = int(rng.integers(1, 9))
                    reqs.append(gp.Request(i, list(range(P)), P * 256, 8))
                    cand = (P - 1) * 256
                    d = gp.GpDemand()
                    d.num_candidates, d.num_units = cand, units
                    e_l = rng.uniform(1.0, max(cand, 1), units)
                    e_s = np.clip(e_l * rng.choice([1.0, 0.5, 1.5, rng.uniform(0.9, 1.1)]), 1.0, max(cand, 1))
                    d.eff_short, d.eff_long = float(e_s.sum()), float(e_l.sum())
                    # D_p sums that would decide the other way: the entropy metric must ignore them
                    d.sum_k_short, d.sum_k_long = (0, 10 ** 6) if e_s.sum() > e_l.sum() else (10 ** 6, 0)
                    dem.append(d)
                free = gp.gp_free_page_count(ctx)
                acts = gp.gp_decide(ctx, reqs, dem)
                granted = 0
                for r, (q, d, a) in enumerate(zip(reqs, dem, acts)):
                    P = q.num_pages
                    delta = og.demand_trend([d.eff_short], [d.eff_long], d.num_candidates * d.num_units) \
                        if P > 1 else 0.0
                    ref = og.decide(delta, P, free - granted, 0, tau, policy=policy)
                    assert (a.kind, bool(a.fallback), bool(a.forced)) == (ref.kind, ref.fallback, ref.forced), \
                        (policy, tau, trial, r, P, delta)
                    granted += int(a.kind == gp.GP_ACT_GROW and not a.forced)
        finally:
            gp.gp_destroy(ctx)


def test_host_only_context_refuses_entropy_readback():
    ctx = _host_ctx(demand_metric=gp.GP_METRIC_ENTROPY)
    try:
        with pytest.raises(gp.GrowPageError):
            gp.gp_debug_entropy(ctx, 0, 4)
    finally:
        gp.gp_destroy(ctx)


def test_config_defaults_are_the_papers():
    """gp_config_default against the values the pages fix: 256-token blocks
    and the 16-token recent window (Sec. 5.1), the per-block quota
    k_loc = 64 (App. D.2), p = 0.99 (Sec. 3.2), beta_S = 0.9 and
    beta_L = 0.999 (the default row of Table 2, Sec. 5.3), tau = 0 (Grow iff
    Delta > 0, Sec. 3.2), 512 summary slots (App. E.1 Eq. 11), Random(0.7),
    the Shrink threshold -0.005 of Eq. 13 and its 1024-token floor
    (App. H.1), and the Top-p working-set metric."""
    cfg = gp.gp_config_default()
    assert (cfg.page_size, cfg.recent_window, cfg.k_loc) == (256, 16, 64)
    assert (cfg.beta_s, cfg.beta_l, cfg.p, cfg.tau) == (0.9, 0.999, 0.99, 0.0)
    assert cfg.max_slots == 512
    assert cfg.policy == gp.GP_POLICY_GROWPAGE and cfg.demand_metric == gp.GP_METRIC_TOP_P
    assert cfg.random_compress == 0.7 and cfg.shrink_threshold == -0.005
    assert cfg.shrink_floor_pages * cfg.page_size == 1024
    assert cfg.reserve_pages == 0
