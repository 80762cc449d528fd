"""GPU parity of the continuous-batching stream at full size, through the C ABI.

256 seats of the Llama-8B-like shape in 32 prefix groups of 8 sharing a
32-page prefix, lognormal private parts, about 1/8 of the live requests at a
boundary each step, 1000 decode steps, a free pool of 256 spare pages (about
155 GB of K/V).  The lifecycle (synth/stream.py) drives the engine; this
test checks it against the fp64 oracle:

* every step, exactly: the page tables the engine produced for each Grow
  (lowest free page appended), Compress & Hold (copy-on-write plan: every
  shared page replaced by the lowest free page, in logical order; private
  pages kept; replaced pages released), finish, preemption and admission are
  replayed on the oracle's page pool from the tables at the start of the
  step, and the engine's reference counts and free count must equal the
  replay's;
* on sampled steps (replayed from the GPU's pre-step state, so an allowed
  tie difference cannot cascade): the summaries after the update (1e-12),
  D_p (tie rule), the demand probabilities (1e-4 absolute) and importance of
  sampled units of the boundary requests; the whole decision of one request
  from every unit; the Eq. 10 keep masks and the compacted K/V bytes of the
  sampled units of requests that compressed;
* the stream exercises Grow, Compress & Hold with copy-on-write, fallback,
  preemption on GP_ERR_NO_PAGES, finishes and admissions.
"""

import gc

import numpy as np
import pytest
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth
from synth.stream import ContinuousBatch

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256
STEPS = 1000
SAMPLED = set(range(8, 16)) | set(range(50, STEPS, 50))
FULL_DECISION = {8, 100, 500, 900}


class Checker:
    def __init__(self, w, units):
        self.w = w
        self.units = units
        self.pre = {}          # seat -> (summaries before the update, q, first)
        self.snap = {}         # (seat, unit) -> (keys, values) before compaction
        self.oracle = {}       # (seat, unit) -> oracle unit result
        self.checked = 0
        self.decisions = 0
        self.compared_masks = 0
        self.rng = np.random.default_rng(5)

    def _sample_seats(self, drv, t):
        b = [s for s in drv.live() if drv.at_boundary(s, t)]
        b = [s for s in b if drv.seats[s].req.num_pages < drv.maxp]
        return b[:2]

    def pre_update(self, drv, t, live, q_live):
        self.pre.clear()
        self.snap.clear()
        self.oracle.clear()
        if t not in SAMPLED:
            return
        sh = self.w.shape
        for s in self._sample_seats(drv, t):
            st = drv.seats[s]
            summ = gp.gp_read_summaries(drv.ctx, st.req.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            q = q_live[:, live.index(s)].double().cpu().numpy()
            self.pre[s] = (summ, q, st.first_pending)

    def post_demand(self, drv, t, bseats, q_b, dem, acts):
        if not self.pre:
            return
        sh = self.w.shape
        G = sh.group
        for s, (summ, q, first) in self.pre.items():
            if s not in bseats:
                continue
            r = bseats.index(s)
            req = drv.seats[s].req
            P = req.num_pages
            # A1: the engine's update against the oracle's, from the same pre-step state
            s_new, l_new = og.ema_update(summ[:, 0], summ[:, 1], q, first, 0.9, 0.999)
            got = gp.gp_read_summaries(drv.ctx, req.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            for x, ref in ((0, s_new), (1, l_new)):
                scale = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)) + 1e-30
                err = float(np.max(np.abs(got[:, x] - ref) / scale))
                assert err <= hz.SUMMARY_REL, f"step {t} seat {s}: summary error {err}"
            qt = og.summary_queries(s_new, l_new, q, req.pos, sh.rope_theta)
            ks = gp.gp_debug_demand_k(drv.ctx, r, self.units)
            assert dem[r].sum_k_short == int(ks[:, 0].sum()) and dem[r].sum_k_long == int(ks[:, 1].sum())
            probs = gp.gp_debug_probs(drv.ctx, r, self.units, (P - 1) * PAGE)
            scores = gp.gp_debug_scores(drv.ctx, r, self.units, P * PAGE - 16)
            sample = sorted({0, self.units - 1, *self.rng.choice(np.arange(1, self.units - 1), 2,
                                                                 replace=False).tolist()})
            full = t in FULL_DECISION and s == next(iter(self.pre))
            todo = range(self.units) if full else sample
            kk, ties = np.zeros((self.units, 2), np.int64), 0
            for idx in todo:
                layer, h = divmod(idx, sh.num_kv_heads)
                u = hz.oracle_unit_dev(qt, self.w.k_cache, req.pages, layer, h, G)
                for x in range(2):
                    ok, msg = hz.dp_ok(int(ks[idx, x]), u.a_dem[x], 0.99)
                    assert ok, f"step {t} seat {s} (P={P}) unit {idx} x {x}: {msg}"
                    ties += int(ks[idx, x] != u.k[x])
                kk[idx] = u.k
                if idx in sample:
                    err = np.abs(probs[idx].astype(np.float64) - u.a_dem).max()
                    assert err <= hz.PROB_ABS, f"step {t} seat {s} unit {idx}: probability error {err}"
                    sg = np.exp2(scores[idx].astype(np.float64))
                    big = u.s > 1e-30
                    rel = np.abs(sg[big] - u.s[big]) / u.s[big]
                    assert rel.max() < 2e-5, f"step {t} seat {s} unit {idx}: importance error {rel.max()}"
                    self.oracle[(s, idx)] = u
                    if acts[r].kind != gp.GP_ACT_GROW:
                        self.snap[(s, idx)] = (hz.unit_keys_dev(self.w.k_cache, req.pages, layer, h),
                                               hz.unit_keys_dev(self.w.v_cache, req.pages, layer, h))
                self.checked += 1
            if full:
                free_before = gp.gp_free_page_count(drv.ctx)
                grants = sum(1 for a in acts[:r] if a.kind == gp.GP_ACT_GROW and not a.forced)
                ok, msg = hz.decision_ok(acts[r], kk, ks, P, free_before - grants)
                assert ok, f"step {t} seat {s}: {msg}"
                self.decisions += 1

    def post_compress(self, drv, t, cseats):
        for i, s in enumerate(cseats):
            units = [(k[1], v) for k, v in self.oracle.items() if k[0] == s]
            if not units:
                continue
            req = drv.seats[s].req
            P = req.num_pages
            masks = gp.unpack_mask(gp.gp_debug_keep_mask(drv.ctx, i, self.units, P), P * PAGE)
            sh = self.w.shape
            for idx, u in units:
                keep = masks[idx]
                ok, _, msg = hz.topk_ok(keep, u.s, P)
                assert ok, f"step {t} seat {s} (P={P}) unit {idx}: {msg}"
                layer, h = divmod(idx, sh.num_kv_heads)
                kp, vp = self.snap[(s, idx)]
                kept = np.nonzero(keep)[0]
                n_live = (P - 1) * PAGE
                assert np.array_equal(hz.unit_keys_dev(self.w.k_cache, req.pages, layer, h)[:n_live], kp[kept])
                assert np.array_equal(hz.unit_keys_dev(self.w.v_cache, req.pages, layer, h)[:n_live], vp[kept])
                self.compared_masks += 1

    def post_step(self, drv, t, log):
        """Replay the step's page operations on the oracle's pool."""
        pool = og.PagePool(self.w.num_pages)
        for table in log.live_before.values():
            for pg in table:
                pool.refcount[pg] += 1
        for kind, s, before, after in log.actions:
            if kind == "grow":
                exp = og.grow(before, pool)
                assert after == exp, f"step {t} seat {s}: grow {after[-1]} vs oracle {exp[-1]}"
            elif kind == "compress":
                exp, replaced = og.cow_plan(before, pool)
                assert after == exp, f"step {t} seat {s}: copy-on-write table differs from the oracle's plan"
                og.release_replaced(replaced, pool)
            else:  # finish / preempt: every reference dropped
                for pg in before:
                    pool.unref(pg)
        for s, table in log.admitted:
            for pg in table:
                if pool.refcount[pg] > 0:
                    pool.ref(pg)               # shared prefix page
                else:
                    assert pool.alloc() == pg, f"step {t} seat {s}: admission took page {pg} out of order"
        live_now = {s: list(drv.seats[s].req.pages) for s in drv.live()}
        expect = [0] * self.w.num_pages
        for table in live_now.values():
            for pg in table:
                expect[pg] += 1
        assert expect == pool.refcount, f"step {t}: live tables and the replayed pool disagree"
        assert gp.gp_free_page_count(drv.ctx) == pool.free_count(), f"step {t}: free count"
        if t % 25 == 0 or t == STEPS - 1:
            eng = [gp.gp_page_refcount(drv.ctx, pg) for pg in range(self.w.num_pages)]
            assert eng == pool.refcount, f"step {t}: engine refcounts differ from the replay"


@pytest.fixture(scope="module")
def stream():
    w = synth.make_workload("stream256", device="cuda")
    cfg = hz.engine_config(w, max_slots=256, max_pages_per_req=128)
    ctx = gp.gp_create(cfg, w.k_cache, w.v_cache, None)
    drv = ContinuousBatch(gp, ctx, w, 128)
    yield w, cfg, drv
    gp.gp_destroy(ctx)
    del drv, w
    gc.collect()
    torch.cuda.empty_cache()


def test_stream256_thousand_steps(stream):
    w, cfg, drv = stream
    chk = Checker(w, cfg.num_layers * cfg.num_kv_heads)
    for t in range(STEPS):
        drv.step(t, hooks=chk)
    torch.cuda.synchronize()
    c = drv.counts
    print("stream256 counts:", c, "mean live:", drv.live_sum / STEPS, "units checked:", chk.checked,
          "decisions:", chk.decisions, "masks:", chk.compared_masks)
    assert c["grow"] > 0 and c["compress"] > 0 and c["cow_pages"] > 0
    assert c["finish"] > 0 and c["admit"] > 0
    assert c["fallback"] + c["preempt"] > 0            # the bounded pool ran out
    assert chk.checked >= 100 and chk.compared_masks >= 20 and chk.decisions >= 1
    st = gp.gp_stats(drv.ctx)
    assert st["cow_pages"] == c["cow_pages"]
