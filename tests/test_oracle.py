"""Pins of the fp64 oracle to what the GrowPage paper and mathematics fix.

Every check here is independent of the oracle's own code path: hand-derived
golden values (tests/golden/*.json), closed forms, invariants, brute force on
tiny inputs, and special cases that reduce to a library routine.  The last
group plants plausible mistakes in the oracle (on the CPU) and checks that a
pin catches each one.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from oracle import growpage as og

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Eq. 2: p-coverage demand
# ---------------------------------------------------------------------------

def check_dp_golden(dp=og.coverage_demand):
    for case in _golden("coverage_demand.json")["cases"]:
        if "a_uniform" in case:
            n = case["a_uniform"]
            a = np.full(n, 1.0 / n)
        else:
            a = np.array(case["a"], dtype=np.float64)
        got = dp(a, case["p"])
        assert got == case["expect"], (case, got)


def test_dp_golden():
    check_dp_golden()


@pytest.mark.parametrize("n", [3, 7, 100, 1000, 4093])
def test_dp_uniform_closed_form(n):
    # uniform weights: sum of k weights is k/n, so D_p = ceil(p n) when p n is
    # not an integer (Eq. 2)
    rng = np.random.default_rng(n)
    for p in rng.uniform(0.01, 0.999, size=20):
        if abs(p * n - round(p * n)) < 1e-6:
            continue
        assert og.coverage_demand(np.full(n, 1.0 / n), p) == math.ceil(p * n)


def test_dp_one_hot_and_monotone():
    rng = np.random.default_rng(1)
    for n in (1, 2, 17, 300):
        e = np.zeros(n)
        e[rng.integers(n)] = 1.0
        assert og.coverage_demand(e, 0.99) == 1
    for _ in range(50):
        n = int(rng.integers(1, 400))
        a = rng.gamma(0.3, size=n)
        a /= a.sum()
        ps = np.sort(rng.uniform(0, 1, size=30))
        ds = [og.coverage_demand(a, p) for p in ps]
        assert all(x <= y for x, y in zip(ds, ds[1:]))     # monotone in p
        assert all(1 <= x <= n for x in ds)


def test_dp_bruteforce_small():
    # D_p is the size of the smallest subset whose mass reaches p (the largest
    # mass of a k-subset is that of the top-k weights): enumerate subsets.
    rng = np.random.default_rng(2)
    for _ in range(200):
        n = int(rng.integers(1, 9))
        a = rng.dirichlet(np.full(n, 0.5))
        p = float(rng.uniform(0.05, 0.999))
        best = None
        for k in range(1, n + 1):
            if max(sum(a[list(s)]) for s in itertools.combinations(range(n), k)) >= p:
                best = k
                break
        assert og.coverage_demand(a, p) == best


# ---------------------------------------------------------------------------
# Eqs. 3-5, Theorem 3.1 (brute force over all subsets, N <= 12)
# ---------------------------------------------------------------------------

def check_theorem31(dp=og.coverage_demand, seed=3, trials=40):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        n = int(rng.integers(1, 13))
        if t % 3 == 0:
            a = rng.dirichlet(np.full(n, 0.2))          # concentrated
        elif t % 3 == 1:
            a = rng.dirichlet(np.full(n, 5.0))          # diffuse
        else:
            a = np.sort(rng.dirichlet(np.ones(n)))[::-1]
        vmax = float(rng.uniform(0.5, 3.0))
        delta = float(rng.uniform(0.01, 2 * vmax - 0.01))
        cap = og.worst_case_capacity(a, delta, vmax)
        assert cap == dp(a, 1.0 - delta / (2.0 * vmax)), (a, delta, vmax)


def test_theorem31_bruteforce():
    check_theorem31()


def test_theorem31_golden():
    for case in _golden("theorem31.json")["cases"]:
        a = np.array(case["a"])
        if "expect_capacity" in case:
            got = og.worst_case_capacity(a, case["delta"], case["vmax"])
            assert got == case["expect_capacity"]
            assert og.coverage_demand(a, 1 - case["delta"] / (2 * case["vmax"])) == got
        else:
            got = og.worst_case_error(a, case["subset"], case["vmax"])
            assert got == pytest.approx(case["expect_error"], abs=1e-15)


def test_eq5_tight_construction_and_bound():
    # App. C: with v_i = -Vmax u on S and +Vmax u off S the error equals
    # 2 Vmax (1 - m(S)); no admissible v exceeds it.
    rng = np.random.default_rng(4)
    for _ in range(60):
        n = int(rng.integers(2, 10))
        d = int(rng.integers(1, 6))
        a = rng.dirichlet(np.ones(n))
        vmax = float(rng.uniform(0.1, 4))
        k = int(rng.integers(1, n))
        sub = sorted(rng.choice(n, size=k, replace=False).tolist())
        u = rng.normal(size=d)
        u /= np.linalg.norm(u)
        v = np.array([(-vmax if i in sub else vmax) * u for i in range(n)])
        err = np.linalg.norm(og.attention_output(a, v) -
                             og.renormalised_output(a, v, sub))
        bound = og.worst_case_error(a, sub, vmax)
        assert err == pytest.approx(bound, rel=1e-12, abs=1e-14)
        for _ in range(20):
            w = rng.normal(size=(n, d))
            w *= (vmax * rng.uniform(0, 1, size=(n, 1))) / np.linalg.norm(w, axis=1, keepdims=True)
            e2 = np.linalg.norm(og.attention_output(a, w) - og.renormalised_output(a, w, sub))
            assert e2 <= bound * (1 + 1e-12) + 1e-14


# ---------------------------------------------------------------------------
# Eq. 6 and App. E.1: EMA
# ---------------------------------------------------------------------------

def check_ema_golden(update=og.ema_update):
    g = _golden("ema.json")
    d = 3
    s = l = None
    seq = [np.zeros(d), np.ones(d)] + [np.zeros(d)] * 4
    hist_s, hist_l = {}, {}
    for t, q in enumerate(seq):
        s, l = update(s, l, q, t == 0, g["beta_s"], g["beta_l"])
        hist_s[t], hist_l[t] = s[0], l[0]
    for t, v in g["short_after_steps"].items():
        assert hist_s[int(t)] == pytest.approx(v, rel=1e-12)
    for t, v in g["long_after_steps"].items():
        assert hist_l[int(t)] == pytest.approx(v, rel=1e-12)


def test_ema_impulse_golden():
    check_ema_golden()


def test_ema_constant_fixed_point_and_beta0():
    rng = np.random.default_rng(5)
    q = rng.normal(size=(2, 4, 8))
    s, l = og.ema_update(None, None, q, True, 0.9, 0.999)   # init (App. E.1)
    assert np.array_equal(s, q) and np.array_equal(l, q)
    for _ in range(100):
        s, l = og.ema_update(s, l, q, False, 0.9, 0.999)
    assert np.allclose(s, q, rtol=1e-13) and np.allclose(l, q, rtol=1e-13)
    # beta_S = 0 reduces the short summary to the current query (Sec. 5.3)
    q2 = rng.normal(size=q.shape)
    s2, _ = og.ema_update(s, l, q2, False, 0.0, 0.999)
    assert np.array_equal(s2, q2)
    # the init overwrites stale state without clearing
    s3, l3 = og.ema_update(s2 * 7, l * 3, q, True, 0.9, 0.999)
    assert np.array_equal(s3, q) and np.array_equal(l3, q)


def test_ema_matches_geometric_sum():
    # closed form of the recursion: qbar_T = beta^T q_0 + sum_t (1-beta) beta^(T-t) q_t
    rng = np.random.default_rng(6)
    qs = rng.normal(size=(30, 5))
    for beta in (0.9, 0.999, 0.5):
        s = None
        for t, q in enumerate(qs):
            s, _ = og.ema_update(s, s, q, t == 0, beta, beta)
        T = len(qs) - 1
        ref = beta ** T * qs[0] + sum((1 - beta) * beta ** (T - t) * qs[t] for t in range(1, T + 1))
        assert np.allclose(s, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Eq. 12 calibration and RoPE
# ---------------------------------------------------------------------------

def test_calibration_restores_rms():
    rng = np.random.default_rng(7)
    q = rng.normal(size=(3, 4, 16)) * rng.uniform(0.1, 5, size=(3, 4, 1))
    qbar = rng.normal(size=(3, 4, 16)) * 0.01
    qt = og.calibrate(qbar, q)
    assert np.allclose(og.rms(qt), og.rms(q), rtol=1e-13)
    # direction unchanged, positive scale
    cos = np.sum(qt * qbar, -1) / (np.linalg.norm(qt, axis=-1) * np.linalg.norm(qbar, axis=-1))
    assert np.allclose(cos, 1.0, rtol=1e-13)
    assert np.array_equal(og.calibrate(np.zeros((2, 8)), rng.normal(size=(2, 8))), np.zeros((2, 8)))


def test_rope_rotation_properties():
    rng = np.random.default_rng(8)
    for d in (2, 8, 64, 128):
        x = rng.normal(size=(5, d))
        y = rng.normal(size=(5, d))
        theta = 1e4
        assert np.array_equal(og.rope(x, 0, theta), x)                 # identity at 0
        for pos in (1, 17, 1000, 32768):
            rx = og.rope(x, pos, theta)
            assert np.allclose(np.linalg.norm(rx, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
            assert np.allclose(og.rope(rx, -pos, theta), x, atol=1e-9)     # inverse
            # relative position: R_m x . R_n y = x . R_{n-m} y
            m, n = pos, pos + 37
            lhs = np.sum(og.rope(x, m, theta) * og.rope(y, n, theta), -1)
            rhs = np.sum(x * og.rope(y, n - m, theta), -1)
            assert np.allclose(lhs, rhs, rtol=1e-9, atol=1e-9)
    # d = 2: a plain rotation by pos radians (theta^0 = 1)
    x = np.array([1.0, 0.0])
    assert np.allclose(og.rope(x, 1, 1e4), [math.cos(1.0), math.sin(1.0)], atol=1e-15)


# ---------------------------------------------------------------------------
# scores, softmax, GQA mean
# ---------------------------------------------------------------------------

def test_logits_against_loops_and_softmax_against_scipy():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(3, 8))
    k = rng.normal(size=(11, 8))
    z = og.logits(q, k)
    for r in range(3):
        for i in range(11):
            ref = sum(q[r, j] * k[i, j] for j in range(8)) / math.sqrt(8)
            assert z[r, i] == pytest.approx(ref, rel=1e-13, abs=1e-14)
    big = rng.normal(size=(4, 500)) * 30
    assert np.allclose(og.softmax(big), scipy.special.softmax(big, axis=-1), rtol=1e-12, atol=1e-300)
    a = og.kv_head_distribution(big)
    assert a.sum() == pytest.approx(1.0, abs=1e-13)
    # G = 1 reduces to the single query head's softmax
    assert np.allclose(og.kv_head_distribution(big[:1]), scipy.special.softmax(big[0]), rtol=1e-12)


def test_unit_candidate_sets():
    rng = np.random.default_rng(10)
    b, P, R, G, d = 8, 3, 2, 2, 4
    keys = rng.normal(size=(P * b, d))
    qt = rng.normal(size=(2, G, d))
    u = og.unit_boundary(qt, keys, P, b, R, 0.9)
    assert u.a_dem.shape == (2, (P - 1) * b)
    assert u.a_cmp.shape == (2, P * b - R)
    # demand distribution: mean over the G heads of a softmax over Cdem only
    for x in range(2):
        z = np.array([[qt[x, g] @ keys[i] / 2.0 for i in range((P - 1) * b)] for g in range(G)])
        ref = np.mean([scipy.special.softmax(z[g]) for g in range(G)], axis=0)
        assert np.allclose(u.a_dem[x], ref, rtol=1e-12)
    assert np.allclose(u.s, np.maximum(u.a_cmp[0], u.a_cmp[1]))


# ---------------------------------------------------------------------------
# Eq. 8 and the decision rule
# ---------------------------------------------------------------------------

def test_decide_rules():
    assert og.decide(0.01, 4, 10, 0, 0.0).kind == og.GROW
    assert og.decide(0.0, 4, 10, 0, 0.0).kind == og.COMPRESS       # Delta = tau compresses
    assert og.decide(-0.01, 4, 10, 0, 0.0).kind == og.COMPRESS
    a = og.decide(0.01, 4, 0, 0, 0.0)
    assert a.kind == og.COMPRESS and a.fallback                   # fallback (Sec. 4.2)
    a = og.decide(0.01, 4, 3, 3, 0.0)
    assert a.kind == og.COMPRESS and a.fallback                   # reserve respected
    a = og.decide(-1.0, 1, 0, 0, 0.0)
    assert a.kind == og.GROW and a.forced                         # P = 1
    assert og.decide(0.5, 4, 10, 0, 0.0, policy="fixed").kind == og.COMPRESS
    assert og.decide(0.002, 4, 10, 0, 0.003).kind == og.COMPRESS  # tau threshold


def test_demand_trend_forms_agree_in_sign():
    rng = np.random.default_rng(11)
    for _ in range(100):
        ks = rng.integers(1, 500, size=(4, 2))
        kl = rng.integers(1, 500, size=(4, 2))
        n = 768
        d = og.demand_trend(ks, kl, n)
        raw = int(ks.sum() - kl.sum())
        assert np.sign(d) == np.sign(raw)                        # Eq. 8 vs raw D_p difference
        assert d == pytest.approx(raw / (n * ks.size), rel=1e-12, abs=1e-15)


def check_trend_sign_exact(trend=og.demand_trend):
    # Eq. 8 with equal demand sums: Delta is exactly 0 whatever the split over
    # units, so the decision after Eq. 8 compresses (Delta = tau = 0 is not
    # above tau).  Cases written by hand: 3/7 + 5/7 and 4/7 + 4/7 are not
    # equal once each ratio is rounded separately.
    for ks, kl, n in (([3, 5], [4, 4], 7), ([1, 2, 3], [3, 2, 1], 11), ([10, 1, 1, 7], [5, 5, 5, 4], 23)):
        d = trend(np.array(ks), np.array(kl), n)
        assert d == 0.0, (ks, kl, n, d)
        assert og.decide(d, 4, 10, 0, 0.0).kind == og.COMPRESS
    rng = np.random.default_rng(12)
    for _ in range(2000):
        n = int(rng.integers(1, 40000))
        ks = rng.integers(1, n + 1, size=int(rng.integers(2, 300)))
        assert trend(ks, np.roll(ks, 1), n) == 0.0


def test_trend_sign_exact_at_equal_sums():
    check_trend_sign_exact()


def _trend_mean_of_rounded_ratios(k_short, k_long, n_cand):
    return float(np.mean(np.asarray(k_short, float) / n_cand) - np.mean(np.asarray(k_long, float) / n_cand))


def test_pins_catch_trend_rounding_mutant():
    with pytest.raises(AssertionError):
        check_trend_sign_exact(_trend_mean_of_rounded_ratios)


def test_planted_tiny_workloads_take_both_actions():
    # Sec. 3.2: a more concentrated short summary (Delta < 0) compresses; a
    # more diffuse one (Delta > 0) grows.  The synthetic tiny workloads put a
    # concentrated history early or late.
    import synth
    for variant, expect in (("grow", og.GROW), ("compress", og.COMPRESS)):
        w = synth.make_workload("tiny", variant=variant)
        cfg = _cfg(w)
        s = l = None
        for t, q in enumerate(w.history):
            s, l = og.ema_update(s, l, q[:, 0].double().numpy(), t == 0, 0.9, 0.999)
        q_cur = w.history[-1][:, 0].double().numpy()
        res = og.request_boundary(s, l, q_cur, w.k_cache.double().numpy(),
                                  w.block_tables[0], w.positions[0], cfg)
        act = og.decide(res["delta"], len(w.block_tables[0]), 4, 0, 0.0)
        assert act.kind == expect, (variant, res["delta"])


def _cfg(w):
    return {"num_kv_heads": w.shape.num_kv_heads, "rope_theta": w.shape.rope_theta,
            "page_size": w.page_size, "recent_window": 16, "p": 0.99}


# ---------------------------------------------------------------------------
# Eq. 10 and the window mask
# ---------------------------------------------------------------------------

def _check_selection(s, P, b, R, k_loc, keep):
    n_cmp = P * b - R
    k_t = (P - 1) * b - R
    assert keep.sum() == (P - 1) * b                        # exactly one page freed
    assert keep[n_cmp:].all()                               # recent window kept
    quota = min(k_loc, k_t // P)
    for j in range(P):
        lo, hi = j * b, min((j + 1) * b, n_cmp)
        kj = min(quota, hi - lo)
        blk = np.arange(lo, hi)
        # the block's own top-kj (by score, ties to lower index) are kept
        order = sorted(blk.tolist(), key=lambda i: (-s[i], i))
        assert keep[order[:kj]].all()


def test_selection_invariants_and_global_top():
    rng = np.random.default_rng(12)
    for t in range(300):
        b = int(rng.integers(2, 9))
        P = int(rng.integers(2, 6))
        R = int(rng.integers(0, b))
        k_loc = int(rng.integers(0, b + 2))
        s = rng.dirichlet(np.full(P * b, 0.3))
        if t % 5 == 0:
            s = np.round(s * 20) / 20                            # many ties
        keep = og.select_retained(s, P, b, R, k_loc)
        _check_selection(s, P, b, R, k_loc, keep)
        # the global fill is a top set of what the blocks left: no dropped
        # candidate beats a globally added one (ties: lower index first)
        n_cmp = P * b - R
        k_t = (P - 1) * b - R
        quota = min(k_loc, k_t // P)
        loc = np.zeros(P * b, bool)
        for j in range(P):
            lo, hi = j * b, min((j + 1) * b, n_cmp)
            order = sorted(range(lo, hi), key=lambda i: (-s[i], i))
            loc[order[:min(quota, hi - lo)]] = True
        glob = keep.copy()
        glob[loc] = False
        glob[n_cmp:] = False
        dropped = np.nonzero(~keep[:n_cmp])[0]
        for i in np.nonzero(glob)[0]:
            for j in dropped:
                assert (s[i], -i) > (s[j], -j)


def test_selection_kloc0_is_plain_topk():
    # k_loc = 0 leaves only the global top-K_t (special case of Eq. 10)
    rng = np.random.default_rng(13)
    for _ in range(50):
        b, P, R = 16, 4, 3
        s = rng.random(P * b)
        keep = og.select_retained(s, P, b, R, 0)
        k_t = (P - 1) * b - R
        top = np.argsort(-s[:P * b - R], kind="stable")[:k_t]
        ref = np.zeros(P * b, bool)
        ref[top] = True
        ref[P * b - R:] = True
        assert np.array_equal(keep, ref)


def test_selection_kloc_changes_which_not_how_many():
    # App. D.2: k_loc changes which states are kept, not how many
    rng = np.random.default_rng(14)
    s = rng.dirichlet(np.full(5 * 256, 0.2))
    counts = {int(og.select_retained(s, 5, 256, 16, k).sum()) for k in (0, 16, 32, 64, 128)}
    assert counts == {4 * 256}


# ---------------------------------------------------------------------------
# App. E.2: pool, copy-on-write, compaction
# ---------------------------------------------------------------------------

def test_pool_cow_and_compaction():
    rng = np.random.default_rng(15)
    pool = og.PagePool(12)
    a = [pool.alloc() for _ in range(4)]                 # 0..3 lowest first
    assert a == [0, 1, 2, 3]
    pool.ref(0)
    pool.ref(1)                                          # prefix pages 0,1 shared
    total_before = sum(pool.refcount)
    new, replaced = og.cow_plan(a, pool)
    assert replaced == [0, 1] and new == [4, 5, 2, 3]    # lowest free, ascending order
    og.release_replaced(replaced, pool)
    assert pool.refcount[0] == 1 and pool.refcount[1] == 1
    assert sum(pool.refcount) == total_before + 2 - 2
    # not enough pages: nothing changes
    pool2 = og.PagePool(3)
    t = [pool2.alloc(), pool2.alloc(), pool2.alloc()]
    pool2.ref(0)
    pool2.ref(1)
    before = list(pool2.refcount)
    with pytest.raises(MemoryError):
        og.cow_plan(t, pool2)
    assert pool2.refcount == before
    # compaction of one request, two layers, one head
    L, b, d = 2, 4, 3
    P = 3
    k = rng.normal(size=(L, 12, 1, b, d))
    v = rng.normal(size=(L, 12, 1, b, d))
    old = [7, 2, 9]
    newt = [7, 11, 9]
    keep = np.zeros((L, 1, P * b), bool)
    for layer in range(L):
        keep[layer, 0, rng.choice(P * b - 1, size=(P - 1) * b - 1, replace=False)] = True
        keep[layer, 0, P * b - 1] = True
    k2, v2 = og.compress_cache(k, v, old, newt, keep, b)
    for layer in range(L):
        rows = og.gather_logical(k, old, layer, 0)[keep[layer, 0]]
        got = og.gather_logical(k2, newt, layer, 0)[:(P - 1) * b]
        assert np.array_equal(got, rows)                 # order kept, bytes equal
    assert np.array_equal(k2[:, 2], k[:, 2])             # replaced page untouched


# ---------------------------------------------------------------------------
# Sec. 5.3, Table 2: the entropy metric's effective support size exp(H)
# ---------------------------------------------------------------------------

def check_entropy_support(es=og.entropy_support):
    rng = np.random.default_rng(11)
    # a point mass spreads over one token, a uniform distribution over all of them
    assert es(np.eye(1, 37, 5)[0]) == 1.0
    for n in (1, 2, 7, 256, 8176):
        assert abs(es(np.full(n, 1.0 / n)) - n) <= 1e-9 * n
    # uniform over m of n slots, zeros elsewhere: m (zeros carry no entropy)
    a = np.zeros(1000)
    a[rng.choice(1000, 40, replace=False)] = 1.0 / 40
    assert abs(es(a) - 40) <= 1e-9
    # scipy's Shannon entropy (natural log) on random distributions
    for n in (3, 50, 4096):
        a = rng.dirichlet(np.full(n, 0.3))
        assert abs(math.log(es(a)) - scipy.stats.entropy(a)) <= 1e-10 * max(1.0, scipy.stats.entropy(a))
    # additivity over a product distribution, and the bounds 1/max(a) <= exp(H) <= N
    x, y = rng.dirichlet(np.ones(9)), rng.dirichlet(np.full(13, 0.5))
    assert abs(es(np.outer(x, y).ravel()) - es(x) * es(y)) <= 1e-9 * es(x) * es(y)
    for _ in range(20):
        a = rng.dirichlet(np.full(64, rng.uniform(0.05, 3.0)))
        assert 1.0 / a.max() - 1e-9 <= es(a) <= 64 + 1e-9
    # permutation invariance
    a = rng.dirichlet(np.ones(100))
    assert abs(es(a) - es(rng.permutation(a))) <= 1e-12 * es(a)


def test_entropy_support():
    check_entropy_support()


def test_entropy_trend_and_decision():
    """With exp(H) in place of K^x, Eq. 8 and the decision keep their form:
    a short summary spread wider than the long one grows, a narrower one compresses."""
    n_cand = 7 * 256
    wide = og.entropy_support(np.full(n_cand, 1.0 / n_cand))
    narrow = og.entropy_support(np.full(64, 1.0 / 64))
    assert wide == pytest.approx(n_cand) and narrow == pytest.approx(64)
    d = og.demand_trend([wide, narrow], [narrow, narrow], n_cand)
    assert d == pytest.approx((n_cand - 64) / (2 * n_cand))
    assert og.decide(d, 8, 10, 0, 0.0).kind == og.GROW
    assert og.decide(-d, 8, 10, 0, 0.0).kind == og.COMPRESS


# ---------------------------------------------------------------------------
# summary queries (Eq. 12 then RoPE), importance (Eq. 9), retention, gather
# ---------------------------------------------------------------------------

def check_summary_queries(sq=og.summary_queries):
    rng = np.random.default_rng(21)
    L, hq, d = 2, 4, 64
    qs, ql, q = (rng.normal(size=(L, hq, d)) * sc for sc in (0.3, 2.0, 1.0))
    out = sq(qs, ql, q, 37, 1e4)
    assert out.shape == (L, 2, hq, d)
    # Eq. 12 restores the current query's RMS, and RoPE keeps the norm
    for x in range(2):
        assert np.allclose(np.sqrt(np.mean(out[:, x] ** 2, axis=-1)), np.sqrt(np.mean(q ** 2, axis=-1)),
                           rtol=1e-12)
    # x = 0 is the short summary: swapping the summaries swaps the rows
    sw = sq(ql, qs, q, 37, 1e4)
    assert np.allclose(sw[:, 0], out[:, 1]) and np.allclose(sw[:, 1], out[:, 0])
    # at position 0 the row is the summary itself, rescaled by a positive factor
    z = sq(qs, ql, q, 0, 1e4)
    for x, qb in ((0, qs), (1, ql)):
        ratio = z[:, x] / qb
        assert np.all(ratio > 0) and np.allclose(ratio, ratio[..., :1], rtol=1e-12)
    # logits depend on relative position only: rows at pos m against keys rotated to n
    k = rng.normal(size=(5, d))
    a = og.logits(sq(qs, ql, q, 90, 1e4)[0, 0], og.rope(k, 30, 1e4))
    b = og.logits(sq(qs, ql, q, 60, 1e4)[0, 0], k)
    assert np.allclose(a, b, rtol=1e-10, atol=1e-12)


def test_summary_queries():
    check_summary_queries()


def test_importance_is_the_larger_of_the_two_distributions():
    rng = np.random.default_rng(22)
    a_s, a_l = rng.dirichlet(np.ones(300)), rng.dirichlet(np.full(300, 0.2))
    s = og.importance(a_s, a_l)
    assert np.all(s >= a_s) and np.all(s >= a_l)
    assert np.all((s == a_s) | (s == a_l))
    assert np.array_equal(s, og.importance(a_l, a_s))
    assert np.array_equal(og.importance(a_s, a_s), a_s)


def test_retention_budget_frees_exactly_drop_pages():
    for P in (2, 5, 33, 160):
        for drop in (1, 2):
            if P - drop < 1:
                continue
            kt = og.retention_budget(P, 256, 16, drop)
            assert P * 256 - (kt + 16) == drop * 256     # the kept set fills (P - drop) pages exactly
    assert og.retention_budget(32, 256, 16) == 7920      # K_t = (P - 1) b - R at 32 pages


def test_compact_unit_keeps_order_and_rows():
    rng = np.random.default_rng(23)
    rows = np.arange(4 * 256 * 3, dtype=np.float64).reshape(4 * 256, 3)   # row i holds 3i, 3i+1, 3i+2
    keep = np.zeros(4 * 256, bool)
    keep[rng.choice(4 * 256, 3 * 256, replace=False)] = True
    out = og.compact_unit(rows, keep)
    assert out.shape == (3 * 256, 3)
    src = (out[:, 0] / 3).astype(int)                  # which slot each output row came from
    assert np.all(np.diff(src) > 0)                    # ascending slot order, no repeats
    assert np.all(keep[src]) and src.size == keep.sum()


# ---------------------------------------------------------------------------
# planted mistakes (in the oracle, on the CPU) are caught by the pins
# ---------------------------------------------------------------------------

def _dp_strict(a, p):
    srt = np.sort(np.asarray(a, float))[::-1]
    cum = np.cumsum(srt)
    hit = np.nonzero(cum > p)[0]
    return int(hit[0]) + 1 if hit.size else srt.size


def _dp_off_by_one(a, p):
    return og.coverage_demand(a, p) + (1 if len(a) > 3 else 0)


def _dp_ascending(a, p):
    srt = np.sort(np.asarray(a, float))
    cum = np.cumsum(srt)
    hit = np.nonzero(cum >= p)[0]
    return int(hit[0]) + 1 if hit.size else srt.size


def _ema_swapped(s, l, q, first, bs, bl):
    q = np.asarray(q, float)
    if first:
        return q.copy(), q.copy()
    return (1 - bs) * s + bs * q, (1 - bl) * l + bl * q


@pytest.mark.parametrize("mutant", [_dp_strict, _dp_off_by_one, _dp_ascending])
def test_pins_catch_dp_mutants(mutant):
    caught = 0
    for check in (lambda: check_dp_golden(mutant), lambda: check_theorem31(mutant)):
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught >= 1


def test_pins_catch_ema_mutant():
    with pytest.raises(AssertionError):
        check_ema_golden(_ema_swapped)


def _entropy_sign_flipped(a):
    nz = np.asarray(a, float)
    nz = nz[nz > 0]
    return float(np.exp(np.sum(nz * np.log(nz))))


def _entropy_log2(a):
    nz = np.asarray(a, float)
    nz = nz[nz > 0]
    return float(np.exp(-np.sum(nz * np.log2(nz))))


def _entropy_unweighted(a):
    nz = np.asarray(a, float)
    nz = nz[nz > 0]
    return float(np.exp(-np.mean(np.log(nz))))


@pytest.mark.parametrize("mutant", [_entropy_sign_flipped, _entropy_log2, _entropy_unweighted])
def test_pins_catch_entropy_mutants(mutant):
    with pytest.raises(AssertionError):
        check_entropy_support(mutant)


def _summary_queries_swapped(qs, ql, q, pos, theta):
    return og.summary_queries(ql, qs, q, pos, theta)


def _summary_queries_uncalibrated(qs, ql, q, pos, theta):
    return np.stack([og.rope(np.asarray(x, float), pos, theta) for x in (qs, ql)], axis=1)


@pytest.mark.parametrize("mutant", [_summary_queries_swapped, _summary_queries_uncalibrated])
def test_pins_catch_summary_query_mutants(mutant):
    with pytest.raises(AssertionError):
        check_summary_queries(mutant)


def test_oracle_exports():
    for name in ("ema_update", "calibrate", "rope", "logits", "softmax",
                 "coverage_demand", "select_retained", "cow_plan", "compress_cache",
                 "worst_case_capacity"):
        assert hasattr(oracle, name)


# ---------------------------------------------------------------------------
# policy variants (App. H.1) and their counter-based draws
# ---------------------------------------------------------------------------

def test_splitmix64_published_sequence():
    # the reference generator's first outputs for seed 1234567 (state
    # advanced by the golden-ratio increment before each output)
    x, out = 1234567, []
    for _ in range(5):
        out.append(og.splitmix64(x))
        x = (x + 0x9E3779B97F4A7C15) % (1 << 64)
    assert out == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_policy_draws_are_uniform_and_keyed():
    u = [og.policy_draw(7, k) for k in range(20000)]
    assert all(0.0 <= x < 1.0 for x in u)
    assert abs(np.mean(u) - 0.5) < 0.01 and abs(np.mean(np.array(u) < 0.7) - 0.7) < 0.01
    assert og.policy_draw(7, 3) != og.policy_draw(8, 3)


def test_eq13_shrink_zones():
    d = lambda delta, P=16, free=10: og.decide(delta, P, free, 0, 0.0, policy="shrink")
    assert d(0.001).kind == og.GROW
    assert d(0.0).kind == og.COMPRESS                     # -0.005 <= Delta <= 0
    assert d(-0.005).kind == og.COMPRESS
    assert d(-0.0051).kind == og.SHRINK
    assert d(-0.2, P=4).kind == og.COMPRESS                # 1024-token floor: 4 pages
    assert d(-0.2, P=5).kind == og.SHRINK
    assert d(0.3, free=0).kind == og.COMPRESS and d(0.3, free=0).fallback


def test_inverse_fixed_random_rules():
    assert og.decide(0.1, 8, 5, 0, 0.0, policy="inverse").kind == og.COMPRESS
    assert og.decide(0.0, 8, 5, 0, 0.0, policy="inverse").kind == og.GROW
    assert og.decide(-0.1, 8, 5, 0, 0.0, policy="inverse").kind == og.GROW
    assert og.decide(0.5, 8, 5, 0, 0.0, policy="fixed").kind == og.COMPRESS
    assert og.decide(0.5, 1, 5, 0, 0.0, policy="fixed").forced
    assert og.decide(-0.5, 8, 5, 0, 0.0, policy="random", draw=0.69).kind == og.COMPRESS
    assert og.decide(-0.5, 8, 5, 0, 0.0, policy="random", draw=0.7).kind == og.GROW


def test_shrink_selection_keeps_two_pages_less():
    rng = np.random.default_rng(3)
    for P in (3, 5, 9):
        s = rng.random(P * 256 - 16)
        keep = og.select_retained(s, P, 256, 16, 64, drop=2)
        assert keep.sum() == (P - 2) * 256
        assert keep[P * 256 - 16:].all()
        quota = min(64, ((P - 2) * 256 - 16) // P)
        for j in range(P):
            lo, hi = j * 256, min((j + 1) * 256, P * 256 - 16)
            top = np.argsort(-s[lo:hi], kind="stable")[:quota] + lo
            assert keep[top].all()
        # everything kept outranks everything dropped outside the block quotas
        loc = np.zeros(P * 256, bool)
        for j in range(P):
            lo, hi = j * 256, min((j + 1) * 256, P * 256 - 16)
            loc[np.argsort(-s[lo:hi], kind="stable")[:quota] + lo] = True
        cand = ~loc
        cand[P * 256 - 16:] = False
        kept, dropped = s[keep[:P * 256 - 16] & cand[:P * 256 - 16]], s[~keep[:P * 256 - 16]]
        assert kept.min() >= dropped.max()


def test_shrink_release_returns_the_last_page():
    pool = og.PagePool(10)
    table = [pool.alloc() for _ in range(4)]
    new = og.shrink_release(table, pool)
    assert new == table[:3] and pool.refcount[table[3]] == 0 and pool.free_count() == 7


def test_hole_fill_by_hand():
    # P = 2 pages of 4 slots: one hole in the first page, filled by the last
    # page's only kept row
    rows = np.arange(8.0)[:, None]
    keep = np.array([1, 0, 1, 1, 0, 1, 0, 0], bool)
    assert og.hole_fill_unit(rows, keep, 2, 4)[:, 0].tolist() == [0.0, 5.0, 2.0, 3.0]
    # no hole: nothing moves
    keep = np.array([1, 1, 1, 1, 0, 0, 0, 0], bool)
    assert og.hole_fill_unit(rows, keep, 2, 4)[:, 0].tolist() == [0.0, 1.0, 2.0, 3.0]


# ---------------------------------------------------------------------------
# input widening, rotary frequencies and the logical gather, each pinned to
# hand-written values (tests/golden/bf16.json, rope.json, gather.json)
# ---------------------------------------------------------------------------

def check_widen_bf16(widen=og.widen_bf16):
    cases = _golden("bf16.json")["cases"]
    bits = np.array([int(c["bits"], 16) for c in cases], dtype=np.uint16)
    got = np.asarray(widen(bits), dtype=np.float64)
    assert got.dtype == np.float64 and got.shape == bits.shape
    for c, g in zip(cases, got):
        want = c["value"]
        if want == "nan":
            assert math.isnan(g), c["note"]
        elif want in ("inf", "-inf"):
            assert g == float(want), c["note"]
        else:
            w = float.fromhex(want)
            assert g == w and math.copysign(1.0, g) == math.copysign(1.0, w), (c["note"], g, w)


def test_widen_bf16_golden():
    check_widen_bf16()


def check_rope_golden(rope=og.rope):
    gd = _golden("rope.json")
    d, theta = gd["d"], gd["theta"]
    half = d // 2
    for pos, rec in gd["positions"].items():
        c, s = np.array(rec["cos"]), np.array(rec["sin"])
        out = np.asarray(rope(np.ones(d), int(pos), theta))
        assert np.allclose(out[:half], c - s, rtol=0, atol=1e-15), (pos, out)
        assert np.allclose(out[half:], c + s, rtol=0, atol=1e-15), (pos, out)
        for j in range(half):
            e = np.zeros(d)
            e[j] = 1.0
            col = np.asarray(rope(e, int(pos), theta))
            want = np.zeros(d)
            want[j], want[j + half] = c[j], s[j]
            assert np.allclose(col, want, rtol=0, atol=1e-15), (pos, j, col)


def test_rope_golden_every_frequency():
    check_rope_golden()


def check_gather_golden(gather=og.gather_logical):
    gd = _golden("gather.json")
    L, npg, hkv, b = gd["layers"], gd["pages"], gd["kv_heads"], gd["page_size"]
    cache = np.zeros((L, npg, hkv, b, 1))
    for layer, p, h, s in itertools.product(range(L), range(npg), range(hkv), range(b)):
        cache[layer, p, h, s, 0] = 1000 * layer + 100 * p + 10 * h + s
    for c in gd["cases"]:
        got = np.asarray(gather(cache, c["block_table"], c["layer"], c["kv_head"]))
        assert got.shape == (len(c["rows"]), 1), got.shape
        assert got[:, 0].tolist() == c["rows"], (c, got[:, 0].tolist())


def test_gather_logical_golden():
    check_gather_golden()


def _widen_shift15(bits):
    u = np.asarray(bits).astype(np.uint32) << np.uint32(15)
    return u.view(np.float32).astype(np.float64)


def _widen_as_fp16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _widen_unsigned(bits):
    u = (np.asarray(bits).astype(np.uint32) & np.uint32(0x7FFF)) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("mutant", [_widen_shift15, _widen_as_fp16, _widen_unsigned])
def test_pins_catch_widen_mutants(mutant):
    with pytest.raises(AssertionError):
        check_widen_bf16(mutant)


def _rope_exponent_i_over_d(x, pos, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = float(pos) * np.power(float(theta), -np.arange(half) / d)
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[..., :half] * c - x[..., half:] * s, x[..., half:] * c + x[..., :half] * s], -1)


def _rope_interleaved(x, pos, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    ang = float(pos) * np.power(float(theta), -2.0 * np.arange(d // 2) / d)
    c, s = np.cos(ang), np.sin(ang)
    ev, od = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = ev * c - od * s
    out[..., 1::2] = od * c + ev * s
    return out


def _rope_clockwise(x, pos, theta):
    return og.rope(x, -pos, theta)


@pytest.mark.parametrize("mutant", [_rope_exponent_i_over_d, _rope_interleaved, _rope_clockwise])
def test_pins_catch_rope_mutants(mutant):
    with pytest.raises(AssertionError):
        check_rope_golden(mutant)


def _gather_sorted_pages(cache, table, layer, h):
    return og.gather_logical(cache, sorted(table), layer, h)


def _gather_head_layer_swapped(cache, table, layer, h):
    return np.concatenate([np.asarray(cache[h, pg, layer]) for pg in table], axis=0)


def _gather_first_page_only(cache, table, layer, h):
    return np.concatenate([np.asarray(cache[layer, table[0], h]) for _ in table], axis=0)


@pytest.mark.parametrize("mutant", [_gather_sorted_pages, _gather_head_layer_swapped, _gather_first_page_only])
def test_pins_catch_gather_mutants(mutant):
    with pytest.raises((AssertionError, IndexError)):
        check_gather_golden(mutant)
