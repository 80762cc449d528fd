"""CPU checks of the comparison helpers the GPU parity tests rely on."""

import numpy as np

import oracle.growpage as og

import harness as hz


def test_topk_ok_accepts_oracle_and_tie_swaps_only():
    rng = np.random.default_rng(0)
    P, b, R = 4, 256, 16
    s = rng.dirichlet(np.full(P * b - R, 0.3))
    keep = og.select_retained(s, P, b, R, 64)
    ok, nd, msg = hz.topk_ok(keep, s, P)
    assert ok and nd == 0, msg
    # swap the global k-th kept slot with the best dropped one: allowed only
    # if their scores are within 1e-5 relative
    dropped = np.nonzero(~keep[:P * b - R])[0]
    best_drop = dropped[np.argmax(s[dropped])]
    kept_glob = np.nonzero(keep[:P * b - R])[0]
    worst_kept = kept_glob[np.argmin(s[kept_glob])]
    bad = keep.copy()
    bad[worst_kept], bad[best_drop] = False, True
    ok, nd, msg = hz.topk_ok(bad, s, P)
    assert not ok
    s2 = s.copy()
    s2[best_drop] = s2[worst_kept] * (1 - 2e-6)     # near-tie at the threshold
    keep2 = og.select_retained(s2, P, b, R, 64)
    bad2 = keep2.copy()
    bad2[worst_kept], bad2[best_drop] = False, True
    ok, nd, msg = hz.topk_ok(bad2, s2, P)
    assert ok and nd == 2, msg
    # wrong counts and a dropped recent window are rejected
    wrong = keep.copy()
    wrong[P * b - 1] = False
    assert not hz.topk_ok(wrong, s, P)[0]


def test_dp_ok_tie_band():
    a = np.full(1024, 1.0 / 1024)
    assert hz.dp_ok(1014, a, 0.99)[0]
    assert not hz.dp_ok(1015, a, 0.99)[0]
    # p exactly at a cumulative point: D and D+1 ... only the tie side
    ok, why = hz.dp_ok(769, a, 0.75)
    assert ok and why == "tie-above"
    assert not hz.dp_ok(770, a, 0.75)[0]
