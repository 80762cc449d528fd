"""The work split of the tensor-core decode-attention kernel (host logic of
gp_decode_attention, through gp_debug_attention_plan on a host-only context):
every (request, KV head) pair's attended pages laid end to end and cut into
one even range per SM.  Checked on seeded token mixes: every pair present,
its pieces consecutive and numbered, no more than 64 of them, their tiles
covering exactly the attended tokens; CTAs in order, at most one per SM, no
range above the even share; whole pairs inside a range, only its first and
last items shared with a neighbour."""

import numpy as np
import pytest

import paged_kv_cache_step_gb300 as gp

PAGE = 256


def _ctx(hkv, max_pages=256):
    cfg = gp.gp_config_default(num_layers=2, num_q_heads=4 * hkv, num_kv_heads=hkv, head_dim=128, num_pages=8,
                               max_slots=4, max_pages_per_req=max_pages, rope_theta=1e4)
    return gp.gp_create(cfg, None, None, None)


def _check_plan(items, ntok, hkv, sms):
    npg = [(t + PAGE - 1) // PAGE for t in ntok]
    total = sum(npg) * hkv
    w = max(1, -(-total // sms), (max(npg) + 61) // 63)
    ctas = items[:, 7]
    assert ctas[0] == 0 and np.all(np.diff(ctas) >= 0) and np.all(np.diff(ctas) <= 1)
    n_ctas = int(ctas[-1]) + 1
    assert n_ctas <= sms
    pages_of = np.zeros(n_ctas, dtype=np.int64)
    seen = {}
    for k, (r, h, piece, pieces, p0, tiles, first, cta) in enumerate(items.tolist()):
        seen.setdefault((r, h), []).append((k, piece, pieces, p0, tiles, first, cta))
    assert set(seen) == {(r, h) for r in range(len(ntok)) for h in range(hkv)}
    for (r, h), ps in seen.items():
        ks = [p[0] for p in ps]
        assert ks == list(range(ks[0], ks[0] + len(ps))), "a pair's pieces are consecutive"
        assert [p[1] for p in ps] == list(range(len(ps)))
        assert all(p[2] == len(ps) for p in ps) and len(ps) <= 64
        assert all(p[5] == ks[0] for p in ps), "first item of the pair"
        assert sum(p[4] for p in ps) == -(-ntok[r] // 128), "tiles cover exactly the attended tokens"
        if ntok[r] == 0:
            assert len(ps) == 1 and ps[0][4] == 0
        p0 = 0
        for i, p in enumerate(ps):
            assert p[3] == p0
            pages = p[4] // 2 if i + 1 < len(ps) else npg[r] - p0
            assert i + 1 == len(ps) or p[4] % 2 == 0, "inner pieces are whole pages"
            pages_of[p[6]] += pages
            p0 += pages
        assert p0 == npg[r]
    assert np.all(pages_of <= w), (pages_of.max(), w)
    # inside a CTA's list only the first and last items may be pieces of shared pairs
    for c in range(n_ctas):
        ks = np.nonzero(ctas == c)[0]
        for k in ks[1:-1]:
            assert items[k, 3] == 1 or all(items[j, 7] == c for j in range(items[k, 6], items[k, 6] + items[k, 3]))
    return n_ctas, int(pages_of.max()), w


def test_plan_small_example():
    ctx = _ctx(2, max_pages=8)
    try:
        items = gp.gp_debug_attention_plan(ctx, [3 * PAGE - 100, 1, 0, 2 * PAGE], 4)
        # W = 12 pages / 4 SMs = 3: request 3's first head is split over CTAs 2 and 3
        expect = [[0, 0, 0, 1, 0, 6, 0, 0], [0, 1, 0, 1, 0, 6, 1, 1], [1, 0, 0, 1, 0, 1, 2, 2],
                  [1, 1, 0, 1, 0, 1, 3, 2], [2, 0, 0, 1, 0, 0, 4, 2], [2, 1, 0, 1, 0, 0, 5, 2],
                  [3, 0, 0, 2, 0, 2, 6, 2], [3, 0, 1, 2, 1, 2, 6, 3], [3, 1, 0, 1, 0, 4, 8, 3]]
        assert items.tolist() == expect
    finally:
        gp.gp_destroy(ctx)


def test_plan_balances_equal_pairs():
    """16 requests of 128 pages, 8 KV heads over 152 SMs: every range within
    108 pages (a split per pair gives ranges of 128)."""
    ctx = _ctx(8)
    try:
        items = gp.gp_debug_attention_plan(ctx, [128 * PAGE] * 16, 152)
        n_ctas, most, w = _check_plan(items, [128 * PAGE] * 16, 8, 152)
        assert n_ctas == 152 and most == w == 108
    finally:
        gp.gp_destroy(ctx)


@pytest.mark.parametrize("hkv", [1, 2, 8])
@pytest.mark.parametrize("sms", [1, 7, 152])
def test_plan_invariants_on_seeded_mixes(hkv, sms):
    rng = np.random.default_rng(1000 * hkv + sms)
    ctx = _ctx(hkv)
    try:
        for _ in range(40):
            n = int(rng.integers(1, 48))
            ntok = [int(rng.integers(0, PAGE * int(rng.integers(1, 257)) + 1)) for _ in range(n)]
            if rng.random() < 0.2:
                ntok[int(rng.integers(0, n))] = 0
            items = gp.gp_debug_attention_plan(ctx, ntok, sms)
            _check_plan(items, ntok, hkv, sms)
        # one long request on one KV head: pieces capped at 64
        items = gp.gp_debug_attention_plan(ctx, [256 * PAGE], sms)
        _check_plan(items, [256 * PAGE], hkv, sms)
        with pytest.raises(gp.GrowPageError):
            gp.gp_debug_attention_plan(ctx, [257 * PAGE], sms)
    finally:
        gp.gp_destroy(ctx)
