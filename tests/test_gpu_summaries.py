"""The summary update (GrowPage Sec. 3.2 Eq. 6 with the App. E.1 first-step
initialisation) element by element against its exactly rounded value.

The kernel evaluates Eq. 6 in fp64 as one fused multiply-add per element,
qbar <- RN(beta * qbar + c) with c = RN((1 - beta) * q) (the product read from
a per-block table of rounded products, or an fp64 multiply for the queries
the table does not cover; the multiply-add on the fp64 pipe).  Each new value is
checked against the nearest double (ties to even) of the exact rational
beta * old + c, computed with fractions.Fraction, so the check rests on
IEEE 754's rounding rule alone.  The queries span magnitudes 2^-30 .. 2^30,
include zeros, and steer the short and long summaries into near-total
cancellation.  The fused update inside decode attention must give the same
bits.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import paged_kv_cache_step_gb300 as gp

pytestmark = pytest.mark.gpu

L, HQ, HKV, D = 2, 8, 2, 128
BETA = (0.9, 0.999)


def _ctx(n):
    k = torch.zeros(L, 2, HKV, 256, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    cfg = gp.gp_config_default(num_layers=L, num_q_heads=HQ, num_kv_heads=HKV, head_dim=D, kv_dtype=0, q_dtype=0,
                               max_slots=n, num_pages=2, max_pages_per_req=2, rope_theta=1e4)
    ctx = gp.gp_create(cfg, k, v, None)
    return ctx, k, v, [gp.gp_slot_acquire(ctx) for _ in range(n)]


def _queries(g, n, prev=None):
    """bf16 queries [L][n][Hq][D]: spread magnitudes, zeros, and (given the
    summaries before the step) values that cancel most of beta * old."""
    q = torch.randn(L, n, HQ, D, generator=g, dtype=torch.float64)
    q *= torch.exp2(torch.randint(-30, 31, (L, n, HQ, D), generator=g).double())
    q[torch.rand(L, n, HQ, D, generator=g) < 0.02] = 0.0
    if prev is not None:
        pick = torch.randint(0, 4, (L, n, HQ, D), generator=g)
        for x, beta in enumerate(BETA):
            cancel = torch.from_numpy(-beta / (1.0 - beta) * prev[:, :, x])
            q = torch.where(pick == x + 1, cancel, q)
    return q.to(torch.bfloat16)


def _read(ctx, slots):
    return np.stack([gp.gp_read_summaries(ctx, s, L, HQ, D) for s in slots], axis=1)  # [L][n][2][Hq][D]


def _rounded_update(old, q):
    """RN(beta * old + RN((1 - beta) q)) per element, exactly."""
    out = np.empty_like(old)
    for x, beta in enumerate(BETA):
        fb, w = Fraction(beta), 1.0 - beta
        o = old[:, :, x].reshape(-1)
        qq = q.reshape(-1)
        r = out[:, :, x].reshape(-1)
        for i in range(o.size):
            ov = float(o[i])
            c = w * float(qq[i])  # one correctly rounded fp64 product
            exact = fb * Fraction(ov) + Fraction(c)
            if exact == 0:  # IEEE 754: -0 only for (-0) + (-0), else +0
                r[i] = -0.0 if (np.signbit(ov) and np.signbit(c)) else 0.0
            else:
                r[i] = float(exact)
        out[:, :, x] = r.reshape(out[:, :, x].shape)
    return out


def test_summary_update_is_one_correctly_rounded_fma():
    n = 3
    ctx, _, _, slots = _ctx(n)
    g = torch.Generator().manual_seed(11)
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    first = torch.ones(n, dtype=torch.uint8, device="cuda")
    nfirst = torch.zeros_like(first)
    try:
        q0 = _queries(g, n)
        gp.gp_update_summaries(ctx, n, sl, q0.cuda(), first)
        s = _read(ctx, slots)
        q0d = q0.double().numpy()
        for x in range(2):  # the first step sets both summaries to the query
            assert np.array_equal(s[:, :, x], q0d)
        for step in range(4):
            old = _read(ctx, slots)
            q = _queries(g, n, prev=old)
            gp.gp_update_summaries(ctx, n, sl, q.cuda(), nfirst)
            got = _read(ctx, slots)
            want = _rounded_update(old, q.double().numpy())
            bad = np.flatnonzero(got.view(np.int64) != want.view(np.int64))
            assert bad.size == 0, (f"step {step}: {bad.size} elements differ, first at {bad[0]}: "
                                   f"got {got.reshape(-1)[bad[0]]!r} want {want.reshape(-1)[bad[0]]!r}")
    finally:
        gp.gp_destroy(ctx)


def _edge_queries(g, n):
    """bf16 queries at the edges of the format: subnormals (which the kernel
    multiplies in fp64 instead of taking its product table), the smallest and
    largest normal exponents, and ordinary values beside them."""
    bits = torch.randint(0x0080, 0x7f80, (L, n, HQ, D), generator=g, dtype=torch.int32)
    kind = torch.randint(0, 5, (L, n, HQ, D), generator=g)
    bits = torch.where(kind == 0, torch.randint(1, 0x80, bits.shape, generator=g, dtype=torch.int32), bits)  # subnormal
    bits = torch.where(kind == 1, 0x0080 + torch.randint(0, 0x80, bits.shape, generator=g, dtype=torch.int32), bits)
    bits = torch.where(kind == 2, 0x7f00 + torch.randint(0, 0x80, bits.shape, generator=g, dtype=torch.int32), bits)
    sign = torch.randint(0, 2, bits.shape, generator=g, dtype=torch.int32) << 15
    return (bits | sign).to(torch.int16).view(torch.bfloat16)


def test_summary_update_edge_queries():
    """Subnormal and extreme-exponent bf16 queries take the same correctly
    rounded update; an infinite or NaN query gives the IEEE 754 result."""
    n = 2
    ctx, _, _, slots = _ctx(n)
    g = torch.Generator().manual_seed(23)
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    first = torch.ones(n, dtype=torch.uint8, device="cuda")
    nfirst = torch.zeros_like(first)
    try:
        gp.gp_update_summaries(ctx, n, sl, _queries(g, n).cuda(), first)
        for step in range(2):
            old = _read(ctx, slots)
            q = _edge_queries(g, n)
            gp.gp_update_summaries(ctx, n, sl, q.cuda(), nfirst)
            got = _read(ctx, slots)
            want = _rounded_update(old, q.double().numpy())
            bad = np.flatnonzero(got.view(np.int64) != want.view(np.int64))
            assert bad.size == 0, (f"step {step}: {bad.size} elements differ, first at {bad[0]}: "
                                   f"got {got.reshape(-1)[bad[0]]!r} want {want.reshape(-1)[bad[0]]!r}")
        # non-finite queries on a few elements of otherwise ordinary rows
        old = _read(ctx, slots)
        q = _queries(g, n).double()
        special = torch.zeros(q.shape, dtype=torch.bool)
        special[0, 0, 0, :3] = True
        q[0, 0, 0, 0], q[0, 0, 0, 1], q[0, 0, 0, 2] = float("inf"), float("-inf"), float("nan")
        gp.gp_update_summaries(ctx, n, sl, q.to(torch.bfloat16).cuda(), nfirst)
        got = _read(ctx, slots)
        qd = q.to(torch.bfloat16).double().numpy()
        for x in range(2):
            assert got[0, 0, x, 0, 0] == np.inf and got[0, 0, x, 0, 1] == -np.inf
            assert np.isnan(got[0, 0, x, 0, 2])
        qd_f = np.where(special.numpy(), 0.0, qd)
        want = _rounded_update(old, qd_f)
        mask = np.broadcast_to(~special.numpy()[:, :, None], got.shape)
        assert np.array_equal(got.view(np.int64)[mask], want.view(np.int64)[mask])
    finally:
        gp.gp_destroy(ctx)


def test_fused_attention_update_gives_the_same_bits():
    n = 3
    ctxa, _, _, sa = _ctx(n)
    ctxb, _, _, sb = _ctx(n)
    g = torch.Generator().manual_seed(12)
    try:
        page = gp.gp_page_alloc(ctxb)  # zero keys: the attention itself is not under test here
        reqs = [gp.Request(s, [page], 256, 2) for s in sb]
        out = torch.empty(n, HQ, D, device="cuda")
        sla = torch.tensor(sa, dtype=torch.int32, device="cuda")
        first = torch.ones(n, dtype=torch.uint8, device="cuda")
        nfirst = torch.zeros_like(first)
        prev = None
        for step in range(6):
            q = _queries(g, n, prev=prev).cuda()
            f = first if step == 0 else nfirst
            gp.gp_update_summaries(ctxa, n, sla, q, f)
            for layer in range(L):
                gp.gp_decode_attention(ctxb, layer, reqs, [256] * n, q[layer].contiguous(), f, out)
            torch.cuda.synchronize()
            prev = _read(ctxa, sa)
            assert np.array_equal(prev.view(np.int64), _read(ctxb, sb).view(np.int64)), f"step {step}"
    finally:
        gp.gp_destroy(ctxa)
        gp.gp_destroy(ctxb)


def test_summary_update_full_size_sampled():
    """The batch workload's size: 64 requests of the Llama-8B shape (32
    layers, 32 query heads, d = 128; a 134 MB pool, larger than L2), one
    first step and two updates, 20,000 sampled elements of each summary
    checked against the exactly rounded value."""
    L8, HQ8, D8, n = 32, 32, 128, 64
    k = torch.zeros(L8, 2, 8, 256, D8, dtype=torch.bfloat16, device="cuda")
    cfg = gp.gp_config_default(num_layers=L8, num_q_heads=HQ8, num_kv_heads=8, head_dim=D8, kv_dtype=0, q_dtype=0,
                               max_slots=n, num_pages=2, max_pages_per_req=2, rope_theta=5e5)
    ctx = gp.gp_create(cfg, k, torch.zeros_like(k), None)
    g = torch.Generator().manual_seed(13)
    rng = np.random.default_rng(13)
    try:
        slots = [gp.gp_slot_acquire(ctx) for _ in range(n)]
        sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
        first = torch.ones(n, dtype=torch.uint8, device="cuda")
        q = torch.randn(L8, n, HQ8, D8, generator=g).to(torch.bfloat16)
        gp.gp_update_summaries(ctx, n, sl, q.cuda(), first)
        for step in range(2):
            old = np.stack([gp.gp_read_summaries(ctx, s, L8, HQ8, D8) for s in slots], axis=1)
            q = (torch.randn(L8, n, HQ8, D8, generator=g) * (1 + step)).to(torch.bfloat16)
            gp.gp_update_summaries(ctx, n, sl, q.cuda(), torch.zeros_like(first))
            got = np.stack([gp.gp_read_summaries(ctx, s, L8, HQ8, D8) for s in slots], axis=1)
            qd = q.double().numpy()
            for x, beta in enumerate(BETA):
                fb, w = Fraction(beta), 1.0 - beta
                idx = rng.integers(0, qd.size, size=20000)
                o, gx, qq = old[:, :, x].reshape(-1), got[:, :, x].reshape(-1), qd.reshape(-1)
                for i in idx:
                    want = float(fb * Fraction(float(o[i])) + Fraction(w * float(qq[i])))
                    assert gx[i] == want, f"step {step} summary {x} element {i}: {gx[i]!r} != {want!r}"
    finally:
        gp.gp_destroy(ctx)
