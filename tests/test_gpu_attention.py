"""Decode attention with the summary update fused in (gp_decode_attention),
through the C ABI, against the fp64 oracle.

* Attention: RoPE of the pre-RoPE query at the request's position, logits
  over the first num_tokens logical slots (keys stored rotated), softmax,
  the weighted sum of values.  Tolerance: |out - ref| <= 1e-4 * max|v| + 1e-5
  * |ref| (fp32 dot products over d and fp32 sums over up to 33k weights).
* Summaries: the layer's two summaries updated exactly as the standalone
  update does (fp64 on both sides), other layers untouched.
* Theorem 3.1 on the whole path: after Compress & Hold, attention over the
  compacted cache equals the oracle's renormalised output o^(S) of the full
  distribution over the kept set S (Eq. 3), and ||o - o^(S)||_2 <=
  2 Vmax (1 - m(S)) (Eq. 5) with Vmax the largest value norm.
"""

import numpy as np
import pytest
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp
import synth
from synth.workloads import ModelShape

import harness as hz

pytestmark = pytest.mark.gpu

PAGE = 256
SHAPES = {
    "bf16_g4_d128": ModelShape(2, 8, 2, 128, "bf16", "bf16", 5.0e5),
    "bf16_g2_d128": ModelShape(2, 4, 2, 128, "bf16", "bf16", 5.0e5),
    "bf16_g2_d64": ModelShape(2, 4, 2, 64, "bf16", "bf16", 1.0e4),
    "f32_g4_d128": ModelShape(2, 8, 2, 128, "f32", "f32", 5.0e5),
}
# the kernels each shape runs on: the tensor-core kernel (forced, so that a
# shape it cannot take fails instead of falling back) where it applies, and
# the CUDA-core kernel everywhere
KERNELS = {"tensor_core": gp.GP_SCAN_TENSOR_CORE, "cuda_core": gp.GP_SCAN_CUDA_CORE}
CASES = [(s, k) for s in sorted(SHAPES) for k in sorted(KERNELS)
         if k == "cuda_core" or (SHAPES[s].kv_dtype == "bf16" and SHAPES[s].head_dim == 128)]


def _oracle_attention(q_pre, keys, values, pos, theta):
    """q_pre [G][d] pre-RoPE; keys/values [N][d] (rotated keys); -> [G][d]."""
    qr = og.rope(q_pre, pos, theta)
    a = og.softmax(og.logits(qr, keys))
    return a @ values, a


@pytest.mark.parametrize("shape_name,kernel", CASES)
def test_decode_attention_matches_oracle(shape_name, kernel):
    sh = SHAPES[shape_name]
    sizes = [1, 3, 33, 5]
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=sizes, seed_xor=41)
    run = hz.EngineRun(w)
    try:
        gp.gp_set_scan_kernel(run.ctx, KERNELS[kernel])
        run.feed_history()
        n = len(sizes)
        ntok = [PAGE, 3 * PAGE - 100, 1, 0]
        layer = 1
        dt = torch.float32 if sh.q_dtype == "f32" else torch.bfloat16
        q = torch.randn(n, sh.num_q_heads, sh.head_dim, device="cuda").to(dt)
        first = torch.zeros(n, dtype=torch.uint8, device="cuda")
        first[0] = 1
        before = [gp.gp_read_summaries(run.ctx, r.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
                  for r in run.reqs]
        out = torch.full((n, sh.num_q_heads, sh.head_dim), float("nan"), device="cuda")
        gp.gp_decode_attention(run.ctx, layer, run.reqs, ntok, q, first, out)
        torch.cuda.synchronize()
        out = out.cpu().numpy().astype(np.float64)
        qn = q.double().cpu().numpy()
        G = sh.group
        for r, req in enumerate(run.reqs):
            # summaries: this layer updated as Eq. 6 / App. E.1 say, the other untouched
            after = gp.gp_read_summaries(run.ctx, req.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            s_new, l_new = og.ema_update(before[r][layer, 0], before[r][layer, 1], qn[r], bool(first[r]), 0.9, 0.999)
            for x, ref in ((0, s_new), (1, l_new)):
                scale = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)) + 1e-30
                assert np.max(np.abs(after[layer, x] - ref) / scale) <= hz.SUMMARY_REL
            assert np.array_equal(after[1 - layer], before[r][1 - layer])
            for h in range(sh.num_kv_heads):
                keys = hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:ntok[r]]
                vals = hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:ntok[r]]
                got = out[r, h * G:(h + 1) * G]
                if ntok[r] == 0:
                    assert np.all(got == 0.0)
                    continue
                ref, _ = _oracle_attention(qn[r, h * G:(h + 1) * G], keys, vals, req.pos, sh.rope_theta)
                tol = 1e-4 * np.abs(vals).max() + 1e-5 * np.abs(ref)
                assert np.all(np.abs(got - ref) <= tol), \
                    f"{shape_name} request {r} head {h}: error {np.abs(got - ref).max()}"
    finally:
        run.close()


def test_fused_update_equals_standalone_update():
    sh = SHAPES["bf16_g4_d128"]
    wa = synth.make_workload("custom", device="cuda", shape=sh, sizes=[4, 9], seed_xor=42)
    wb = synth.make_workload("custom", device="cuda", shape=sh, sizes=[4, 9], seed_xor=42)
    ra, rb = hz.EngineRun(wa), hz.EngineRun(wb)
    try:
        out = torch.empty(2, sh.num_q_heads, sh.head_dim, device="cuda")
        for t, q in enumerate(wa.history[:8]):
            ra.update(q, t == 0)
            first = (rb.first_dev if t == 0 else rb.notfirst_dev)
            for layer in range(sh.num_layers):
                gp.gp_decode_attention(rb.ctx, layer, rb.reqs, [x.num_pages * PAGE for x in rb.reqs],
                                       q[layer].contiguous(), first, out)
        torch.cuda.synchronize()
        for x, y in zip(ra.reqs, rb.reqs):
            sa = gp.gp_read_summaries(ra.ctx, x.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            sb = gp.gp_read_summaries(rb.ctx, y.slot, sh.num_layers, sh.num_q_heads, sh.head_dim)
            scale = np.sqrt(np.mean(sa * sa, axis=-1, keepdims=True)) + 1e-30
            assert np.max(np.abs(sa - sb) / scale) <= hz.SUMMARY_REL
    finally:
        ra.close()
        rb.close()


def test_theorem31_bound_after_compress_and_hold():
    """Attention before and after Compress & Hold for the same query: the
    compacted result is o^(S), and the error stays within 2 Vmax (1 - m(S))."""
    sh = SHAPES["bf16_g4_d128"]
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=[33, 8], seed_xor=43)
    run = hz.EngineRun(w)
    try:
        run.feed_history()
        gp.gp_boundary_demand(run.ctx, run.reqs, w.history[-1])
        n, G = len(run.reqs), sh.group
        tables = [list(x.pages) for x in run.reqs]
        P = [x.num_pages for x in run.reqs]
        pre_k = {(r, l, h): hz.unit_keys_dev(w.k_cache, tables[r], l, h)
                 for r in range(n) for l in range(sh.num_layers) for h in range(sh.num_kv_heads)}
        pre_v = {(r, l, h): hz.unit_keys_dev(w.v_cache, tables[r], l, h)
                 for r in range(n) for l in range(sh.num_layers) for h in range(sh.num_kv_heads)}
        q = torch.randn(sh.num_layers, n, sh.num_q_heads, sh.head_dim, device="cuda").to(torch.bfloat16)
        notfirst = torch.zeros(n, dtype=torch.uint8, device="cuda")
        full = torch.empty(sh.num_layers, n, sh.num_q_heads, sh.head_dim, device="cuda")
        for layer in range(sh.num_layers):
            gp.gp_decode_attention(run.ctx, layer, run.reqs, [p * PAGE for p in P], q[layer].contiguous(),
                                   notfirst, full[layer])
        gp.gp_compress_hold(run.ctx, run.reqs)
        comp = torch.empty_like(full)
        for layer in range(sh.num_layers):
            gp.gp_decode_attention(run.ctx, layer, run.reqs, [(p - 1) * PAGE for p in P], q[layer].contiguous(),
                                   notfirst, comp[layer])
        torch.cuda.synchronize()
        full, comp = full.cpu().numpy().astype(np.float64), comp.cpu().numpy().astype(np.float64)
        qn = q.double().cpu().numpy()
        checked = 0
        for r in range(n):
            masks = gp.unpack_mask(gp.gp_debug_keep_mask(run.ctx, r, run.units, P[r]), P[r] * PAGE)
            pos = run.reqs[r].pos
            for layer in range(sh.num_layers):
                for h in range(sh.num_kv_heads):
                    keep = masks[layer * sh.num_kv_heads + h]
                    keys, vals = pre_k[(r, layer, h)], pre_v[(r, layer, h)]
                    o, a = _oracle_attention(qn[layer, r, h * G:(h + 1) * G], keys, vals, pos, sh.rope_theta)
                    vmax = np.linalg.norm(vals, axis=1).max()
                    for gi in range(G):
                        S = np.nonzero(keep)[0]
                        o_s = og.renormalised_output(a[gi], vals, S)
                        m_s = a[gi][S].sum()
                        got_full = full[layer, r, h * G + gi]
                        got_comp = comp[layer, r, h * G + gi]
                        tol = 1e-4 * np.abs(vals).max()
                        assert np.abs(got_full - o[gi]).max() <= tol + 1e-5 * np.abs(o[gi]).max()
                        assert np.abs(got_comp - o_s).max() <= tol + 1e-5 * np.abs(o_s).max(), \
                            f"request {r} layer {layer} head {h * G + gi}: compacted output is not o^(S)"
                        bound = og.worst_case_error(a[gi], S, vmax)
                        assert np.linalg.norm(got_full - got_comp) <= bound + 1e-3 * vmax
                        checked += 1
        assert checked == n * sh.num_layers * sh.num_q_heads
    finally:
        run.close()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_decode_attention_multi_page_splits(kernel):
    """Enough pages that a split spans several pages (the persistent
    tensor-core kernel cuts all pairs' pages into one even range per SM, so
    the long requests' pairs are shared between CTAs; the CUDA-core kernel
    aims at six waves of two CTAs per SM, 1824 CTAs, where the 64-split cap
    applies to the longest request); ragged token counts end inside a tile
    or stage."""
    sh = SHAPES["bf16_g4_d128"]
    sizes = [160, 150, 130, 97, 40, 5]  # 582 pages x 2 KV heads: 1 or 2 pages per CUDA-core CTA, 8 per tensor-core one
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=sizes, seed_xor=44)
    run = hz.EngineRun(w)
    try:
        gp.gp_set_scan_kernel(run.ctx, KERNELS[kernel])
        run.feed_history()
        n, G, layer = len(sizes), sh.group, 0
        ntok = [160 * PAGE, 150 * PAGE - 77, 130 * PAGE - 1, 97 * PAGE - 255, 40 * PAGE - 128, 5 * PAGE - 130]
        q = torch.randn(n, sh.num_q_heads, sh.head_dim, device="cuda").to(torch.bfloat16)
        first = torch.zeros(n, dtype=torch.uint8, device="cuda")
        out = torch.full((n, sh.num_q_heads, sh.head_dim), float("nan"), device="cuda")
        gp.gp_decode_attention(run.ctx, layer, run.reqs, ntok, q, first, out)
        torch.cuda.synchronize()
        out = out.cpu().numpy().astype(np.float64)
        qn = q.double().cpu().numpy()
        for r, req in enumerate(run.reqs):
            for h in range(sh.num_kv_heads):
                keys = hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:ntok[r]]
                vals = hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:ntok[r]]
                ref, _ = _oracle_attention(qn[r, h * G:(h + 1) * G], keys, vals, req.pos, sh.rope_theta)
                got = out[r, h * G:(h + 1) * G]
                tol = 1e-4 * np.abs(vals).max() + 1e-5 * np.abs(ref)
                assert np.all(np.abs(got - ref) <= tol), \
                    f"request {r} head {h}: error {np.abs(got - ref).max()}"
    finally:
        run.close()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_unattended_slots_do_not_reach_the_output(kernel):
    """The slots past num_tokens in a request's last attended page may hold
    any bits (the caller's cache): filled here with NaN and +-inf in K and V,
    they must change nothing -- their weight is 0, and 0 x inf must not
    reach the output through the weighted sum.  The output buffer starts 4
    bytes into its allocation, so the 16-byte stores of the merge must not
    be taken for granted either."""
    sh = SHAPES["bf16_g4_d128"]
    sizes = [3, 2, 1]
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=sizes, seed_xor=45)
    run = hz.EngineRun(w)
    try:
        gp.gp_set_scan_kernel(run.ctx, KERNELS[kernel])
        run.feed_history()
        n, G, layer = len(sizes), sh.group, 1
        ntok = [2 * PAGE + 77, PAGE + 1, 130]
        for req, t in zip(run.reqs, ntok):
            pg, off = req.pages[t // PAGE], t % PAGE
            w.k_cache[:, pg, :, off:] = float("nan")
            w.v_cache[:, pg, :, off::2] = float("inf")
            w.v_cache[:, pg, :, off + 1::2] = float("-inf")
            w.v_cache[:, pg, :, off::3] = float("nan")
        q = torch.randn(n, sh.num_q_heads, sh.head_dim, device="cuda").to(torch.bfloat16)
        first = torch.zeros(n, dtype=torch.uint8, device="cuda")
        flat = torch.full((n * sh.num_q_heads * sh.head_dim + 1,), float("nan"), device="cuda")
        out = flat[1:].view(n, sh.num_q_heads, sh.head_dim)
        assert out.data_ptr() % 16 == 4
        gp.gp_decode_attention(run.ctx, layer, run.reqs, ntok, q, first, out)
        torch.cuda.synchronize()
        assert torch.isnan(flat[0])  # nothing written before the buffer
        out = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(out))
        qn = q.double().cpu().numpy()
        for r, req in enumerate(run.reqs):
            for h in range(sh.num_kv_heads):
                keys = hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:ntok[r]]
                vals = hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:ntok[r]]
                assert np.all(np.isfinite(keys)) and np.all(np.isfinite(vals))
                ref, _ = _oracle_attention(qn[r, h * G:(h + 1) * G], keys, vals, req.pos, sh.rope_theta)
                got = out[r, h * G:(h + 1) * G]
                tol = 1e-4 * np.abs(vals).max() + 1e-5 * np.abs(ref)
                assert np.all(np.abs(got - ref) <= tol), f"request {r} head {h}: error {np.abs(got - ref).max()}"
    finally:
        run.close()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_decode_attention_many_requests(kernel):
    """More pairs than SMs: the persistent tensor-core kernel's CTAs take
    several items each -- whole pairs, pieces of pairs shared with the
    neighbouring range, empty ones (no attended token), one-token ones, and
    the pieces of a long request; every output against the oracle."""
    sh = SHAPES["bf16_g4_d128"]
    rng = np.random.default_rng(46)
    sizes = [int(x) for x in rng.integers(1, 4, size=95)] + [40]
    w = synth.make_workload("custom", device="cuda", shape=sh, sizes=sizes, seed_xor=46)
    run = hz.EngineRun(w)
    try:
        gp.gp_set_scan_kernel(run.ctx, KERNELS[kernel])
        run.feed_history()
        n, G, layer = len(sizes), sh.group, 1
        ntok = [int(rng.integers(0, p * PAGE + 1)) for p in sizes]
        ntok[0], ntok[1], ntok[-1] = 0, 1, 40 * PAGE - 3
        q = torch.randn(n, sh.num_q_heads, sh.head_dim, device="cuda").to(torch.bfloat16)
        first = torch.zeros(n, dtype=torch.uint8, device="cuda")
        out = torch.full((n, sh.num_q_heads, sh.head_dim), float("nan"), device="cuda")
        gp.gp_decode_attention(run.ctx, layer, run.reqs, ntok, q, first, out)
        torch.cuda.synchronize()
        out = out.cpu().numpy().astype(np.float64)
        qn = q.double().cpu().numpy()
        for r, req in enumerate(run.reqs):
            for h in range(sh.num_kv_heads):
                got = out[r, h * G:(h + 1) * G]
                if ntok[r] == 0:
                    assert np.all(got == 0.0)
                    continue
                keys = hz.unit_keys_dev(w.k_cache, req.pages, layer, h)[:ntok[r]]
                vals = hz.unit_keys_dev(w.v_cache, req.pages, layer, h)[:ntok[r]]
                ref, _ = _oracle_attention(qn[r, h * G:(h + 1) * G], keys, vals, req.pos, sh.rope_theta)
                tol = 1e-4 * np.abs(vals).max() + 1e-5 * np.abs(ref)
                assert np.all(np.abs(got - ref) <= tol), f"request {r} head {h}: error {np.abs(got - ref).max()}"
    finally:
        run.close()
