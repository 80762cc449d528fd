"""Helpers shared by the GPU parity tests, __graft_entry__.smoke() and the
bench's CPU baseline: drive a synthetic workload through the C-ABI engine and
through the fp64 oracle, and compare them with the stated tolerances.

Tolerances (GrowPage boundary engine):
  * decision, page tables, gathered K/V bytes for a given index set: exact.
    The decision is checked twice: it must follow exactly from the GPU's own
    D_p values, and it must equal the oracle's unless the units where the two
    D_p differ by the allowed 1 (t of them) could move the demand difference
    across zero, i.e. unless -t < (sum K^S - sum K^L)_oracle <= t;
  * D_p: may differ by 1, only where the oracle's sorted cumulative mass at
    the crossing lies within 1e-6 (relative) of p;
  * top-k sets: identical except members whose oracle score is within 1e-5
    (relative) of the k-th score (global fill or their block's local quota);
  * softmax probabilities: within 1e-4 absolute;
  * summaries (fp64 on both sides; only the FMA rounding differs): within
    1e-12 relative to the row scale.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle.growpage as og
import paged_kv_cache_step_gb300 as gp

PAGE = 256
DP_TIE_REL = 1e-6
TOPK_REL = 1e-5
PROB_ABS = 1e-4
SUMMARY_REL = 1e-12


# ---------------------------------------------------------------------------
# engine setup
# ---------------------------------------------------------------------------

def engine_config(w, **over):
    sh = w.shape
    cfg = gp.gp_config_default(
        num_layers=sh.num_layers, num_q_heads=sh.num_q_heads, num_kv_heads=sh.num_kv_heads,
        head_dim=sh.head_dim,
        kv_dtype=gp.GP_DTYPE_F32 if sh.kv_dtype == "f32" else gp.GP_DTYPE_BF16,
        q_dtype=gp.GP_DTYPE_F32 if sh.q_dtype == "f32" else gp.GP_DTYPE_BF16,
        max_slots=max(4, w.n), num_pages=w.num_pages, max_pages_per_req=256,
        rope_theta=sh.rope_theta)
    for k, v in over.items():
        setattr(cfg, k, v)
    return cfg


class EngineRun:
    """An engine bound to a workload's caches, with the workload's requests."""

    def __init__(self, w, stream=None, **cfg_over):
        self.w = w
        self.cfg = engine_config(w, **cfg_over)
        self.ctx = gp.gp_create(self.cfg, w.k_cache, w.v_cache, stream)
        # mirror the workload's page ownership in the engine's pool
        used = set()
        for bt in w.block_tables:
            used.update(bt)
        for _ in range(w.num_pages):
            gp.gp_page_alloc(self.ctx)
        for pg in range(w.num_pages):
            if pg not in used:
                gp.gp_page_unref(self.ctx, pg)
        self.reqs = []
        for r, bt in enumerate(w.block_tables):
            slot = gp.gp_slot_acquire(self.ctx)
            self.reqs.append(gp.Request(slot, bt, w.positions[r], self.cfg.max_pages_per_req))
        dev = w.device
        self.slots_dev = torch.tensor([q.slot for q in self.reqs], dtype=torch.int32, device=dev)
        self.first_dev = torch.ones(len(self.reqs), dtype=torch.uint8, device=dev)
        self.notfirst_dev = torch.zeros(len(self.reqs), dtype=torch.uint8, device=dev)

    def close(self):
        if self.ctx:
            gp.gp_destroy(self.ctx)
            self.ctx = None

    def update(self, q, first: bool):
        gp.gp_update_summaries(self.ctx, len(self.reqs), self.slots_dev, q.contiguous(),
                               self.first_dev if first else self.notfirst_dev)

    def feed_history(self):
        for t, q in enumerate(self.w.history):
            self.update(q, t == 0)

    @property
    def units(self):
        return self.cfg.num_layers * self.cfg.num_kv_heads


# ---------------------------------------------------------------------------
# oracle side
# ---------------------------------------------------------------------------

def oracle_cfg(w, p=0.99, recent=16):
    return {"num_kv_heads": w.shape.num_kv_heads, "rope_theta": w.shape.rope_theta,
            "page_size": w.page_size, "recent_window": recent, "p": p}


def oracle_summaries(history, req: int, beta_s=0.9, beta_l=0.999):
    """Oracle EMA over a history of [L][n][Hq][d] tensors for request req."""
    s = l = None
    for t, q in enumerate(history):
        qr = q[:, req].double().cpu().numpy()
        s, l = og.ema_update(s, l, qr, t == 0, beta_s, beta_l)
    return s, l


def cache_f64(cache: torch.Tensor, pages) -> dict:
    """float64 copy of the given physical pages: {page: [L][Hkv][b][d]}."""
    idx = torch.as_tensor(list(pages), device=cache.device, dtype=torch.long)
    sub = cache.index_select(1, idx).double().cpu().numpy()
    return {pg: sub[:, i] for i, pg in enumerate(pages)}


def unit_keys_dev(cache: torch.Tensor, table, layer: int, h: int) -> np.ndarray:
    """float64 keys (or values) of one (layer, KV head) in logical order,
    copied from the device cache without touching the other units."""
    idx = torch.as_tensor(list(table), device=cache.device, dtype=torch.long)
    sub = cache[layer].index_select(0, idx)[:, h]          # [P][b][d]
    return sub.double().cpu().numpy().reshape(len(table) * PAGE, -1)


def oracle_unit_dev(qt, cache: torch.Tensor, table, layer, h, G, p=0.99, recent=16):
    qt_unit = qt[layer][:, h * G:(h + 1) * G, :]
    keys = unit_keys_dev(cache, table, layer, h)
    return og.unit_boundary(qt_unit, keys, len(table), PAGE, recent, p)


def unit_keys(pages_f64: dict, table, layer: int, h: int):
    return np.concatenate([pages_f64[pg][layer, h] for pg in table], axis=0)


def oracle_unit(qt, pages_f64, table, layer, h, G, p=0.99, recent=16):
    qt_unit = qt[layer][:, h * G:(h + 1) * G, :]
    keys = unit_keys(pages_f64, table, layer, h)
    return og.unit_boundary(qt_unit, keys, len(table), PAGE, recent, p)


# ---------------------------------------------------------------------------
# comparisons
# ---------------------------------------------------------------------------

def dp_ok(gpu_k: int, a_oracle: np.ndarray, p: float):
    """D_p within the stated tolerance.  Returns (ok, detail)."""
    k, before, at = og.coverage_demand_detail(a_oracle, p)
    if gpu_k == k:
        return True, ""
    if gpu_k == k + 1 and (at - p) <= DP_TIE_REL * p:
        return True, "tie-above"
    if gpu_k == k - 1 and (p - before) <= DP_TIE_REL * p:
        return True, "tie-below"
    return False, f"gpu {gpu_k} oracle {k} (C_(D-1)={before!r}, C_D={at!r})"


def topk_ok(gpu_keep: np.ndarray, s: np.ndarray, P: int, recent=16, k_loc=64, drop=1):
    """Compare a GPU keep mask with the oracle's Eq. 10 selection.

    Returns (ok, n_diff, message).  Differences are allowed only for slots
    whose oracle score is within 1e-5 (relative) of the global k-th score or
    of their own block's local k-th score.
    """
    b = PAGE
    n = P * b
    ncmp = n - recent
    kt = (P - drop) * b - recent
    ref = og.select_retained(s, P, b, recent, k_loc, drop)
    gk = np.asarray(gpu_keep[:n], dtype=bool)
    # validity of the GPU set on its own
    if gk.sum() != (P - drop) * b:
        return False, -1, f"kept {gk.sum()} != {(P - drop) * b}"
    if not gk[ncmp:].all():
        return False, -1, "recent window not kept"
    quota = min(k_loc, kt // P)
    local_thr = np.full(P, np.nan)
    for j in range(P):
        lo, hi = j * b, min((j + 1) * b, ncmp)
        kj = min(quota, hi - lo)
        if kj > 0:
            order = sorted(range(lo, hi), key=lambda i: (-s[i], i))
            local_thr[j] = s[order[kj - 1]]
            if gk[lo:hi].sum() < kj:
                return False, -1, f"block {j} keeps fewer than {kj}"
    # global k-th score: the smallest score the oracle adds in the global fill
    loc = np.zeros(n, bool)
    for j in range(P):
        lo, hi = j * b, min((j + 1) * b, ncmp)
        kj = min(quota, hi - lo)
        order = sorted(range(lo, hi), key=lambda i: (-s[i], i))
        loc[order[:kj]] = True
    glob = ref & ~loc
    glob[ncmp:] = False
    gthr = s[glob[:ncmp]].min() if glob.any() else np.nan
    diff = np.nonzero(gk != ref)[0]
    bad = []
    for i in diff:
        si = s[i]
        near_g = not np.isnan(gthr) and abs(si - gthr) <= TOPK_REL * gthr
        lt = local_thr[i // b] if i < ncmp else np.nan
        near_l = not np.isnan(lt) and abs(si - lt) <= TOPK_REL * lt
        if not (near_g or near_l):
            bad.append(int(i))
    if bad:
        return False, len(diff), f"{len(bad)} slots differ beyond tolerance, e.g. {bad[:5]}"
    return True, len(diff), ""


def summaries_ok(gpu: np.ndarray, ref: np.ndarray):
    """fp32 summaries vs fp64, relative to each row's RMS."""
    scale = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)) + 1e-30
    err = np.abs(gpu.astype(np.float64) - ref) / scale
    return float(err.max())


def decision_ok(act, k_oracle, k_gpu, num_pages, free_pages, reserve=0, tau=0.0):
    """The GrowPage decision (after Eq. 8, Sec. 4.2) of the GPU for one request.

    k_oracle, k_gpu: [units][2] D_p values (x = 0 short, 1 long) of the
    oracle and of the GPU, already checked unit by unit with dp_ok.  The
    GPU's action must (1) be og.decide applied to its own D_p values, and
    (2) equal og.decide applied to the oracle's unless the t tie units could
    flip Delta across tau.  Returns (ok, message)."""
    P = num_pages
    k_oracle = np.asarray(k_oracle, np.int64)
    k_gpu = np.asarray(k_gpu, np.int64)
    ncand = (P - 1) * PAGE
    d_gpu = og.demand_trend(k_gpu[:, 0], k_gpu[:, 1], ncand) if P > 1 else 0.0
    d_ora = og.demand_trend(k_oracle[:, 0], k_oracle[:, 1], ncand) if P > 1 else 0.0
    got = (int(act.kind), bool(act.fallback), bool(act.forced))
    mine = og.decide(d_gpu, P, free_pages, reserve, tau)
    if got != (mine.kind, mine.fallback, mine.forced):
        return False, f"action {got} does not follow from the GPU's own D_p (expected {mine})"
    ref = og.decide(d_ora, P, free_pages, reserve, tau)
    if got == (ref.kind, ref.fallback, ref.forced):
        return True, ""
    t = int(np.abs(k_gpu - k_oracle).sum())
    if P > 1 and tau == 0.0:
        diff = int(k_oracle[:, 0].sum() - k_oracle[:, 1].sum())
        ambiguous = -t < diff <= t
    else:
        ambiguous = P > 1 and abs(d_ora - tau) <= t / (ncand * len(k_oracle))
    if ambiguous:
        return True, "tie"
    return False, f"action {got} vs oracle {ref} with {t} tie units"


_POOL = None


def oracle_pool() -> ThreadPoolExecutor:
    """Threads for oracle work over many units (numpy and the device copies
    release the interpreter lock)."""
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(2, min(32, os.cpu_count() or 2)))
    return _POOL


def request_dp_check(w, req, qt, ks_gpu, keep=(), p=0.99, recent=16):
    """D_p of every (layer, KV head) unit of one request against the oracle.

    The oracle runs unit by unit on a thread pool (keys widened exactly to
    float64).  Returns (k_oracle [units][2], failures [str], {idx: UnitResult}
    for idx in keep)."""
    sh = w.shape
    units = sh.num_layers * sh.num_kv_heads
    keep = set(keep)

    def one(idx):
        layer, h = divmod(idx, sh.num_kv_heads)
        u = oracle_unit_dev(qt, w.k_cache, req.pages, layer, h, sh.group, p, recent)
        bad = []
        if req.num_pages > 1:
            for x in range(2):
                ok, msg = dp_ok(int(ks_gpu[idx, x]), u.a_dem[x], p)
                if not ok:
                    bad.append(f"unit {idx} x {x}: {msg}")
        return idx, np.array(u.k, np.int64), bad, (u if idx in keep else None)

    k_or = np.zeros((units, 2), np.int64)
    fails, kept = [], {}
    for idx, k, bad, u in oracle_pool().map(one, range(units)):
        k_or[idx] = k
        fails.extend(bad)
        if u is not None:
            kept[idx] = u
    return k_or, fails, kept
