"""Plain fp64 CPU oracle for GrowPage's capacity-boundary engine.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path (no kernels, headers, helpers or tables).

Every step is written out directly from its definition in the GrowPage paper
("GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning Serving",
arXiv 2609.03494), in float64, with no blocking, fusion or reordering beyond
what the definition states.  Library primitives used as single steps: matrix
products (numpy), a sort (numpy), cumulative sums (numpy).

Readings of the paper where it is silent or ambiguous:

* EMA convention: the stored beta is the decay, the weight on the previous
  summary (Sec. 3.2, Eq. 6); beta_S = 0.9 < beta_L = 0.999, so the short
  summary moves faster.
* Calibration and RoPE: Eq. 12 per (layer, query head), then rotate-half RoPE
  at the current decode position (App. E.1).  The RoPE variant and theta are
  not given by the paper: rotate-half with theta as a parameter is a
  convention, so its parity is "unpinned by the paper" beyond the generic
  rotation invariants the tests check.
* Logit scale 1/sqrt(d) (standard scaled dot-product attention; not stated).
* Demand candidates exclude the most recent physical block (Sec. 3.2,
  App. E.1): Cdem = [0, (P-1) b).  Compression candidates exclude only the
  protected recent window R (Sec. 3.3, Sec. 5.1): Ccmp = [0, P b - R).
* GQA: the per-KV-head distribution is the arithmetic mean of the G query
  heads' softmax distributions (App. E.1 keeps the native GQA mapping; Eqs. 7
  and 9 are per KV head).
* Decision: Grow iff Delta > tau, else Compress & Hold (Sec. 3.2, after
  Eq. 8); P = 1 forces Grow (nothing to compress); a Grow that the free pool
  cannot grant above the reserve becomes a fallback Compress (Sec. 4.2).
* Eq. 10 per-block quota k_loc' = min(k_loc, |B_j|, floor(K_t / P)); blocks
  are the request's logical 256-slot blocks; ties go to the lower slot index.
* Copy-on-write (App. E.2): every block-table entry with refcount > 1 is
  replaced by a fresh page, lowest free id first, in ascending logical order;
  private pages are kept in place.
"""

from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

import numpy as np

GROW = 0
COMPRESS = 1
SHRINK = 2


# ---------------------------------------------------------------------------
# input widening (exact)
# ---------------------------------------------------------------------------

def widen_bf16(bits) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns (uint16 array)."""
    u = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Sec. 3.2 Eq. 6 and App. E.1: dual-timescale query summaries
# ---------------------------------------------------------------------------

def ema_update(qbar_s, qbar_l, q, first: bool, beta_s: float, beta_l: float):
    """One decode step of the two summaries of one request.

    GrowPage, Sec. 3.2, Eq. 6: qbar^x_t = beta_x qbar^x_{t-1} + (1 - beta_x) q_t
    for x in {S, L}.  App. E.1 ("Initialization and online update"): on the
    first decoding step of a newly bound slot both summaries are set to q_t.
    Arrays are [L][Hq][d] (any shape works; the update is elementwise).
    """
    q = np.asarray(q, dtype=np.float64)
    if first:
        return q.copy(), q.copy()
    new_s = beta_s * np.asarray(qbar_s, np.float64) + (1.0 - beta_s) * q
    new_l = beta_l * np.asarray(qbar_l, np.float64) + (1.0 - beta_l) * q
    return new_s, new_l


# ---------------------------------------------------------------------------
# App. E.1 Eq. 12: RMS calibration, then RoPE at the current position
# ---------------------------------------------------------------------------

def rms(x, axis=-1):
    """Root mean square over the head dimension."""
    x = np.asarray(x, np.float64)
    return np.sqrt(np.mean(x * x, axis=axis))


def calibrate(qbar, q):
    """GrowPage, App. E.1, Eq. 12: gamma = RMS(q_t) / RMS(qbar), q~ = gamma qbar.

    Per (layer, query head): the last axis is the head dimension.  A zero
    summary gets gamma = 0 (the paper does not cover it).
    """
    qbar = np.asarray(qbar, np.float64)
    num = rms(q)
    den = rms(qbar)
    gamma = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
    return gamma[..., None] * qbar


def rope(x, pos: int, theta: float):
    """Rotate-half rotary embedding at position ``pos``.

    Pairs (i, i + d/2), i in [0, d/2), are rotated by pos * theta^(-2i/d).
    The paper applies RoPE to the calibrated summaries "using the current
    decoding position" (App. E.1) without fixing the variant; this is the
    common rotate-half form.
    """
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * np.power(float(theta), -2.0 * i / d)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def summary_queries(qbar_s, qbar_l, q, pos: int, theta: float):
    """Calibrated, rotated short and long summaries of one request.

    Inputs [L][Hq][d]; output [L][2][Hq][d] with x = 0 short, 1 long
    (App. E.1, Eq. 12 followed by RoPE at the current position).
    """
    out = []
    for qbar in (qbar_s, qbar_l):
        out.append(rope(calibrate(qbar, q), pos, theta))
    return np.stack(out, axis=1)


# ---------------------------------------------------------------------------
# Scores, softmax, GQA mean  (Sec. 3.2, App. E.1)
# ---------------------------------------------------------------------------

def logits(qrows, keys):
    """z[r, i] = q_r . k_i / sqrt(d) for query rows [R][d] and keys [N][d]."""
    qrows = np.asarray(qrows, np.float64)
    keys = np.asarray(keys, np.float64)
    return (qrows @ keys.T) / math.sqrt(qrows.shape[-1])


def softmax(z):
    """Row-wise softmax over the last axis (max-shifted, fp64)."""
    z = np.asarray(z, np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def kv_head_distribution(z_group):
    """Mean over the G query heads of a KV group of their softmax rows."""
    return np.mean(softmax(z_group), axis=0)


# ---------------------------------------------------------------------------
# Sec. 3.1 Eq. 2: p-coverage demand
# ---------------------------------------------------------------------------

def coverage_demand(a, p: float) -> int:
    """D_p(a) = min{k : sum_{i<=k} a_(i) >= p}, a_(1) >= a_(2) >= ... (Eq. 2)."""
    return coverage_demand_detail(a, p)[0]


def coverage_demand_detail(a, p: float):
    """(D_p, C_{D-1}, C_D): D_p and the sorted cumulative mass before/at it."""
    a = np.asarray(a, np.float64)
    if a.size == 0:
        return 0, 0.0, 0.0
    srt = np.sort(a)[::-1]
    cum = np.cumsum(srt)
    hit = np.nonzero(cum >= p)[0]
    k = int(hit[0]) + 1 if hit.size else int(a.size)
    before = float(cum[k - 2]) if k >= 2 else 0.0
    return k, before, float(cum[k - 1])


# ---------------------------------------------------------------------------
# Sec. 5.3, Table 2: attention entropy in place of the Top-p working set
# ---------------------------------------------------------------------------

def entropy_support(a) -> float:
    """exp(H(a)) with H(a) = -sum_i a_i ln a_i over the a_i > 0.

    The dual-timescale ablation of Sec. 5.3 (Table 2) swaps the Top-p
    working-set metric for attention entropy and gives no formula.  The
    reading taken here is the entropy's effective support size: the number
    of equally weighted tokens with the same entropy (1 for a point mass, N
    for the uniform distribution over N).  It stands where K^x = D_p stands
    in Eq. 8, so Delta = mean over (layer, KV head) of
    (exp H(a^S) - exp H(a^L)) / |C_t| (demand_trend with these values).
    """
    a = np.asarray(a, np.float64)
    nz = a[a > 0]
    if nz.size == 0:
        return 0.0
    return float(np.exp(-np.sum(nz * np.log(nz))))


# ---------------------------------------------------------------------------
# One (request, layer, KV head) unit at a capacity boundary
# ---------------------------------------------------------------------------

@dataclass
class UnitResult:
    a_dem: np.ndarray      # [2][|Cdem|]  short / long distributions over Cdem
    a_cmp: np.ndarray      # [2][|Ccmp|]  short / long distributions over Ccmp
    k: np.ndarray          # [2] int: K^S, K^L (Eq. 7)
    s: np.ndarray          # [|Ccmp|] importance (Eq. 9)


def unit_boundary(qt_unit, keys, num_pages: int, page_size: int,
                  recent: int, p: float) -> UnitResult:
    """Demand and importance for one (layer, KV head) of one request.

    qt_unit: [2][G][d] calibrated, rotated summaries of the G query heads of
    this KV head (x = 0 short, 1 long).  keys: [num_pages * page_size][d], the
    request's keys in logical slot order.

    Sec. 3.2 / App. E.1: the demand candidates exclude the most recent
    physical block, Cdem = [0, (P-1) b); each summary induces a normalised
    distribution over Cdem; K^x = D_p of it (Eq. 7).  Sec. 3.3, Eq. 9: the
    importance of a compression candidate is max(a^S, a^L); the compression
    candidates exclude the protected recent window, Ccmp = [0, P b - R), and
    their distributions are a fresh softmax over Ccmp.
    """
    n_dem = (num_pages - 1) * page_size
    n_cmp = num_pages * page_size - recent
    keys = np.asarray(keys, np.float64)
    a_dem = np.zeros((2, max(n_dem, 0)))
    a_cmp = np.zeros((2, max(n_cmp, 0)))
    ks = np.zeros(2, dtype=np.int64)
    for x in range(2):
        z = logits(qt_unit[x], keys[:max(n_cmp, 0)])     # [G][n_cmp]
        if n_dem > 0:
            a_dem[x] = kv_head_distribution(z[:, :n_dem])
            ks[x] = coverage_demand(a_dem[x], p)
        if n_cmp > 0:
            a_cmp[x] = kv_head_distribution(z)
    s = importance(a_cmp[0], a_cmp[1]) if n_cmp > 0 else np.zeros(0)
    return UnitResult(a_dem=a_dem, a_cmp=a_cmp, k=ks, s=s)


def gather_logical(cache, block_table, layer: int, kv_head: int):
    """Keys (or values) of one unit in logical slot order.

    cache: [L][num_pages][Hkv][b][d]; block_table: physical page of each
    logical block.
    """
    return np.concatenate([np.asarray(cache[layer, pg, kv_head])
                           for pg in block_table], axis=0)


def request_boundary(qbar_s, qbar_l, q_cur, k_cache, block_table, pos: int,
                     cfg) -> dict:
    """Full boundary estimation for one request: all (layer, KV head) units.

    qbar_*, q_cur: [L][Hq][d]; k_cache: [L][pages][Hkv][b][d] (float64 view).
    Returns K[L][Hkv][2], the units' UnitResults and Delta (Eq. 8).
    """
    L, hq, d = np.asarray(q_cur).shape
    hkv = cfg["num_kv_heads"]
    g = hq // hkv
    qt = summary_queries(qbar_s, qbar_l, q_cur, pos, cfg["rope_theta"])
    P = len(block_table)
    units = {}
    kk = np.zeros((L, hkv, 2), dtype=np.int64)
    for layer in range(L):
        for h in range(hkv):
            keys = gather_logical(k_cache, block_table, layer, h)
            qt_unit = qt[layer][:, h * g:(h + 1) * g, :]   # [2][G][d]
            u = unit_boundary(qt_unit, keys, P, cfg["page_size"],
                              cfg["recent_window"], cfg["p"])
            units[(layer, h)] = u
            kk[layer, h] = u.k
    n_cand = (P - 1) * cfg["page_size"]
    return {"K": kk, "units": units, "qt": qt,
            "delta": demand_trend(kk[..., 0], kk[..., 1], n_cand)}


# ---------------------------------------------------------------------------
# Sec. 3.2 Eqs. 7-8 and Sec. 4.2: trend and decision
# ---------------------------------------------------------------------------

def demand_trend(k_short, k_long, n_cand: int) -> float:
    """Delta = r^S - r^L with r^x = mean over (layer, KV head) of K^x / |C_t|.

    GrowPage, Sec. 3.2, Eqs. 7-8 (all layers participate).  |C_t| is the
    same for every (layer, KV head) of a request, so Delta equals
    (sum K^S - sum K^L) / (|C_t| * units).  It is evaluated in that form: the
    sums of integer demands are exact in float64, so the sign of Delta -- and
    with it the decision, where Delta = 0 compresses -- is exact, which two
    separately rounded means would not guarantee.
    """
    if n_cand <= 0:
        return 0.0
    ks = np.asarray(k_short, np.float64)
    kl = np.asarray(k_long, np.float64)
    return float((np.sum(ks) - np.sum(kl)) / (float(n_cand) * ks.size))


@dataclass
class Action:
    kind: int
    fallback: bool = False
    forced: bool = False


def decide(delta: float, num_pages: int, free_pages: int, reserve: int,
           tau: float, policy: str = "growpage", draw: float = 0.0,
           random_compress: float = 0.7, shrink_threshold: float = -0.005,
           shrink_floor_pages: int = 4) -> Action:
    """The capacity decision for one request at a boundary.

    GrowPage (Sec. 3.2, after Eq. 8): Grow iff Delta > tau, else Compress &
    Hold.  P = 1 forces Grow (there is no history to compress).  A Grow the
    free pool cannot grant above ``reserve`` pages falls back to Compress
    (Sec. 4.2; App. H.2 defines a fallback).  The alternatives of App. H.1:
    "fixed" never grows; "random" compresses with probability
    ``random_compress`` (the uniform ``draw`` decides), whatever Delta;
    "inverse" grows iff Delta <= tau; "shrink" follows Eq. 13: Shrink if
    Delta < -0.005, Compress & Hold if -0.005 <= Delta <= 0, Grow if
    Delta > 0, with no Shrink at or below the 1024-token floor.
    """
    if num_pages <= 1:
        return Action(GROW, forced=True)
    shrink = False
    if policy == "growpage":
        want_grow = delta > tau
    elif policy == "fixed":
        want_grow = False
    elif policy == "random":
        want_grow = not (draw < random_compress)
    elif policy == "inverse":
        want_grow = not (delta > tau)
    elif policy == "shrink":
        want_grow = delta > tau
        shrink = (not want_grow) and delta < shrink_threshold and num_pages > shrink_floor_pages
    else:
        raise ValueError(policy)
    if want_grow:
        if free_pages > reserve:
            return Action(GROW)
        return Action(COMPRESS, fallback=True)
    if shrink:
        return Action(SHRINK)
    return Action(COMPRESS)


# SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
# generators", OOPSLA 2014): one output of the generator whose state is x,
# i.e. x advanced by the golden-ratio increment and then mixed.
_M64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def policy_draw(seed: int, k: int) -> float:
    """Uniform [0, 1) draw of the k-th decision for the random policy:
    the top 53 bits of splitmix64(seed * 2^32 + k), scaled by 2^-53."""
    return (splitmix64(((seed << 32) + k) & _M64) >> 11) / float(1 << 53)


# ---------------------------------------------------------------------------
# Sec. 3.3 Eqs. 9-10: importance and retention
# ---------------------------------------------------------------------------

def importance(a_s, a_l):
    """s_i = max(a^S_i, a^L_i) (Eq. 9)."""
    return np.maximum(np.asarray(a_s, np.float64), np.asarray(a_l, np.float64))


def _top_by_score(cands: np.ndarray, s: np.ndarray, k: int) -> np.ndarray:
    """The k candidates with the largest score; equal scores: lower slot first."""
    if k <= 0 or cands.size == 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((cands, -s[cands]))
    return cands[order[:k]]


def retention_budget(num_pages: int, page_size: int, recent: int, drop: int = 1) -> int:
    """K_t: historical tokens kept so that (P - drop) b slots stay occupied
    (drop = 1 for Compress & Hold, 2 for Shrink, App. H.1)."""
    return (num_pages - drop) * page_size - recent


def select_retained(s, num_pages: int, page_size: int, recent: int,
                    k_loc: int, drop: int = 1) -> np.ndarray:
    """Keep mask over the P*b slots of one (layer, KV head) (Eq. 10).

    S_loc = union over blocks j of TopK_{k_loc'}(B_j; s);
    S = S_loc  union  TopK_{K_t - |S_loc|}(Ccmp minus S_loc; s);
    the protected recent window [P b - R, P b) is always kept (Sec. 3.3,
    Sec. 5.1).  Exactly (P - drop) b slots are kept: one page freed by
    Compress & Hold, two pages' worth by Shrink (App. H.1).
    """
    s = np.asarray(s, np.float64)
    n = num_pages * page_size
    n_cmp = n - recent
    k_t = retention_budget(num_pages, page_size, recent, drop)
    keep = np.zeros(n, dtype=bool)
    keep[n_cmp:] = True
    quota = min(k_loc, k_t // num_pages) if num_pages > 0 else 0
    for j in range(num_pages):
        lo, hi = j * page_size, min((j + 1) * page_size, n_cmp)
        if hi <= lo:
            continue
        kj = min(quota, hi - lo)
        keep[_top_by_score(np.arange(lo, hi), s, kj)] = True
    n_loc = int(np.count_nonzero(keep[:n_cmp]))
    rest = np.nonzero(~keep[:n_cmp])[0]
    keep[_top_by_score(rest, s, k_t - n_loc)] = True
    return keep


# ---------------------------------------------------------------------------
# Sec. 4.2 and App. E.2: page pool, Grow, copy-on-write, compaction
# ---------------------------------------------------------------------------

@dataclass
class PagePool:
    """Free-page pool with per-page reference counts (App. E.2).

    Pages are handed out lowest id first (a deterministic choice; the paper
    only needs "a page from the global free-page pool", Sec. 4.2).
    """
    num_pages: int
    refcount: list = field(default_factory=list)

    def __post_init__(self):
        if not self.refcount:
            self.refcount = [0] * self.num_pages

    def free_count(self) -> int:
        return sum(1 for r in self.refcount if r == 0)

    def alloc(self) -> int:
        for i, r in enumerate(self.refcount):
            if r == 0:
                self.refcount[i] = 1
                return i
        raise MemoryError("no free pages")

    def ref(self, page: int):
        if self.refcount[page] <= 0:
            raise ValueError("ref of a free page")
        self.refcount[page] += 1

    def unref(self, page: int):
        if self.refcount[page] <= 0:
            raise ValueError("refcount underflow")
        self.refcount[page] -= 1


def grow(block_table: list, pool: PagePool) -> list:
    """Grow by One Page: append a fresh page to the block table (Sec. 3.3)."""
    return list(block_table) + [pool.alloc()]


def cow_plan(block_table, pool: PagePool):
    """Target block table for a compression (App. E.2).

    A page referenced by more than one request is never written in place: it
    is replaced by a fresh page; private pages are reused.  Fresh pages are
    taken lowest id first, in ascending logical order.  Raises MemoryError
    (and changes nothing) if the pool cannot supply every replacement.
    Returns (new_table, replaced_pages).
    """
    shared = [pg for pg in block_table if pool.refcount[pg] > 1]
    if len(shared) > pool.free_count():
        raise MemoryError("not enough free pages for copy-on-write")
    new_table, replaced = [], []
    for pg in block_table:
        if pool.refcount[pg] > 1:
            new_table.append(pool.alloc())
            replaced.append(pg)
        else:
            new_table.append(pg)
    return new_table, replaced


def release_replaced(replaced, pool: PagePool):
    """After compaction the request drops its references to replaced pages."""
    for pg in replaced:
        pool.unref(pg)


def shrink_release(new_table, pool: PagePool) -> list:
    """Shrink (App. H.1): after two pages' worth of history has been
    compacted into logical slots [0, (P-2) b), the emptied last page of the
    block table goes back to the pool; the request keeps P - 1 pages, the
    last of them with b free slots."""
    pool.unref(new_table[-1])
    return list(new_table[:-1])


def hole_fill_unit(rows, keep, num_pages: int, page_size: int):
    """Hole-fill variant of the compaction (order-destroying; not the
    paper's): kept rows of the first P-1 pages stay in their slots, and the
    k-th kept row of the last page (ascending) fills the k-th dropped slot of
    the first P-1 pages (ascending).  Returns rows [(P-1) b][d]."""
    rows = np.asarray(rows)
    keep = np.asarray(keep, dtype=bool)
    lastp = (num_pages - 1) * page_size
    out = rows[:lastp].copy()
    holes = np.nonzero(~keep[:lastp])[0]
    fillers = np.nonzero(keep[lastp:num_pages * page_size])[0] + lastp
    assert holes.size == fillers.size
    out[holes] = rows[fillers]
    return out


def compact_unit(rows, keep):
    """Retained rows (keys or values) of one unit in ascending slot order.

    The k-th kept slot becomes logical slot k of the compacted request
    (App. E.2: retained states are compacted into at most (P-1) b slots).
    rows: [P*b][d]; returns [(P-1) b][d].
    """
    return np.asarray(rows)[np.nonzero(keep)[0]]


def compress_cache(k_cache, v_cache, old_table, new_table, keep_masks,
                   page_size: int):
    """Apply Compress & Hold to copies of the paged caches of one request.

    keep_masks: [L][Hkv][P*b] bool.  Returns new (k_cache, v_cache): logical
    slots [0, (P-1) b) of the new block table hold the retained rows in
    order; the last logical page is left as it was (free slots); pages not
    in the new table are untouched.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    L, _, hkv = k_out.shape[:3]
    for layer in range(L):
        for h in range(hkv):
            for src, dst in ((k_cache, k_out), (v_cache, v_out)):
                rows = gather_logical(src, old_table, layer, h)
                kept = compact_unit(rows, keep_masks[layer][h])
                for i, row in enumerate(kept):
                    pg = new_table[i // page_size]
                    dst[layer, pg, h, i % page_size] = row
    return k_out, v_out


# ---------------------------------------------------------------------------
# Sec. 3.1 Eqs. 3-5 and Theorem 3.1 (checked by brute force in the tests)
# ---------------------------------------------------------------------------

def attention_output(a, values):
    """o = sum_i a_i v_i (Eq. 3)."""
    return np.asarray(a, np.float64) @ np.asarray(values, np.float64)


def renormalised_output(a, values, subset):
    """o^(S) = sum_{i in S} a_i / m(S) v_i, m(S) = sum_{i in S} a_i (Eq. 3)."""
    a = np.asarray(a, np.float64)
    idx = np.asarray(sorted(subset), dtype=np.int64)
    m = np.sum(a[idx])
    return (a[idx] / m) @ np.asarray(values, np.float64)[idx]


def worst_case_error(a, subset, vmax: float) -> float:
    """sup over ||v_i|| <= Vmax of ||o - o^(S)|| = 2 Vmax (1 - m(S)) (Eq. 5)."""
    a = np.asarray(a, np.float64)
    m = float(np.sum(a[list(subset)]))
    return 2.0 * vmax * (1.0 - m)


def worst_case_capacity(a, delta: float, vmax: float) -> int:
    """C^wc_delta by enumeration of every non-empty subset (Eq. 4 with Eq. 5)."""
    a = np.asarray(a, np.float64)
    n = a.size
    for size in range(1, n + 1):
        for sub in itertools.combinations(range(n), size):
            if worst_case_error(a, sub, vmax) <= delta:
                return size
    return n
