"""Seeded synthetic paged-KV workloads (inputs only, no method arithmetic).

Recipe (the same for every configuration; sizes per configuration below):

* K and V caches have the layout [L][num_pages][Hkv][page_size][d]; entries
  are N(0, 1) drawn with a seeded torch generator and rounded to the cache
  dtype (bf16 round-to-nearest-even, or fp32).
* Attention concentration is produced by *planted* keys: a per-(request,
  layer, KV head) direction u with unit RMS, supported on the lowest-
  frequency eighth of the rotary pairs (dims i and i + d/2 with i >= 7d/16),
  so that rotating a query at any position used here barely moves its
  alignment with u.  A planted key is ``scale * u``.
* Queries: "concentrated" steps draw q = 3 u + N(0, 1) for every query head
  of the KV group; "diffuse" steps draw q = N(0, 1).
* Qwen3-like shapes rescale every query and key vector to unit RMS (a
  stand-in for the model's QK-norm).
* Physical pages are a seeded permutation of the pool; block tables take
  consecutive runs of it.

* Continuous-batching stream (``stream256``): 256 seats in 32 prefix groups
  of 8.  A group's members share a 32-page prefix (one reference per
  member) and a direction u (their queries follow one topic); each request
  adds a private part of lognormal length (median 2048 tokens, sigma 1.0,
  clipped to 512..16384, rounded up to whole pages) and finishes after a
  geometric number of boundary events (mean 12).  A seat's queries
  alternate 64-step concentrated and diffuse phases from a seeded offset.
  The free pool holds a bounded number of spare pages beyond the initial
  allocation (256).  The request lifecycle that uses these draws lives in
  synth/stream.py.

Seeds: ``0x47505047 ^ config_id``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 0x47505047


@dataclass(frozen=True)
class ModelShape:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str          # "bf16" or "f32"
    q_dtype: str           # "bf16" or "f32"
    rope_theta: float
    qk_norm: bool = False

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


LLAMA8B = ModelShape(32, 32, 8, 128, "bf16", "bf16", 5.0e5)
QWEN3_8B = ModelShape(36, 32, 8, 128, "bf16", "bf16", 1.0e6, qk_norm=True)
TINY = ModelShape(2, 4, 2, 64, "f32", "f32", 1.0e4)

CONFIGS = {
    # id, shape, description
    "tiny": (1, TINY, "1 request, 2L, 4q/2kv, d64, fp32 K/V, 4 pages x 256, "
                      "64-step query history, 8 planted keys (scale 4)"),
    "llama8b_single": (2, LLAMA8B, "1 request, 32L, 32q/8kv, d128, bf16, "
                                   "32 pages x 256 = 8192 tokens, 512-step "
                                   "concentrated/diffuse query phases"),
    "batch64": (3, LLAMA8B, "64 requests, 4..128 pages each, shuffled shared "
                            "pool, all at a boundary"),
    "qwen3_8b": (4, QWEN3_8B, "16 requests x 128 pages, 36L, QK-normed, 30% "
                              "concentrated units"),
    "stream256": (5, LLAMA8B, "256-request continuous-batching stream with "
                              "32-page shared prefixes"),
    "custom": (6, TINY, "any shape and request sizes (edge cases)"),
}

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def config_seed(name: str) -> int:
    return SEED_BASE ^ CONFIGS[name][0]


@dataclass
class Workload:
    """A paged cache at (or near) a capacity boundary plus its query source."""
    name: str
    shape: ModelShape
    page_size: int
    num_pages: int                     # physical pages in the pool
    k_cache: torch.Tensor              # [L][num_pages][Hkv][b][d]
    v_cache: torch.Tensor
    block_tables: list                 # per request: list of physical pages
    positions: list                    # per request: current decode position
    directions: torch.Tensor           # [n][L][Hkv][d] fp32, unit RMS
    concentrated: torch.Tensor         # [n][L][Hkv] bool (unit kind)
    gen: torch.Generator               # device-side draws
    hgen: torch.Generator              # host-side draws (sizes, permutations)
    plant_frac: float = 0.02
    plant_scale: float = 6.0
    history: list = field(default_factory=list)   # list of q tensors [L][n][Hq][d]
    phase_len: int = 512
    extra: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return len(self.block_tables)

    @property
    def device(self):
        return self.k_cache.device

    def free_pages(self) -> list:
        used = set()
        for bt in self.block_tables:
            used.update(bt)
        return [p for p in range(self.num_pages) if p not in used]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _gens(device, seed: int):
    return _gen(device, seed), _gen("cpu", seed ^ 0x5A5A5A5A)


def low_freq_directions(count_shape, d: int, gen, device) -> torch.Tensor:
    """Random unit-RMS vectors supported on the lowest-frequency rotary pairs."""
    u = torch.zeros(*count_shape, d, dtype=torch.float32, device=device)
    half = d // 2
    lo = (7 * d) // 16
    idx = torch.cat([torch.arange(lo, half), torch.arange(lo + half, d)]).to(device)
    vals = torch.randn(*count_shape, idx.numel(), generator=gen, device=device)
    u[..., idx] = vals
    norm = torch.linalg.vector_norm(u, dim=-1, keepdim=True)
    return u / norm * math.sqrt(d)


def _unit_rms(x: torch.Tensor) -> torch.Tensor:
    d = x.shape[-1]
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True) * math.sqrt(d)


def _random_cache(shape: ModelShape, num_pages: int, page_size: int, gen,
                  device, extra_pages: int = 0) -> torch.Tensor:
    """[L][num_pages + extra_pages][Hkv][b][d]: the first num_pages pages
    drawn N(0, 1) (the same draws whatever extra_pages is), the extra pages
    zero (a free reserve that the caller fills before reading)."""
    dt = TORCH_DTYPE[shape.kv_dtype]
    out = torch.empty(shape.num_layers, num_pages + extra_pages, shape.num_kv_heads,
                      page_size, shape.head_dim, dtype=dt, device=device)
    if extra_pages:
        out[:, num_pages:].zero_()
    for layer in range(shape.num_layers):
        # chunk over pages to bound temporaries
        step = max(1, (1 << 28) // (shape.num_kv_heads * page_size * shape.head_dim))
        for p0 in range(0, num_pages, step):
            p1 = min(num_pages, p0 + step)
            blk = torch.randn(p1 - p0, shape.num_kv_heads, page_size,
                              shape.head_dim, generator=gen, device=device,
                              dtype=torch.float32)
            if shape.qk_norm:
                blk = _unit_rms(blk)
            out[layer, p0:p1] = blk.to(dt)
    return out


def _plant(w: Workload, req: int, pages, slot_mask=None):
    """Overwrite ~plant_frac of the keys of ``pages`` of request ``req`` with
    scale * u for its concentrated units.  slot_mask optionally restricts the
    candidate slots ([len(pages)][b] bool)."""
    sh = w.shape
    dev = w.device
    pages_t = torch.as_tensor(list(pages), device=dev, dtype=torch.long)
    npg = pages_t.numel()
    if npg == 0:
        return
    for layer in range(sh.num_layers):
        m = torch.rand(npg, sh.num_kv_heads, w.page_size, generator=w.gen,
                       device=dev) < w.plant_frac
        if slot_mask is not None:
            m &= slot_mask[:, None, :]
        m &= w.concentrated[req, layer][None, :, None]
        u = w.directions[req, layer]                       # [Hkv][d]
        planted = w.plant_scale * u
        if sh.qk_norm:
            planted = _unit_rms(planted)
        blk = w.k_cache[layer, pages_t].float()            # [npg][Hkv][b][d]
        blk = torch.where(m[..., None], planted[None, :, None, :], blk)
        w.k_cache[layer, pages_t] = blk.to(w.k_cache.dtype)


def query_step(w: Workload, kinds) -> torch.Tensor:
    """One decode step's queries [L][n][Hq][d].

    kinds: [n] bool or [n][L][Hkv] bool -- True draws a concentrated query
    (3 u + N(0,1)) for that unit's query heads, False a diffuse N(0,1) one.
    """
    sh = w.shape
    dev = w.device
    kinds = torch.as_tensor(kinds, device=dev)
    if kinds.dim() == 1:
        kinds = kinds[:, None, None].expand(w.n, sh.num_layers, sh.num_kv_heads)
    kinds = kinds & w.concentrated
    noise = torch.randn(sh.num_layers, w.n, sh.num_q_heads, sh.head_dim,
                        generator=w.gen, device=dev)
    u = w.directions.permute(1, 0, 2, 3)                   # [L][n][Hkv][d]
    u = u.repeat_interleave(sh.group, dim=2)                # [L][n][Hq][d]
    k = kinds.permute(1, 0, 2).repeat_interleave(sh.group, dim=2)  # [L][n][Hq]
    q = torch.where(k[..., None], 3.0 * u + noise, noise)
    if sh.qk_norm:
        q = _unit_rms(q)
    return q.to(TORCH_DTYPE[sh.q_dtype])


def fill_page(w: Workload, req: int, phys_page: int):
    """Write a fresh page of tokens (N(0,1), planted like the rest)."""
    fill_pages(w, req, [phys_page])


def fill_pages(w: Workload, req: int, phys_pages):
    """Write fresh tokens into several pages of request ``req`` at once."""
    sh = w.shape
    dev = w.device
    pages = list(phys_pages)
    if not pages:
        return
    idx = torch.as_tensor(pages, device=dev, dtype=torch.long)
    for cache in (w.k_cache, w.v_cache):
        blk = torch.randn(sh.num_layers, len(pages), sh.num_kv_heads, w.page_size,
                          sh.head_dim, generator=w.gen, device=dev)
        if sh.qk_norm:
            blk = _unit_rms(blk)
        cache.index_copy_(1, idx, blk.to(cache.dtype))
    _plant(w, req, pages)


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------

def _tiny(device, variant: str = "grow", **_):
    sh = TINY
    b = 256
    gen, hgen = _gens(device, config_seed("tiny") ^ (0 if variant == "grow" else 1))
    num_pages = 8
    P = 4
    perm = torch.randperm(num_pages, generator=hgen).tolist()
    bt = perm[:P]
    k = _random_cache(sh, num_pages, b, gen, device)
    v = _random_cache(sh, num_pages, b, gen, device)
    u = low_freq_directions((1, sh.num_layers, sh.num_kv_heads), sh.head_dim,
                            gen, device)
    conc = torch.ones(1, sh.num_layers, sh.num_kv_heads, dtype=torch.bool,
                      device=device)
    w = Workload("tiny", sh, b, num_pages, k, v, [bt], [P * b], u, conc, gen,
                 hgen, plant_frac=0.0, plant_scale=4.0)
    # 8 planted keys per (layer, KV head) at seeded slots of Cdem
    n_dem = (P - 1) * b
    for layer in range(sh.num_layers):
        for h in range(sh.num_kv_heads):
            slots = torch.randperm(n_dem, generator=hgen)[:8]
            for s in slots.tolist():
                w.k_cache[layer, bt[s // b], h, s % b] = (
                    4.0 * u[0, layer, h]).to(w.k_cache.dtype)
    # 64-step history.  "grow": 16 concentrated steps then 48 diffuse ones
    # (the long summary stays aligned, the short one turns diffuse);
    # "compress": 48 diffuse steps then 16 concentrated ones.
    for t in range(64):
        kind = (t < 16) if variant == "grow" else (t >= 48)
        w.history.append(query_step(w, [kind]))
    return w


def _llama_single(device, num_pages: int = 64, P: int = 32, **_):
    sh = LLAMA8B
    b = 256
    gen, hgen = _gens(device, config_seed("llama8b_single"))
    perm = torch.randperm(num_pages, generator=hgen).tolist()
    bt = perm[:P]
    k = _random_cache(sh, num_pages, b, gen, device)
    v = _random_cache(sh, num_pages, b, gen, device)
    u = low_freq_directions((1, sh.num_layers, sh.num_kv_heads), sh.head_dim,
                            gen, device)
    conc = torch.ones(1, sh.num_layers, sh.num_kv_heads, dtype=torch.bool,
                      device=device)
    w = Workload("llama8b_single", sh, b, num_pages, k, v, [bt], [P * b], u,
                 conc, gen, hgen)
    _plant(w, 0, bt)
    return w


def _batch(device, name="batch64", shape=LLAMA8B, n=64, p_lo=4, p_hi=128,
           spare_per_req=2, conc_prob=None, sizes=None, seed_xor=0, extra_pages=0, **_):
    sh = shape
    b = 256
    gen, hgen = _gens(device, config_seed(name) ^ seed_xor)
    if sizes is None:
        sizes = torch.randint(p_lo, p_hi + 1, (n,), generator=hgen).tolist()
    else:
        sizes = list(sizes)
        n = len(sizes)
    num_pages = sum(sizes) + spare_per_req * n
    perm = torch.randperm(num_pages, generator=hgen).tolist()
    bts, off = [], 0
    for s in sizes:
        bts.append(perm[off:off + s])
        off += s
    k = _random_cache(sh, num_pages, b, gen, device, extra_pages)
    v = _random_cache(sh, num_pages, b, gen, device, extra_pages)
    num_pages += extra_pages
    u = low_freq_directions((n, sh.num_layers, sh.num_kv_heads), sh.head_dim,
                            gen, device)
    if conc_prob is None:
        conc = torch.ones(n, sh.num_layers, sh.num_kv_heads, dtype=torch.bool,
                          device=device)
    else:
        conc = torch.rand(n, sh.num_layers, sh.num_kv_heads, generator=gen,
                          device=device) < conc_prob
    w = Workload(name, sh, b, num_pages, k, v, bts, [s * b for s in sizes], u,
                 conc, gen, hgen)
    for r in range(n):
        _plant(w, r, bts[r])
    # 64-step history per request: half concentrated, half diffuse, order seeded
    conc_first = (torch.rand(n, generator=hgen) < 0.5).tolist()
    if conc_prob is not None:
        conc_first = [True] * n
    for t in range(64):
        kinds = [cf if t < 32 else (not cf) for cf in conc_first]
        if conc_prob is not None:
            kinds = [True] * n
        w.history.append(query_step(w, kinds))
    w.extra["conc_first"] = conc_first
    return w


def batch_kinds(w: Workload, step: int, phase_len: int = 512) -> list:
    """Per request: True if its query at decode step ``step`` is a
    concentrated one.  Steps 0..63 are the 64-step history (the request's
    seeded first kind, then the other one); after it the request keeps the
    history's second kind until step 64 + phase_len - 128, then alternates in
    phases of phase_len steps, as the single-request decode stream does.  The
    flips fall halfway between boundaries (every 256 steps from step 64), so
    at every boundary the requests in a diffuse phase have spent at least
    128 steps in it."""
    ph = (step - 64 + 128) // phase_len if step >= 64 else -1
    out = []
    for cf in w.extra["conc_first"]:
        if step < 64:
            out.append(cf if step < 32 else (not cf))
        else:
            out.append((not cf) if ph % 2 == 0 else cf)
    return out


STREAM_DEFAULTS = dict(seats=256, group=8, prefix_pages=32, spare_pages=256, median_tokens=2048,
                       sigma=1.0, min_tokens=512, max_tokens=16384, mean_events=12, phase_len=64,
                       max_pages=128)


def private_pages(hgen, n: int, median_tokens=2048, sigma=1.0, min_tokens=512, max_tokens=16384,
                  page_size=256) -> list:
    """Private-part lengths in pages: lognormal tokens, clipped, rounded up."""
    z = torch.randn(n, generator=hgen, dtype=torch.float64)
    tok = torch.exp(math.log(median_tokens) + sigma * z).clamp(min_tokens, max_tokens)
    return torch.ceil(tok / page_size).to(torch.int64).tolist()


def event_counts(hgen, n: int, mean: float = 12.0) -> list:
    """Boundary events before a request finishes: geometric on {1, 2, ...}."""
    u = torch.rand(n, generator=hgen, dtype=torch.float64).clamp_min(1e-300)
    q = 1.0 - 1.0 / mean
    return (torch.floor(torch.log(u) / math.log(q)) + 1).to(torch.int64).tolist()


def _stream(device, shape=LLAMA8B, **kw):
    """Initial state of the continuous-batching stream (config 5).

    Pages [0, G * prefix) are the groups' prefixes, then each seat's private
    pages in seat order, then the spare pages.  ``extra`` holds the recipe
    parameters, the groups' prefix pages and the seeded per-seat draws the
    lifecycle consumes (phase offsets, event counts).
    """
    p = dict(STREAM_DEFAULTS)
    p.update({k: v for k, v in kw.items() if k in STREAM_DEFAULTS})
    sh = shape
    b = 256
    gen, hgen = _gens(device, config_seed("stream256") ^ kw.get("seed_xor", 0))
    seats, group, npre = p["seats"], p["group"], p["prefix_pages"]
    ngroups = (seats + group - 1) // group
    priv = private_pages(hgen, seats, p["median_tokens"], p["sigma"], p["min_tokens"], p["max_tokens"], b)
    priv = [min(x, p["max_pages"] - npre - 1) for x in priv]
    prefixes = [list(range(g * npre, (g + 1) * npre)) for g in range(ngroups)]
    nxt = ngroups * npre
    bts = []
    for s_ in range(seats):
        bts.append(prefixes[s_ // group] + list(range(nxt, nxt + priv[s_])))
        nxt += priv[s_]
    num_pages = nxt + p["spare_pages"]
    k = _random_cache(sh, num_pages, b, gen, device)
    v = _random_cache(sh, num_pages, b, gen, device)
    ug = low_freq_directions((ngroups, sh.num_layers, sh.num_kv_heads), sh.head_dim, gen, device)
    u = ug.repeat_interleave(group, dim=0)[:seats].contiguous()
    conc = torch.ones(seats, sh.num_layers, sh.num_kv_heads, dtype=torch.bool, device=device)
    w = Workload("stream256", sh, b, num_pages, k, v, bts, [len(t) * b for t in bts], u, conc, gen, hgen,
                 phase_len=p["phase_len"])
    for g in range(ngroups):
        _plant(w, g * group, prefixes[g])
    for s_ in range(seats):
        _plant(w, s_, bts[s_][npre:])
    w.extra.update(p)
    w.extra["prefixes"] = prefixes
    w.extra["phase_offset"] = torch.randint(0, 2 * p["phase_len"], (seats,), generator=hgen).tolist()
    w.extra["events"] = event_counts(hgen, seats, p["mean_events"])
    return w


def stream_kinds(w: Workload, step: int) -> list:
    """Per seat: True if its query at this step is a concentrated one."""
    L = w.extra["phase_len"]
    return [((step + off) // L) % 2 == 0 for off in w.extra["phase_offset"]]


def make_workload(name: str, device="cpu", **kw) -> Workload:
    """Build configuration ``name`` on ``device`` (see CONFIGS)."""
    if name == "tiny":
        return _tiny(device, **kw)
    if name == "llama8b_single":
        return _llama_single(device, **kw)
    if name == "batch64":
        return _batch(device, **kw)
    if name == "qwen3_8b":
        kw.setdefault("n", 16)
        kw.setdefault("p_lo", 128)
        kw.setdefault("p_hi", 128)
        kw.setdefault("spare_per_req", 1)
        return _batch(device, name="qwen3_8b", shape=QWEN3_8B, conc_prob=0.3,
                      **kw)
    if name == "stream256":
        return _stream(device, **kw)
    if name == "custom":
        # explicit shape and request sizes: kw shape=ModelShape, sizes=[P, ...]
        return _batch(device, name="custom", **kw)
    raise KeyError(name)
