"""Continuous-batching stream over the engine: the request lifecycle of the
256-seat workload (``make_workload("stream256")``).

This is a synthetic serving loop, not part of the engine and free of the
method's arithmetic: it admits, steps, finishes and preempts requests and
writes synthetic tokens into pages; every GrowPage step runs in the engine
through its C ABI (``paged_kv_cache_step_gb300``).

One step t:

1. queries for every seat (concentrated or diffuse by the seat's phase);
2. ``gp_update_summaries`` over the live requests (``first`` on a request's
   first step: the summaries are initialised, App. E.1);
3. the boundary requests are the live ones with ``(seat + t) %
   boundary_every == 0`` admitted at least ``boundary_every`` steps ago (a
   page of decoding); the loop writes fresh synthetic tokens into each
   one's last logical page, which is full again.  A request whose block
   table is full finishes there (it has reached its maximum length);
4. ``gp_boundary_demand`` over them, ``gp_decide``, ``gp_grow_page`` for each
   Grow (in request order) and one ``gp_compress_hold`` call for the
   Compress & Hold requests.  If the pool cannot supply the copy-on-write
   pages of the whole call (``GP_ERR_NO_PAGES``, nothing changed), the
   requests are compressed one call each, in order, and a request whose call
   still fails is preempted (its slot and pages are released);
5. requests whose boundary-event count has run out finish (slot released,
   every page unreferenced);
6. each empty seat admits a new request of its group when the pool can hold
   it and keep ``admit_headroom`` pages free: the group's prefix is shared
   (one reference per page) while it is unmodified, else a fresh prefix is
   written; the private part has the recipe's lognormal length.

A group's prefix stays shareable while at least one member holds it
unmodified: a member that compresses while it is the prefix's only holder
compacts those pages in place, after which the group needs a new prefix.

Decode positions: a request admitted with N tokens is at position N, and
each step stands for ``tokens_per_step`` decode tokens (a page per
``boundary_every`` steps), so RoPE positions advance like real decoding.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

from .workloads import event_counts, fill_page, fill_pages, private_pages, query_step, stream_kinds


@dataclass
class Seat:
    req: object = None          # engine Request (binding) or None
    group: int = 0
    events_left: int = 0
    admitted_at: int = -1       # step of admission
    first_pending: bool = True  # next summary update initialises
    holds_prefix: bool = False  # its table starts with the group's current prefix
    tokens: int = 0


@dataclass
class StepLog:
    step: int
    live_before: dict = field(default_factory=dict)   # seat -> table at the start of the action phase
    boundary: list = field(default_factory=list)       # seats at a boundary, in call order
    actions: list = field(default_factory=list)        # (kind, seat, table_before, table_after)
    admitted: list = field(default_factory=list)       # (seat, table)
    counts: dict = field(default_factory=dict)


class ContinuousBatch:
    """The stream, driven through an engine context ``ctx`` created over the
    workload's caches with at least ``seats`` summary slots."""

    def __init__(self, gp, ctx, w, max_pages_per_req: int, boundary_every: int = 8,
                 admit_headroom: int = 32):
        self.gp, self.ctx, self.w = gp, ctx, w
        self.maxp = max_pages_per_req
        self.every = boundary_every
        self.tokens_per_step = w.page_size // boundary_every
        self.headroom = admit_headroom
        self.x = w.extra
        self.group_size = self.x["group"]
        self.npre = self.x["prefix_pages"]
        ngroups = len(self.x["prefixes"])
        self.prefix = [list(p) for p in self.x["prefixes"]]
        self.prefix_alive = [True] * ngroups
        self.seats = []
        dev = w.device
        self.device = dev
        for s, table in enumerate(w.block_tables):
            seat = Seat(group=s // self.group_size, events_left=self.x["events"][s], admitted_at=-1,
                        holds_prefix=True, tokens=len(table) * w.page_size)
            self.seats.append(seat)
        # the engine's pool mirrors the initial ownership: one reference per table entry
        refs = {}
        for table in w.block_tables:
            for pg in table:
                refs[pg] = refs.get(pg, 0) + 1
        for _ in range(w.num_pages):
            gp.gp_page_alloc(ctx)
        for pg in range(w.num_pages):
            r = refs.get(pg, 0)
            if r == 0:
                gp.gp_page_unref(ctx, pg)
            for _ in range(r - 1):
                gp.gp_page_ref(ctx, pg)
        for s, table in enumerate(w.block_tables):
            slot = gp.gp_slot_acquire(ctx)
            self.seats[s].req = gp.Request(slot, table, self.seats[s].tokens, self.maxp)
        self.counts = dict(grow=0, compress=0, fallback=0, forced=0, cow_pages=0, preempt=0,
                           finish=0, full=0, admit=0, admit_wait=0, boundary=0, batched_retry=0)
        self.live_sum = 0

    # ------------------------------------------------------------------ helpers
    def live(self):
        return [s for s, st in enumerate(self.seats) if st.req is not None]

    def _release(self, s: int):
        gp, st = self.gp, self.seats[s]
        for pg in st.req.pages:
            gp.gp_page_unref(self.ctx, pg)
        gp.gp_slot_release(self.ctx, st.req.slot)
        st.req = None
        st.holds_prefix = False

    def _prefix_holders(self, g: int):
        return [s for s, st in enumerate(self.seats) if st.req is not None and st.group == g and st.holds_prefix]

    def _admit(self, s: int, t: int, log: StepLog):
        gp, w, st = self.gp, self.w, self.seats[s]
        g = st.group
        if self.prefix_alive[g] and not self._prefix_holders(g):
            self.prefix_alive[g] = False
        npriv = private_pages(w.hgen, 1, self.x["median_tokens"], self.x["sigma"], self.x["min_tokens"],
                              self.x["max_tokens"], w.page_size)[0]
        npriv = min(npriv, self.maxp - self.npre - 1)
        need = npriv + (0 if self.prefix_alive[g] else self.npre)
        if gp.gp_free_page_count(self.ctx) - need < self.headroom:
            self.counts["admit_wait"] += 1
            return
        fresh = []
        if not self.prefix_alive[g]:
            self.prefix[g] = [gp.gp_page_alloc(self.ctx) for _ in range(self.npre)]
            fresh += self.prefix[g]
            self.prefix_alive[g] = True
        else:
            for pg in self.prefix[g]:
                gp.gp_page_ref(self.ctx, pg)
        table = list(self.prefix[g])
        for _ in range(npriv):
            table.append(gp.gp_page_alloc(self.ctx))
        fresh += table[self.npre:]
        fill_pages(w, s, fresh)
        slot = gp.gp_slot_acquire(self.ctx)
        st.tokens = len(table) * w.page_size
        st.req = gp.Request(slot, table, st.tokens, self.maxp)
        st.events_left = event_counts(w.hgen, 1, self.x["mean_events"])[0]
        st.admitted_at = t
        st.first_pending = True
        st.holds_prefix = True
        self.counts["admit"] += 1
        log.admitted.append((s, list(table)))

    def at_boundary(self, s: int, t: int) -> bool:
        """A live request is at a boundary every ``boundary_every`` steps, the
        first one a full page of decoding after its admission."""
        st = self.seats[s]
        return st.req is not None and (s + t) % self.every == 0 and st.admitted_at + self.every <= t

    # --------------------------------------------------------------------- step
    def step(self, t: int, hooks=None) -> StepLog:
        gp, w = self.gp, self.w
        log = StepLog(step=t)
        live = self.live()
        self.live_sum += len(live)
        q_all = query_step(w, stream_kinds(w, t))              # [L][seats][Hq][d]
        if live:
            idx = torch.as_tensor(live, device=self.device)
            q_live = q_all.index_select(1, idx).contiguous()
            slots = torch.tensor([self.seats[s].req.slot for s in live], dtype=torch.int32, device=self.device)
            first = torch.tensor([int(self.seats[s].first_pending) for s in live], dtype=torch.uint8,
                                 device=self.device)
            if hooks is not None and hasattr(hooks, "pre_update"):
                hooks.pre_update(self, t, live, q_live)
            gp.gp_update_summaries(self.ctx, len(live), slots, q_live, first)
            for s in live:
                st = self.seats[s]
                st.first_pending = False
                st.tokens += self.tokens_per_step
                st.req.pos = st.tokens
        bseats = [s for s in live if self.at_boundary(s, t)]
        for s in list(bseats):
            if self.seats[s].req.num_pages >= self.maxp:
                # the block table is full: the request has reached its maximum length
                log.actions.append(("finish", s, list(self.seats[s].req.pages), []))
                self._release(s)
                self.counts["finish"] += 1
                self.counts["full"] += 1
                bseats.remove(s)
        log.boundary = list(bseats)
        log.live_before = {s: list(self.seats[s].req.pages) for s in live}
        if bseats:
            self.counts["boundary"] += len(bseats)
            for s in bseats:
                st = self.seats[s]
                fill_page(w, s, st.req.pages[-1])
            idx = torch.as_tensor(bseats, device=self.device)
            q_b = q_all.index_select(1, idx).contiguous()
            reqs = [self.seats[s].req for s in bseats]
            dem = gp.gp_boundary_demand(self.ctx, reqs, q_b)
            acts = gp.gp_decide(self.ctx, reqs, dem)
            if hooks is not None and hasattr(hooks, "post_demand"):
                hooks.post_demand(self, t, bseats, q_b, dem, acts)
            grows = [s for s, a in zip(bseats, acts) if a.kind == gp.GP_ACT_GROW]
            comps = [s for s, a in zip(bseats, acts) if a.kind != gp.GP_ACT_GROW]
            for a in acts:
                self.counts["fallback"] += int(a.fallback)
                self.counts["forced"] += int(a.forced)
            for s in grows:
                st = self.seats[s]
                before = list(st.req.pages)
                gp.gp_grow_page(self.ctx, st.req)
                log.actions.append(("grow", s, before, list(st.req.pages)))
                self.counts["grow"] += 1
            if comps:
                self._compress(t, comps, log, hooks)
            for s in bseats:
                st = self.seats[s]
                if st.req is None:
                    continue
                st.events_left -= 1
                if st.events_left <= 0:
                    log.actions.append(("finish", s, list(st.req.pages), []))
                    self._release(s)
                    self.counts["finish"] += 1
        for s, st in enumerate(self.seats):
            if st.req is None:
                self._admit(s, t, log)
        log.counts = dict(self.counts)
        if hooks is not None and hasattr(hooks, "post_step"):
            hooks.post_step(self, t, log)
        return log

    def _compress(self, t, comps, log, hooks):
        gp = self.gp
        before = {s: list(self.seats[s].req.pages) for s in comps}
        reqs = [self.seats[s].req for s in comps]
        done = []
        try:
            gp.gp_compress_hold(self.ctx, reqs)
            done = [comps]
        except gp.GrowPageError as e:
            if e.status != gp.GP_ERR_NO_PAGES:
                raise
            self.counts["batched_retry"] += 1
            for s in comps:
                try:
                    gp.gp_compress_hold(self.ctx, [self.seats[s].req])
                    done.append([s])
                    if hooks is not None and hasattr(hooks, "post_compress"):
                        hooks.post_compress(self, t, [s])
                except gp.GrowPageError as e2:
                    if e2.status != gp.GP_ERR_NO_PAGES:
                        raise
                    log.actions.append(("preempt", s, before[s], []))
                    self._release(s)
                    self.counts["preempt"] += 1
                    continue
                self._after_compress(s, before[s], log)
            return
        if hooks is not None and hasattr(hooks, "post_compress"):
            hooks.post_compress(self, t, comps)
        for s in comps:
            self._after_compress(s, before[s], log)

    def _after_compress(self, s, before, log):
        st = self.seats[s]
        after = list(st.req.pages)
        self.counts["compress"] += 1
        self.counts["cow_pages"] += sum(1 for a, b in zip(before, after) if a != b)
        if st.holds_prefix:
            g = st.group
            if after[:self.npre] == self.prefix[g]:
                # compacted in place as the prefix's only holder: it is no longer the prefix
                self.prefix_alive[g] = False
            st.holds_prefix = False
        log.actions.append(("compress", s, before, after))
