"""Benchmark of the GrowPage capacity-boundary engine on GB300.

Workload (default, ``--workload batch64``): 64 Llama-8B-shaped requests (32
layers, 32 query / 8 KV heads, d = 128, bf16 K/V) of U{4..128} pages in a
shuffled shared pool (about 142 GB of K/V), every request at a capacity
boundary at each step.  One timed step, through the C ABI: the summary
update of the boundary token (A1), one demand call over the 64 requests --
calibration + RoPE, scoring, softmax, D_p (A2-A5) --, the decision (A6),
Grow (A7) for the requests whose short-term demand rose and one Compress &
Hold call (A8-A10) for the others.  Between steps (untimed) come the 255
decode steps of summary updates to the next boundary, and the page each
request gained or freed is refilled with fresh synthetic tokens.

Output: one JSON line (rank 0).  value = boundary events/s over all GPUs
(replicas; the path does not shard).  roofline = the dominant kernel's
algorithmic HBM bytes per launch / its mean CUDA-event launch time, against
the measured copy bandwidth.  e2e = the same steps on a fresh identical
setup with each step's queries copied from pinned host memory.
cpu_baseline = the fp64 oracle on whole requests of the same workload on the
host cores.  ``--impl reference`` times that oracle as the reference arm.
Other lines: ``--workload llama8b_single`` (one request's decode stream),
``qwen3_8b``, ``stream256``.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "boundary events/s and KV GB/s (fraction of GB300 HBM roofline) vs CPU oracle"
PAGE = 256
PHASE = 512
EVENT_STRIDE = 256


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_OF = {"boundary_demand": "k_demand_tc", "compress_hold": "k_compress"}
# the sources each kernel is built from (its capture is void once they change)
KERNEL_SOURCES = {"k_demand_tc": ["k_demand_tc.cu", "demand_common.cuh", "tc_ptx.cuh", "gp_kernels.h"],
                  "k_compress": ["k_compress.cu", "gp_kernels.h"]}


def _sources_sha(kernel: str) -> str:
    """sha256 over a kernel's source files (file name and bytes, in order)."""
    import hashlib
    d = os.path.join(ROOT, "paged_kv_cache_step_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(b"\0")
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(kernel: str, bytes_per_launch: float):
    """DRAM bytes per launch from the committed ncu capture, scaled by the
    launch's algorithmic bytes; None when the kernel's sources have changed
    since the capture or no capture exists."""
    name = KERNEL_OF.get(kernel, "")
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(name, None)
    except Exception:
        return None
    if not rec or rec.get("source_sha256") != _sources_sha(name):
        return None
    ratio = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["algorithmic_bytes"]
    return ratio * bytes_per_launch


def replica_value(total_ms: float, steps: int):
    """Whole-job events/s of N independent replicas (one per rank): the
    slowest rank's time bounds the job, and every rank processed `steps`
    events.  Returns (events/s over all ranks, max time in ms)."""
    world = torch.distributed.get_world_size() if torch.distributed.is_initialized() else 1
    t = torch.tensor([total_ms], dtype=torch.float64)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(t.item())
    return world * steps / (ms_max / 1e3), ms_max


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Clocks:
    """nvidia-smi sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int, path: str | None):
        self.proc = None
        self.path = path
        self.gpu = gpu
        if path is None:
            return
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1].split()[0]))
                mx = max(mx, float(p[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _metric(args) -> int:
    return 1 if getattr(args, "demand_metric", "top_p") == "entropy" else 0


class Stream:
    """Config-2 decode stream driven through the C ABI."""

    def __init__(self, device, num_pages=64, P=32, fill=False, metric=0):
        import paged_kv_cache_step_gb300 as gp
        self.gp = gp
        gp.load(build_if_missing=False)
        self.w = synth.make_workload("llama8b_single", device=device, num_pages=num_pages, P=P)
        w = self.w
        sh = w.shape
        self.torch_stream = torch.cuda.Stream(device=device)
        cfg = gp.gp_config_default(
            num_layers=sh.num_layers, num_q_heads=sh.num_q_heads, num_kv_heads=sh.num_kv_heads,
            head_dim=sh.head_dim, kv_dtype=gp.GP_DTYPE_BF16, q_dtype=gp.GP_DTYPE_BF16,
            max_slots=8, num_pages=w.num_pages, max_pages_per_req=256, rope_theta=sh.rope_theta)
        cfg.demand_metric = metric
        self.cfg = cfg
        self.ctx = gp.gp_create(cfg, w.k_cache, w.v_cache, self.torch_stream)
        used = set(w.block_tables[0])
        for _ in range(w.num_pages):
            gp.gp_page_alloc(self.ctx)
        for pg in range(w.num_pages):
            if pg not in used:
                gp.gp_page_unref(self.ctx, pg)
        slot = gp.gp_slot_acquire(self.ctx)
        self.req = gp.Request(slot, w.block_tables[0], w.positions[0], cfg.max_pages_per_req)
        self.slots = torch.tensor([slot], dtype=torch.int32, device=device)
        self.first = torch.ones(1, dtype=torch.uint8, device=device)
        self.notfirst = torch.zeros(1, dtype=torch.uint8, device=device)
        self.t = 0            # decode step index of the stream
        self.started = False
        self.units = sh.num_layers * sh.num_kv_heads
        self.row_bytes = sh.head_dim * 2
        self.q_bytes = sh.num_layers * sh.num_q_heads * sh.head_dim * 2
        self.actions = {"grow": 0, "compress": 0, "fallback": 0}
        self.fill = fill   # hole-fill compaction (order-destroying variant) instead of the stable one

    def _query(self):
        # drawn on the engine stream, which reads it: a tensor that the
        # caching allocator hands out on one stream and another stream reads
        # can be overwritten by the next allocation before the read is done
        kind = (self.t // PHASE) % 2 == 0      # concentrated phases first
        with torch.cuda.stream(self.torch_stream):
            return synth.query_step(self.w, [kind])

    def _update(self, q):
        # the engine launches on its own stream, which draws q
        self.gp.gp_update_summaries(self.ctx, 1, self.slots, q,
                                    self.notfirst if self.started else self.first)
        self.started = True
        self.t += 1

    def advance(self, steps: int):
        """Non-boundary decode steps (summary updates only)."""
        for _ in range(steps):
            q = self._query()
            self.torch_stream.wait_stream(torch.cuda.current_stream())
            self._update(q)
        self.req.pos = self.w.positions[0] + self.t

    def event(self, q):
        """One boundary event; q is the boundary token's query (on device)."""
        gp = self.gp
        self._update(q)
        self.req.pos = self.w.positions[0] + self.t
        P = self.req.num_pages
        dem = gp.gp_boundary_demand(self.ctx, [self.req], q)
        act = gp.gp_decide(self.ctx, [self.req], dem)[0]
        scan = (P * PAGE - 16) * self.units * self.row_bytes
        if act.kind == gp.GP_ACT_GROW:
            gp.gp_grow_page(self.ctx, self.req)
            self.actions["grow"] += 1
        else:
            if self.fill:
                gp.gp_compress_fill(self.ctx, [self.req])
            else:
                gp.gp_compress_hold(self.ctx, [self.req])
            self.actions["compress"] += 1
            self.actions["fallback"] += int(act.fallback)
        return scan, act.kind


def _single_size(args):
    """Pages of the single request at its first boundary, and its pool."""
    P = args.single_pages or 32
    return {"P": P, "num_pages": 2 * P}


def _moved(gp, ctx):
    return gp.gp_stats(ctx)["moved_rows"]


def run_gpu(args, world, rank, local):
    import paged_kv_cache_step_gb300 as gp
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peak, peak_src = _peaks()
    s = Stream(device, fill=args.compaction == "fill", metric=_metric(args), **_single_size(args))
    # warm the summaries over the first boundary interval
    s.advance(EVENT_STRIDE - 1)

    def one_event(q):
        return s.event(q)  # (K bytes scanned, action kind)

    # warm-up events (untimed)
    for _ in range(args.warmup):
        q = s._query()
        one_event(q)
        s.advance(EVENT_STRIDE - 1)
    torch.cuda.synchronize()
    gp.gp_reset_timing(s.ctx)
    gp.gp_set_timing(s.ctx, 1)
    moved0 = _moved(gp, s.ctx)
    if world > 1:
        torch.distributed.barrier()
    clock_file = os.path.join(tempfile.gettempdir(), f"growpage_bench_clocks_{os.getpid()}_r{rank}.csv")
    clocks = Clocks(local, clock_file)
    times, kinds = [], []
    scan_bytes = 0
    for _ in range(args.steps):
        q = s._query()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(s.torch_stream)
        sb, kind = one_event(q)
        ev1.record(s.torch_stream)
        scan_bytes += sb
        kinds.append(kind)
        torch.cuda.synchronize()
        times.append(ev0.elapsed_time(ev1))
        s.advance(EVENT_STRIDE - 1)    # not timed
    clk = clocks.stop()
    gp.gp_set_timing(s.ctx, 0)
    moved = _moved(gp, s.ctx) - moved0
    kern = {}
    launches = 0
    for k, name in gp.KERNEL_NAMES.items():
        ms, n = gp.gp_kernel_time(s.ctx, k)
        kern[name] = {"ms": ms, "launches": n}
        launches += n
    total_ms = sum(times)
    # the EMA launches of the untimed decode steps are not in the timed region
    ema_timed = args.steps
    launches = launches - kern["ema_update"]["launches"] + ema_timed

    comp_bytes = moved * s.row_bytes * 2 * 2
    # roofline: dominant kernel by device time inside the boundary events
    dem = kern["boundary_demand"]
    cmp_ = kern["compress_hold"]
    rl = {}
    if dem["launches"]:
        a = scan_bytes / dem["launches"] / (dem["ms"] / dem["launches"] / 1e3) / 1e9
        rl["boundary_demand"] = {"bound": "hbm", "achieved": a, "peak": peak, "unit": "GB/s",
                                 "frac": a / peak, "bytes_per_launch": scan_bytes / dem["launches"],
                                 "ms_per_launch": dem["ms"] / dem["launches"]}
    if cmp_["launches"]:
        a = comp_bytes / cmp_["launches"] / (cmp_["ms"] / cmp_["launches"] / 1e3) / 1e9
        rl["compress_hold"] = {"bound": "hbm", "achieved": a, "peak": peak, "unit": "GB/s",
                               "frac": a / peak, "bytes_per_launch": comp_bytes / cmp_["launches"],
                               "ms_per_launch": cmp_["ms"] / cmp_["launches"]}
    dom = max(rl, key=lambda k: kern[k]["ms"]) if rl else None
    # events by action (event time on the engine stream), and demand alone
    # (device time of its prep and scan kernels)
    by_action = {}
    for kid, name in ((gp.GP_ACT_GROW, "grow"), (gp.GP_ACT_COMPRESS, "compress"), (gp.GP_ACT_SHRINK, "shrink")):
        t = [ms for ms, k in zip(times, kinds) if k == kid]
        if t:
            by_action[name] = {"events": len(t), "ms_mean": sum(t) / len(t), "events_per_s": len(t) / (sum(t) / 1e3)}
    demand_ms = dem["ms"] + kern["prep_queries"]["ms"]
    if dem["launches"] and demand_ms > 0:
        by_action["demand_only"] = {"events": dem["launches"], "ms_mean": demand_ms / dem["launches"],
                                    "events_per_s": dem["launches"] / (demand_ms / 1e3),
                                    "timing": "device time of the prep and demand kernels"}

    actions = dict(s.actions)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(s, args.cpu_seconds)
    gp.gp_destroy(s.ctx)
    del s
    torch.cuda.empty_cache()

    # e2e: the same event sequence on a fresh, identical stream, with the
    # boundary query copied from pinned host memory and the D_p sums read
    # back every step, inside the timed region
    e2e = None
    if not args.no_e2e:
        s = Stream(device, fill=args.compaction == "fill", metric=_metric(args), **_single_size(args))
        s.advance(EVENT_STRIDE - 1)
        for _ in range(args.warmup):
            q = s._query()
            one_event(q)
            s.advance(EVENT_STRIDE - 1)
        torch.cuda.synchronize()
        dev_q = torch.empty_like(s._query(), device=device)
        e2e_times = []
        for _ in range(args.steps):
            q = s._query()
            torch.cuda.synchronize()
            hq = q.cpu().pin_memory()
            torch.cuda.synchronize()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(s.torch_stream)
            with torch.cuda.stream(s.torch_stream):
                dev_q.copy_(hq, non_blocking=True)
            one_event(dev_q)
            ev1.record(s.torch_stream)
            torch.cuda.synchronize()
            e2e_times.append(ev0.elapsed_time(ev1))
            s.advance(EVENT_STRIDE - 1)
        maxp = s.cfg.max_pages_per_req
        h2d = s.q_bytes + 48 + 4 * maxp * 2 + 4
        d2h = 16 + 4 + (s.cfg.num_layers * s.cfg.num_kv_heads * 2 * 8 if _metric(args) else 0)
        e2e = {"value": len(e2e_times) / (sum(e2e_times) / 1e3), "unit": "events/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "step_ms": [round(x, 4) for x in e2e_times],
               "events": "the timed events of the value line, replayed on an identical fresh stream"}
        gp.gp_destroy(s.ctx)

    # aggregate over ranks (replicas): max time, summed events
    value, ms_max = replica_value(total_ms, args.steps)
    kv_gbs = (scan_bytes + comp_bytes) / (total_ms / 1e3) / 1e9
    s_pages = _single_size(args)["P"]
    out = {
        "metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"llama8b_single: 1 request, 32L 32q/8kv d128 bf16, {s_pages} pages x 256 "
                               f"at the first boundary, {2 * s_pages}-page pool, 512-step concentrated/diffuse "
                               "query phases, boundary every 256 decode steps"
                               + ("; hole-fill compaction (order-destroying variant)" if args.compaction == "fill"
                                  else "")
                               + ("; entropy demand metric (Sec. 5.3 ablation)" if _metric(args) else ""),
                   "l2": f"inputs larger than L2 ({16.8 * s_pages / 1000:.2f}+ GB of K scanned per event, "
                         f"{33.6 * 2 * s_pages / 1000:.2f} GB of K/V)",
                   "parallelism": f"replicas x{world}"},
        "step_ms": [round(x, 4) for x in times],
        "kv_gbs": kv_gbs,
        "kv_frac": kv_gbs / peak,
        "scan_bytes": scan_bytes, "compaction_bytes": comp_bytes,
        "actions": actions, "events_by_action": by_action,
        "roofline": dict(rl[dom], kernel=dom, peak_source=peak_src,
                         traffic=_traffic(dom, rl[dom]["bytes_per_launch"])) if dom else None,
        "kernels": {k: dict(v, **({"frac": rl[k]["frac"], "achieved_gbs": rl[k]["achieved"]}
                                  if k in rl else {})) for k, v in kern.items()},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if args.async_overlap:
        out["async_compaction"] = measure_overlap(args, device)
    return out


def measure_overlap(args, device):
    """Compaction on a side stream, overlapped with the decode steps that
    follow a boundary (App. E.3).  Whole boundary intervals -- one event and
    the EVENT_STRIDE - 1 summary updates after it, ending with the engine
    stream waiting for the compaction -- are timed with the compaction on
    the engine stream and on a side stream, each on a fresh, identical
    stream.  Returns the mean interval times and the compaction time hidden."""
    import paged_kv_cache_step_gb300 as gp
    res = {}
    for mode in ("sync", "async"):
        s = Stream(device)
        if mode == "async":
            side = torch.cuda.Stream(device=device)
            gp.gp_set_compaction_stream(s.ctx, side)
        s.advance(EVENT_STRIDE - 1)
        for _ in range(args.warmup):
            s.event(s._query())
            s.advance(EVENT_STRIDE - 1)
            gp.gp_wait_compaction(s.ctx, s.torch_stream)
        torch.cuda.synchronize()
        gp.gp_reset_timing(s.ctx)
        gp.gp_set_timing(s.ctx, 1)
        times = []
        for _ in range(args.overlap_intervals):
            q = s._query()
            torch.cuda.synchronize()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(s.torch_stream)
            s.event(q)
            s.advance(EVENT_STRIDE - 1)
            gp.gp_wait_compaction(s.ctx, s.torch_stream)
            ev1.record(s.torch_stream)
            torch.cuda.synchronize()
            times.append(ev0.elapsed_time(ev1))
        gp.gp_set_timing(s.ctx, 0)
        cms, cn = gp.gp_kernel_time(s.ctx, gp.GP_KERNEL_COMPRESS)
        res[mode] = (sum(times) / len(times), cms / len(times), s.actions["compress"])
        gp.gp_destroy(s.ctx)
        del s
        torch.cuda.empty_cache()
    sync_ms, comp_ms, _ = res["sync"]
    async_ms = res["async"][0]
    return {"interval_ms_sync": sync_ms, "interval_ms_async": async_ms,
            "compaction_ms_per_interval": comp_ms,
            "hidden_frac": (sync_ms - async_ms) / comp_ms if comp_ms > 0 else None,
            "intervals": args.overlap_intervals,
            "interval": f"one boundary event + {EVENT_STRIDE - 1} decode steps (summary updates)"}


# ---------------------------------------------------------------------------
# the other configurations (one JSON line each; not the default line)
# ---------------------------------------------------------------------------

def _engine_over(gp, w, stream, max_slots, max_pages, policy, metric=0):
    sh = w.shape
    cfg = gp.gp_config_default(
        num_layers=sh.num_layers, num_q_heads=sh.num_q_heads, num_kv_heads=sh.num_kv_heads,
        head_dim=sh.head_dim, kv_dtype=gp.GP_DTYPE_BF16, q_dtype=gp.GP_DTYPE_BF16,
        max_slots=max_slots, num_pages=w.num_pages, max_pages_per_req=max_pages, rope_theta=sh.rope_theta)
    if policy == "fixed":
        cfg.policy = gp.GP_POLICY_FIXED
    cfg.demand_metric = metric
    return cfg, gp.gp_create(cfg, w.k_cache, w.v_cache, stream)


def _kernel_report(gp, ctx, peak, scan_bytes, comp_bytes):
    kern, rl = {}, {}
    for k, name in gp.KERNEL_NAMES.items():
        ms, n = gp.gp_kernel_time(ctx, k)
        kern[name] = {"ms": ms, "launches": n}
    for name, nbytes in (("boundary_demand", scan_bytes), ("compress_hold", comp_bytes)):
        k = kern[name]
        if k["launches"] and k["ms"] > 0:
            a = nbytes / (k["ms"] / 1e3) / 1e9
            rl[name] = {"bound": "hbm", "achieved": a, "peak": peak, "unit": "GB/s", "frac": a / peak,
                        "bytes_per_launch": nbytes / k["launches"], "ms_per_launch": k["ms"] / k["launches"]}
            k.update(frac=a / peak, achieved_gbs=a)
    dom = max(rl, key=lambda n: kern[n]["ms"]) if rl else None
    return kern, rl, dom


class Batch:
    """A batch configuration (64 Llama-8B-like requests, or 16 Qwen3-8B-like
    ones) driven through the C ABI, every request at a capacity boundary at
    each step.

    Decode step t of request r draws a concentrated or diffuse query by the
    workload's phase schedule (synth.batch_kinds: 32-step phases alternating
    from the request's seeded first kind, the 64-step history being steps
    0..63).  A boundary comes every 256 decode steps, when the request's last
    page is full: the summary update of the boundary token (A1), one demand
    call over every request (A2-A5), the decision (A6), Grow (A7) for the
    requests that grow and one Compress & Hold call (A8-A10) for the others.
    Between boundaries (untimed) the 255 decode steps update the summaries,
    and the page a Grow added, or the page a Compress & Hold freed, is filled
    with fresh synthetic tokens, so that every request is full again."""

    def __init__(self, gp, name, device, policy="growpage", metric=0, extra_pages=0, n=None, selection=None):
        self.gp = gp
        kw = {"n": n} if n else {}
        self.w = w = synth.make_workload(name, device=device, extra_pages=extra_pages, **kw)
        self.stream = torch.cuda.Stream(device=device)
        self.cfg, self.ctx = _engine_over(gp, w, self.stream, max(4, w.n), 256, policy, metric)
        used = set(p for t in w.block_tables for p in t)
        for _ in range(w.num_pages):
            gp.gp_page_alloc(self.ctx)
        for pg in range(w.num_pages):
            if pg not in used:
                gp.gp_page_unref(self.ctx, pg)
        self.reqs = [gp.Request(gp.gp_slot_acquire(self.ctx), t, w.positions[r], 256)
                     for r, t in enumerate(w.block_tables)]
        if selection:
            gp.gp_set_selection_mode(self.ctx, {"speculative": gp.GP_SELECT_SPECULATIVE,
                                                "in_compaction": gp.GP_SELECT_IN_COMPACTION}[selection])
        self.slots = torch.tensor([q.slot for q in self.reqs], dtype=torch.int32, device=device)
        self.first = torch.ones(w.n, dtype=torch.uint8, device=device)
        self.notfirst = torch.zeros(w.n, dtype=torch.uint8, device=device)
        sh = w.shape
        self.units = sh.num_layers * sh.num_kv_heads
        self.row = sh.head_dim * 2
        self.q_bytes = sh.num_layers * w.n * sh.num_q_heads * sh.head_dim * 2
        self.ema_bytes = w.n * sh.num_layers * sh.num_q_heads * sh.head_dim * (2 + 32)
        self.pos0 = list(w.positions)
        self.t = 0
        self.actions = {"grow": 0, "compress": 0, "fallback": 0}
        for q in w.history:
            self._update(q)

    def _update(self, q):
        # after the refills, which run on the current stream; the engine
        # launches on its own stream
        self.stream.wait_stream(torch.cuda.current_stream())
        self.gp.gp_update_summaries(self.ctx, self.w.n, self.slots, q,
                                    self.first if self.t == 0 else self.notfirst)
        self.t += 1

    def query(self):
        # drawn on the engine stream, which reads it (see Stream._query)
        with torch.cuda.stream(self.stream):
            return synth.query_step(self.w, synth.batch_kinds(self.w, self.t))

    def decode(self, count: int):
        """Non-boundary decode steps: summary updates only."""
        for _ in range(count):
            self._update(self.query())

    def event(self, q):
        """One boundary step of every request; q: the boundary token's queries
        [L][n][Hq][d] on the device.  Returns (K bytes scanned, grown, compressed)."""
        gp = self.gp
        tb = self.t
        self._update(q)
        for r, req in enumerate(self.reqs):
            req.pos = self.pos0[r] + (tb - 64)
        scan = sum((r.num_pages * PAGE - 16) * self.units * self.row for r in self.reqs)
        dem = gp.gp_boundary_demand(self.ctx, self.reqs, q)
        acts = gp.gp_decide(self.ctx, self.reqs, dem)
        grown, comp = [], []
        for i, (r, a) in enumerate(zip(self.reqs, acts)):
            if a.kind == gp.GP_ACT_GROW:
                gp.gp_grow_page(self.ctx, r)
                grown.append(i)
                self.actions["grow"] += 1
            else:
                comp.append(i)
                self.actions["compress"] += 1
                self.actions["fallback"] += int(a.fallback)
        if comp:
            gp.gp_compress_hold(self.ctx, [self.reqs[i] for i in comp])
        return scan, grown, comp

    def refill(self, grown, comp):
        """Fresh tokens in each request's last page (the one a Grow added or a
        Compress & Hold freed); waits for the compaction, which reads it."""
        torch.cuda.current_stream().wait_stream(self.stream)
        self.gp.gp_wait_compaction(self.ctx, torch.cuda.current_stream())
        for i in sorted(grown + comp):
            r = self.reqs[i]
            synth.fill_pages(self.w, i, [int(r.table[r.num_pages - 1])])

    def between(self, grown, comp):
        self.refill(grown, comp)
        self.decode(EVENT_STRIDE - 1)

    def close(self):
        if self.ctx:
            self.gp.gp_destroy(self.ctx)
            self.ctx = None


def measure_overlap_batch(args, device, extra):
    """Compaction on a side stream overlapped with a decode step (App. E.3),
    timed on the device.  Each interval: the boundary step's summary update,
    demand and decision, Grow for the growing requests, one Compress & Hold
    call for the others, then a decode step of attention (all layers) over
    the growing requests' caches on the engine stream, which finally waits
    for the compaction.  Run once with the compaction on the engine stream
    and once on a side stream, on fresh identical setups; CUDA events on the
    engine stream bracket each interval."""
    import paged_kv_cache_step_gb300 as gp
    res = {}
    for mode in ("sync", "async"):
        b = Batch(gp, args.workload, device, args.policy, _metric(args), extra, args.batch_requests,
                  _selection(args))
        sh = b.w.shape
        if mode == "async":
            side = torch.cuda.Stream(device=device)
            gp.gp_set_compaction_stream(b.ctx, side)
        first = torch.zeros(b.w.n, dtype=torch.uint8, device=device)

        def interval(q, timed):
            tb = b.t
            b._update(q)
            for r, req in enumerate(b.reqs):
                req.pos = b.pos0[r] + (tb - 64)
            dem = gp.gp_boundary_demand(b.ctx, b.reqs, q)
            acts = gp.gp_decide(b.ctx, b.reqs, dem)
            grown = [i for i, a in enumerate(acts) if a.kind == gp.GP_ACT_GROW]
            comp = [i for i, a in enumerate(acts) if a.kind != gp.GP_ACT_GROW]
            for i in grown:
                gp.gp_grow_page(b.ctx, b.reqs[i])
            if timed:
                ev0 = torch.cuda.Event(enable_timing=True)
                ev0.record(b.stream)
            if comp:
                gp.gp_compress_hold(b.ctx, [b.reqs[i] for i in comp])
            if grown:
                reqs = [b.reqs[i] for i in grown]
                ntok = [(r.num_pages - 1) * PAGE for r in reqs]
                with torch.cuda.stream(b.stream):
                    qa = torch.randn(sh.num_layers, len(reqs), sh.num_q_heads, sh.head_dim,
                                     device=device).to(torch.bfloat16)
                    out = torch.empty(len(reqs), sh.num_q_heads, sh.head_dim, device=device)
                for layer in range(sh.num_layers):
                    gp.gp_decode_attention(b.ctx, layer, reqs, ntok, qa[layer], first[:len(reqs)], out)
            gp.gp_wait_compaction(b.ctx, b.stream)
            ms = None
            if timed:
                ev1 = torch.cuda.Event(enable_timing=True)
                ev1.record(b.stream)
                torch.cuda.synchronize()
                ms = ev0.elapsed_time(ev1)
            return grown, comp, ms

        for _ in range(args.warmup):
            gr, cm, _ = interval(b.query(), False)
            b.between(gr, cm)
        torch.cuda.synchronize()
        gp.gp_reset_timing(b.ctx)
        times = []
        for _ in range(args.overlap_intervals):
            q = b.query()
            torch.cuda.synchronize()
            gp.gp_set_timing(b.ctx, 1)
            gr, cm, ms = interval(q, True)
            gp.gp_set_timing(b.ctx, 0)
            times.append(ms)
            b.between(gr, cm)
        k_ms = {name: gp.gp_kernel_time(b.ctx, k)[0] for k, name in gp.KERNEL_NAMES.items()}
        res[mode] = {"interval_ms": sum(times) / len(times),
                     "compaction_ms": k_ms["compress_hold"] / len(times),
                     "attention_ms": k_ms["decode_attention"] / len(times)}
        b.close()
        del b
        torch.cuda.empty_cache()
    s_, a_ = res["sync"], res["async"]
    overlapable = min(s_["compaction_ms"], s_["attention_ms"])
    return {"sync": s_, "async": a_, "intervals": args.overlap_intervals,
            "hidden_ms": s_["interval_ms"] - a_["interval_ms"],
            "hidden_frac_of_shorter": (s_["interval_ms"] - a_["interval_ms"]) / overlapable if overlapable > 0 else None,
            "interval": "one Compress & Hold call (the compressing requests) and one decode step of "
                        "attention over the growing requests (all layers), from the compaction's "
                        "launch to the engine stream's wait for it; device time (CUDA events)"}


def _selection(args):
    return None if args.selection == "auto" else args.selection


def _batch_extra_pages(w_n: int, steps: int) -> int:
    """Free pages beyond the configuration's spare ones, so that the Grows of
    every step of the run can be granted (about half the requests grow)."""
    return w_n * (steps + 2) // 2 + w_n


def _batch_desc(name, w, extra, policy, metric):
    sizes = [len(t) for t in w.block_tables]
    return (f"{name}: {synth.CONFIGS[name][2]}; {w.n} requests, P = {min(sizes)}..{max(sizes)} "
            f"(mean {sum(sizes) / len(sizes):.1f}) pages at the first boundary, pool of "
            f"{w.num_pages - extra} pages + {extra} free reserve pages so that every Grow of the run "
            f"is granted; each step every request is at a capacity boundary: summary update of the "
            f"boundary token, one demand call over all {w.n}, decide, Grow or one Compress & Hold "
            f"call (policy {policy}); between steps (untimed) 255 decode steps of summary updates and "
            f"the added or freed page of every request refilled with fresh tokens"
            + ("; entropy demand metric (Sec. 5.3 ablation)" if metric else ""))


def run_batch(args, world, rank, local):
    """The batch line (the default: config 3, 64 requests): value = boundary
    events per second over all ranks (replicas), each step one boundary event
    of every request of the batch."""
    import paged_kv_cache_step_gb300 as gp
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    gp.load(build_if_missing=False)
    peak, peak_src = _peaks()
    n_req = args.batch_requests or (64 if args.workload == "batch64" else 16)
    extra = _batch_extra_pages(n_req, args.warmup + args.steps)
    b = Batch(gp, args.workload, device, args.policy, _metric(args), extra, args.batch_requests,
                  _selection(args))
    w = b.w
    desc = _batch_desc(args.workload, w, extra, args.policy, _metric(args))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_batch(w, args.cpu_seconds)
    for _ in range(args.warmup):
        _, gr, cm = b.event(b.query())
        b.between(gr, cm)
    torch.cuda.synchronize()
    gp.gp_reset_timing(b.ctx)
    moved0 = gp.gp_stats(b.ctx)["moved_rows"]
    acts0 = dict(b.actions)
    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local, os.path.join(tempfile.gettempdir(), f"growpage_clk_{os.getpid()}_r{rank}.csv"))
    times, scan_bytes = [], 0
    for _ in range(args.steps):
        q = b.query()
        torch.cuda.synchronize()
        gp.gp_set_timing(b.ctx, 1)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(b.stream)
        sb, gr, cm = b.event(q)
        ev1.record(b.stream)
        torch.cuda.synchronize()
        gp.gp_set_timing(b.ctx, 0)
        times.append(ev0.elapsed_time(ev1))
        scan_bytes += sb
        b.between(gr, cm)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    comp_bytes = (gp.gp_stats(b.ctx)["moved_rows"] - moved0) * b.row * 4
    kern, rl, dom = _kernel_report(gp, b.ctx, peak, scan_bytes, comp_bytes)
    ema = kern["ema_update"]
    if ema["launches"] and ema["ms"] > 0:
        a = ema["launches"] * b.ema_bytes / (ema["ms"] / 1e3) / 1e9
        ema.update(achieved_gbs=a, frac=a / peak, bytes_per_launch=b.ema_bytes)
    launches = sum(k["launches"] for k in kern.values())
    actions = {k: b.actions[k] - acts0[k] for k in b.actions}
    attn = measure_attention(gp, b.ctx, w, b.reqs, b.stream, peak, args) if args.decode_attention else None
    b.close()
    del b, w
    torch.cuda.empty_cache()
    overlap = None
    if args.async_overlap:
        overlap = measure_overlap_batch(args, device, _batch_extra_pages(
            n_req, args.warmup + args.overlap_intervals))

    # e2e: the same steps on a fresh, identical setup, through the public
    # calls, with each step's boundary queries copied from pinned host memory
    # inside the timed region (gp_boundary_demand reads the D_p sums back)
    e2e = None
    if not args.no_e2e:
        b = Batch(gp, args.workload, device, args.policy, _metric(args), extra, args.batch_requests,
                  _selection(args))
        for _ in range(args.warmup):
            _, gr, cm = b.event(b.query())
            b.between(gr, cm)
        torch.cuda.synchronize()
        dev_q = None
        e2e_times = []
        for _ in range(args.steps):
            q = b.query()
            torch.cuda.synchronize()
            hq = q.cpu().pin_memory()
            if dev_q is None:
                dev_q = torch.empty(hq.shape, dtype=hq.dtype, device=device)
            torch.cuda.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(b.stream)
            with torch.cuda.stream(b.stream):
                dev_q.copy_(hq, non_blocking=True)
            _, gr, cm = b.event(dev_q)
            ev1.record(b.stream)
            torch.cuda.synchronize()
            e2e_times.append(ev0.elapsed_time(ev1))
            b.between(gr, cm)
        n = b.w.n
        h2d = b.q_bytes + n * (48 + 4 * 256) + 8 * (n + 1) + 4 * n
        d2h = 16 * n + 4 + (n * b.units * 2 * 8 if _metric(args) else 0)
        e2e_value = replica_value(sum(e2e_times), args.steps)[0] * n
        e2e = {"value": e2e_value, "unit": "events/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "step_ms": [round(x, 3) for x in e2e_times],
               "events": "the timed steps of the value line, replayed on an identical fresh setup"}
        b.close()
        del b
        torch.cuda.empty_cache()

    total = sum(times)
    value, ms_max = replica_value(total, args.steps)
    value *= n_req
    out = {
        "metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "events_per_step": n_req,
                   "l2": "inputs larger than L2 (tens of GB of K scanned per step)",
                   "parallelism": f"replicas x{world}"},
        "step_ms": [round(x, 3) for x in times],
        "kv_gbs": (scan_bytes + comp_bytes) / (total / 1e3) / 1e9,
        "scan_bytes": scan_bytes, "compaction_bytes": comp_bytes, "actions": actions,
        "roofline": dict(rl[dom], kernel=dom, peak_source=peak_src,
                         traffic=_traffic(dom, rl[dom]["bytes_per_launch"])) if dom else None,
        "kernels": kern, "gpu_launches": launches, "clocks": clk, "e2e": e2e,
        **({"decode_attention": attn} if attn else {}),
        **({"async_compaction": overlap} if overlap else {})}
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def measure_attention(gp, ctx, w, reqs, ts, peak, args):
    """One decode step of attention over every request's whole cache: the
    L layer calls of gp_decode_attention (summary update fused in).
    Algorithmic bytes per layer: K and V of every attended token."""
    sh = w.shape
    n = len(reqs)
    ntok = [r.num_pages * PAGE for r in reqs]
    device = w.device
    q = torch.randn(sh.num_layers, n, sh.num_q_heads, sh.head_dim, device=device).to(torch.bfloat16)
    first = torch.zeros(n, dtype=torch.uint8, device=device)
    out = torch.empty(n, sh.num_q_heads, sh.head_dim, device=device)
    torch.cuda.synchronize()
    row = sh.head_dim * 2
    step_bytes = sum(ntok) * sh.num_kv_heads * row * 2 * sh.num_layers

    def timed():
        for _ in range(2):
            for layer in range(sh.num_layers):
                gp.gp_decode_attention(ctx, layer, reqs, ntok, q[layer], first, out)
        torch.cuda.synchronize()
        times = []
        for _ in range(max(3, args.steps)):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(ts)   # the engine's stream, which the launches go to
            for layer in range(sh.num_layers):
                gp.gp_decode_attention(ctx, layer, reqs, ntok, q[layer], first, out)
            ev1.record(ts)
            torch.cuda.synchronize()
            times.append(ev0.elapsed_time(ev1))
        ms = sum(times) / len(times)
        return ms, step_bytes / (ms / 1e3) / 1e9

    ms, a = timed()                                       # the kernel AUTO picks (tcgen05 for bf16, d 128)
    gp.gp_set_scan_kernel(ctx, gp.GP_SCAN_CUDA_CORE)      # the CUDA-core kernel on the same step, for comparison
    ms_cc, a_cc = timed()
    gp.gp_set_scan_kernel(ctx, gp.GP_SCAN_AUTO)
    return {"ms_per_decode_step": ms, "bytes_per_step": step_bytes, "achieved_gbs": a, "peak": peak,
            "frac": a / peak, "layers": sh.num_layers, "requests": n,
            "cuda_core_kernel": {"ms_per_decode_step": ms_cc, "achieved_gbs": a_cc, "frac": a_cc / peak}}


def run_stream(args, device):
    """The continuous-batching stream: value = boundary events per second of
    engine device time (every engine kernel, timed per launch on its stream);
    the loop's synthetic page fills and host bookkeeping are not engine work."""
    import paged_kv_cache_step_gb300 as gp
    from synth.stream import ContinuousBatch
    peak, peak_src = _peaks()
    w = synth.make_workload("stream256", device=device)
    ts = torch.cuda.Stream(device=device)
    cfg, ctx = _engine_over(gp, w, ts, 256, 128, "growpage")
    drv = ContinuousBatch(gp, ctx, w, 128)
    units = cfg.num_layers * cfg.num_kv_heads
    row = cfg.head_dim * 2
    scan = [0]

    class Hooks:
        def post_demand(self, d, t, bseats, q_b, dem, acts):
            scan[0] += sum((d.seats[s].req.num_pages * PAGE - 16) * units * row for s in bseats)

    with torch.cuda.stream(ts):
        for t in range(args.warmup):
            drv.step(t)
        torch.cuda.synchronize()
        gp.gp_reset_timing(ctx)
        gp.gp_set_timing(ctx, 1)
        b0, moved0 = drv.counts["boundary"], gp.gp_stats(ctx)["moved_rows"]
        live0 = drv.live_sum
        clocks = Clocks(device.index or 0, os.path.join(tempfile.gettempdir(), f"growpage_clk_{os.getpid()}.csv"))
        t0 = time.perf_counter()
        for t in range(args.warmup, args.warmup + args.steps):
            drv.step(t, hooks=Hooks())
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        clk = clocks.stop()
    gp.gp_set_timing(ctx, 0)
    events = drv.counts["boundary"] - b0
    comp_bytes = (gp.gp_stats(ctx)["moved_rows"] - moved0) * row * 4
    kern, rl, dom = _kernel_report(gp, ctx, peak, scan[0], comp_bytes)
    # A1 over every live request of every timed step: n L Hq d (2 + 32) bytes
    ema = kern["ema_update"]
    live = drv.live_sum - live0
    if ema["launches"] and ema["ms"] > 0:
        eb = live * cfg.num_layers * cfg.num_q_heads * cfg.head_dim * (2 + 32)
        a = eb / (ema["ms"] / 1e3) / 1e9
        ema.update(achieved_gbs=a, frac=a / peak, bytes_per_launch=eb / ema["launches"],
                   live_requests_per_launch=live / ema["launches"])
    dev_ms = sum(k["ms"] for k in kern.values())
    counts = dict(drv.counts)
    gp.gp_destroy(ctx)
    return {
        "metric": METRIC, "value": events / (dev_ms / 1e3), "unit": "events/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dev_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "stream256: " + synth.CONFIGS["stream256"][2],
                   "timing": "engine device time (sum of per-launch CUDA events); step wall time separate"},
        "boundary_events": events, "wall_s": wall, "kv_gbs": (scan[0] + comp_bytes) / (dev_ms / 1e3) / 1e9,
        "scan_bytes": scan[0], "compaction_bytes": comp_bytes, "counts": counts,
        "mean_live": drv.live_sum / (args.warmup + args.steps),
        "roofline": dict(rl[dom], kernel=dom, peak_source=peak_src, traffic=None) if dom else None,
        "kernels": kern, "gpu_launches": sum(k["launches"] for k in kern.values()), "clocks": clk}


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def cpu_baseline(s, seconds: float):
    """The oracle as it stands on a bounded sample of the single-request
    workload: whole boundary events of a fresh 32-page request with a 64-step
    history (48 concentrated steps, then 16 diffuse ones), until `seconds`
    are spent."""
    w = synth.make_workload("llama8b_single", device=s.w.device)
    for t in range(64):
        w.history.append(synth.query_step(w, [t < 48]))
    threads = os.cpu_count() or 1
    spent, done = 0.0, 0
    while done == 0 or spent < seconds:
        dt, _ = _oracle_event(w, 0, threads)
        spent += dt
        done += 1
        if done >= 8:
            break
    P = len(w.block_tables[0])
    del w
    return {"value": done / spent, "unit": "events/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} whole boundary events of a {P}-page request of the same shape (every "
                      f"unit: summaries over a 64-step history, Eq. 12 + RoPE, scan, softmax, D_p, "
                      f"Delta, decision, Eq. 10 + K/V gather when compressing); numpy fp64 on "
                      f"{threads} host threads; {spent:.1f} s"}


def _oracle_event(w, r, threads: int):
    """One boundary event of request r at its first boundary, by the fp64
    oracle on the host cores, from the inputs on the device: the summaries
    over the 64-step history (Eq. 6), Eq. 12 and RoPE, every (layer, KV head)
    unit's scan, softmax and D_p (Eqs. 2, 7), Delta and the decision (Eq. 8),
    and for Compress & Hold Eq. 10's selection and the K/V gather of every
    unit.  Inputs are read as bf16 bit patterns and widened exactly.  Units
    run on a pool of `threads` host threads.  Returns (seconds, action)."""
    import oracle.growpage as og
    from concurrent.futures import ThreadPoolExecutor
    sh = w.shape
    assert sh.kv_dtype == "bf16" and sh.q_dtype == "bf16", "bf16 workloads"
    G = sh.group
    table = w.block_tables[r]
    P = len(table)
    units = sh.num_layers * sh.num_kv_heads
    idx = torch.as_tensor(table, dtype=torch.long, device=w.k_cache.device)

    def widen(t):
        return og.widen_bf16(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))

    def rows(cache, u):
        layer, h = divmod(u, sh.num_kv_heads)
        return widen(cache[layer].index_select(0, idx)[:, h]).reshape(P * PAGE, -1)

    t0 = time.perf_counter()
    qs = ql = None
    for t, q in enumerate(w.history):
        qs, ql = og.ema_update(qs, ql, widen(q[:, r]), t == 0, 0.9, 0.999)
    qt = og.summary_queries(qs, ql, widen(w.history[-1][:, r]), w.positions[r], sh.rope_theta)

    def demand(u):
        layer, h = divmod(u, sh.num_kv_heads)
        res = og.unit_boundary(qt[layer][:, h * G:(h + 1) * G], rows(w.k_cache, u), P, PAGE, 16, 0.99)
        return res.k, res.s

    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(demand, range(units)))
        kk = np.array([k for k, _ in res])
        delta = og.demand_trend(kk[:, 0], kk[:, 1], (P - 1) * PAGE)
        act = og.decide(delta, P, len(w.free_pages()), 0, 0.0)
        if act.kind != og.GROW:
            def compress(u):
                keep = og.select_retained(res[u][1], P, PAGE, 16, 64)
                og.compact_unit(rows(w.k_cache, u), keep)
                og.compact_unit(rows(w.v_cache, u), keep)
            list(ex.map(compress, range(units)))
    return time.perf_counter() - t0, act.kind


def cpu_baseline_batch(w, seconds: float):
    """The oracle as it stands on a bounded sample of the batch's first
    boundary step: whole requests (every unit), until `seconds` are spent."""
    threads = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(w.n).tolist()
    spent, done, pages, kinds = 0.0, 0, 0, []
    for r in order:
        dt, kind = _oracle_event(w, r, threads)
        spent += dt
        done += 1
        pages += len(w.block_tables[r])
        kinds.append(kind)
        if spent >= seconds:
            break
    return {"value": done / spent, "unit": "events/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of the {w.n} requests of the first boundary step ({pages} pages, "
                      f"{sum(1 for k in kinds if k != 0)} compressed), every (layer, KV head) unit: "
                      f"summaries over the 64-step history, Eq. 12 + RoPE, scan, softmax, D_p, Delta, "
                      f"decision, and Eq. 10 + K/V gather when compressing; numpy fp64 on {threads} host "
                      f"threads, one unit per task; {spent:.1f} s"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 oracle, timed on the host cores.  Each step is
    one whole boundary event -- request (step mod n) of the batch workload at
    its first boundary -- and ms_per_step is the time it actually took."""
    if rank != 0:
        return None
    if not torch.cuda.is_available():
        return {"impl": "reference",
                "unavailable": "the oracle's inputs (the batch workload's K/V cache, about 142 GB) are "
                               "generated on the CUDA device, and none is visible"}
    torch.cuda.set_device(0)
    w = synth.make_workload(args.workload if args.workload in ("batch64", "qwen3_8b") else "batch64",
                            device="cuda")
    threads = os.cpu_count() or 1
    times, pages = [], []
    for step in range(args.warmup + args.steps):
        r = step % w.n
        dt, _ = _oracle_event(w, r, threads)
        if step >= args.warmup:
            times.append(dt)
            pages.append(len(w.block_tables[r]))
    per = sum(times) / len(times)
    value = 1.0 / per
    sizes = [len(t) for t in w.block_tables]
    return {"metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": f"{w.name}: {synth.CONFIGS[w.name][2]}; {w.n} requests, P = "
                                   f"{min(sizes)}..{max(sizes)} pages; one step = one whole boundary "
                                   f"event of request (step mod {w.n}) at its first boundary "
                                   f"(mean P of the timed steps {sum(pages) / len(pages):.1f})",
                       "events_per_step": 1},
            "step_ms": [round(t * 1e3, 1) for t in times],
            "cpu_baseline": {"value": value, "unit": "events/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.steps} whole boundary events (every unit), numpy fp64 on "
                                       f"{threads} host threads"},
            "e2e": {"value": value, "unit": "events/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="batch64",
                    choices=["batch64", "llama8b_single", "qwen3_8b", "stream256"],
                    help="batch64 (default): 64 requests at a boundary per step; llama8b_single: one "
                         "request's decode stream; qwen3_8b: 16 Qwen3-like requests; stream256: the "
                         "continuous-batching stream")
    ap.add_argument("--policy", default="growpage", choices=["growpage", "fixed"])
    ap.add_argument("--single-pages", type=int, default=0,
                    help="llama8b_single: pages of the request at its first boundary (default 32)")
    ap.add_argument("--selection", default="auto", choices=["auto", "speculative", "in_compaction"],
                    help="batch workloads: where the Eq. 10 selection runs (gp_set_selection_mode)")
    ap.add_argument("--batch-requests", type=int, default=0,
                    help="batch workloads: this many requests instead of the configuration's (a small "
                         "case of the same recipe, e.g. for profiler captures)")
    ap.add_argument("--decode-attention", action="store_true",
                    help="batch workloads: also time a decode step of attention over every cache")
    ap.add_argument("--async-overlap", action="store_true",
                    help="also time compaction on a side stream overlapped with decode work (batch: a "
                         "decode step of attention; llama8b_single: summary updates)")
    ap.add_argument("--overlap-intervals", type=int, default=8)
    ap.add_argument("--demand-metric", default="top_p", choices=["top_p", "entropy"],
                    help="working-set metric of the demand estimation (entropy: the Sec. 5.3 ablation)")
    ap.add_argument("--compaction", default="stable", choices=["stable", "fill"],
                    help="llama8b_single: fill is the order-destroying hole-fill variant")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = _dist()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if torch.cuda.is_available() else "gloo")
    if args.workload == "stream256":
        if world > 1 or rank != 0:
            raise SystemExit("--workload stream256 runs on one GPU")
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        out = run_stream(args, dev)
    elif args.workload == "llama8b_single":
        out = run_gpu(args, world, rank, local)
    else:
        out = run_batch(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
