"""Benchmark of the GrowPage capacity-boundary engine on GB300.

Workload (default): a single Llama-8B-shaped request (32 layers, 32 query /
8 KV heads, d = 128, bf16 K/V) starting with 32 full pages (8192 tokens) in a
64-page pool, fed a decode stream whose queries alternate 512-step
concentrated and diffuse phases, with a capacity boundary every 256 decode
steps.  One timed step = one boundary event through the C ABI: the summary
update for the boundary token (A1), calibration + RoPE + scoring + softmax
+ D_p (A2-A5), the decision (A6), and Grow (A7) or Compress & Hold
(A8-A10).  Between timed steps the stream advances by the other 255 decode
steps (summary updates only, not timed); the freed or new page's slots hold
earlier synthetic tokens, which stand in for the new ones.

Output: one JSON line (rank 0).  value = boundary events/s over all GPUs
(replicas; the path does not shard).  roofline = the dominant kernel's
algorithmic HBM bytes per launch / its mean CUDA-event launch time, against
the measured copy bandwidth.  e2e = the same events/s with the boundary
query copied from pinned host memory every step.  cpu_baseline = the fp64
oracle on a bounded sample of the same workload on the host cores.
``--impl reference`` times that oracle as the reference arm.
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
KERNEL_SOURCES = {"k_demand_tc": ["k_demand_tc.cu", "demand_common.cuh", "gp_kernels.h"],
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
            max_slots=8, num_pages=w.num_pages, max_pages_per_req=128, rope_theta=sh.rope_theta)
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
        kind = (self.t // PHASE) % 2 == 0      # concentrated phases first
        return synth.query_step(self.w, [kind])

    def _update(self, q):
        with torch.cuda.stream(self.torch_stream):
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


def _moved(gp, ctx):
    return gp.gp_stats(ctx)["moved_rows"]


def run_gpu(args, world, rank, local):
    import paged_kv_cache_step_gb300 as gp
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peak, peak_src = _peaks()
    s = Stream(device, fill=args.compaction == "fill", metric=_metric(args))
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
        s = Stream(device, fill=args.compaction == "fill", metric=_metric(args))
        s.advance(EVENT_STRIDE - 1)
        for _ in range(args.warmup):
            q = s._query()
            one_event(q)
            s.advance(EVENT_STRIDE - 1)
        torch.cuda.synchronize()
        dev_q = torch.empty_like(s._query(), device=device)
        e2e_times = []
        for _ in range(args.steps):
            hq = s._query().cpu().pin_memory()
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
    out = {
        "metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "llama8b_single: 1 request, 32L 32q/8kv d128 bf16, 32 pages x 256 "
                               "at the first boundary, 64-page pool, 512-step concentrated/diffuse "
                               "query phases, boundary every 256 decode steps"
                               + ("; hole-fill compaction (order-destroying variant)" if args.compaction == "fill"
                                  else "")
                               + ("; entropy demand metric (Sec. 5.3 ablation)" if _metric(args) else ""),
                   "l2": "inputs larger than L2 (0.54+ GB of K scanned per event, 1.07 GB K/V)",
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


def run_batch(args, device):
    """64 requests (or 16 Qwen3-like ones) all at a boundary: per step the
    summary update, one demand call over every request, the decision and
    the actions (Grow, or Compress & Hold of every compressing request)."""
    import paged_kv_cache_step_gb300 as gp
    peak, peak_src = _peaks()
    w = synth.make_workload(args.workload, device=device)
    sh = w.shape
    ts = torch.cuda.Stream(device=device)
    cfg, ctx = _engine_over(gp, w, ts, max(4, w.n), 256, args.policy, _metric(args))
    used = set(p for t in w.block_tables for p in t)
    for _ in range(w.num_pages):
        gp.gp_page_alloc(ctx)
    for pg in range(w.num_pages):
        if pg not in used:
            gp.gp_page_unref(ctx, pg)
    reqs = [gp.Request(gp.gp_slot_acquire(ctx), t, w.positions[r], 256) for r, t in enumerate(w.block_tables)]
    slots = torch.tensor([q.slot for q in reqs], dtype=torch.int32, device=device)
    first = torch.ones(w.n, dtype=torch.uint8, device=device)
    notfirst = torch.zeros(w.n, dtype=torch.uint8, device=device)
    units = sh.num_layers * sh.num_kv_heads
    row = sh.head_dim * 2
    for t, q in enumerate(w.history):
        with torch.cuda.stream(ts):
            ts.wait_stream(torch.cuda.current_stream())
            gp.gp_update_summaries(ctx, w.n, slots, q, first if t == 0 else notfirst)
    torch.cuda.synchronize()

    def one_step(q):
        with torch.cuda.stream(ts):
            gp.gp_update_summaries(ctx, w.n, slots, q, notfirst)
        scan = sum((r.num_pages * PAGE - 16) * units * row for r in reqs)
        dem = gp.gp_boundary_demand(ctx, reqs, q)
        acts = gp.gp_decide(ctx, reqs, dem)
        comp = []
        for r, a in zip(reqs, acts):
            if a.kind == gp.GP_ACT_GROW:
                gp.gp_grow_page(ctx, r)
            else:
                comp.append(r)
        if comp:
            gp.gp_compress_hold(ctx, comp)
        return scan, len(comp)

    qs = [synth.query_step(w, [True] * w.n) for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup):
        one_step(qs[i])
    torch.cuda.synchronize()
    gp.gp_reset_timing(ctx)
    gp.gp_set_timing(ctx, 1)
    moved0 = gp.gp_stats(ctx)["moved_rows"]
    clocks = Clocks(device.index or 0, os.path.join(tempfile.gettempdir(), f"growpage_clk_{os.getpid()}.csv"))
    times, scan_bytes, ncomp = [], 0, 0
    for i in range(args.steps):
        q = qs[args.warmup + i]
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(ts)
        sb, nc = one_step(q)
        ev1.record(ts)
        torch.cuda.synchronize()
        times.append(ev0.elapsed_time(ev1))
        scan_bytes += sb
        ncomp += nc
    clk = clocks.stop()
    gp.gp_set_timing(ctx, 0)
    comp_bytes = (gp.gp_stats(ctx)["moved_rows"] - moved0) * row * 4
    kern, rl, dom = _kernel_report(gp, ctx, peak, scan_bytes, comp_bytes)
    attn = measure_attention(gp, ctx, w, reqs, ts, peak, args) if args.decode_attention else None
    gp.gp_destroy(ctx)
    total = sum(times)
    launches = sum(k["launches"] for k in kern.values())
    return {
        "metric": METRIC, "value": args.steps * w.n / (total / 1e3), "unit": "events/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {synth.CONFIGS[args.workload][2]}; policy {args.policy}"
                               + ("; entropy demand metric (Sec. 5.3 ablation)" if _metric(args) else ""),
                   "l2": "inputs larger than L2"},
        "kv_gbs": (scan_bytes + comp_bytes) / (total / 1e3) / 1e9,
        "scan_bytes": scan_bytes, "compaction_bytes": comp_bytes, "compress_events": ncomp,
        "roofline": dict(rl[dom], kernel=dom, peak_source=peak_src, traffic=None) if dom else None,
        "kernels": kern, "gpu_launches": launches, "clocks": clk,
        **({"decode_attention": attn} if attn else {})}


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
    a = step_bytes / (ms / 1e3) / 1e9
    return {"ms_per_decode_step": ms, "bytes_per_step": step_bytes, "achieved_gbs": a, "peak": peak,
            "frac": a / peak, "layers": sh.num_layers, "requests": n}


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

def _oracle_units(w, table, qt, unit_ids, P):
    """Oracle work of one boundary event on the given units: demand (A3-A5),
    Eq. 10 selection and the compaction gather."""
    import oracle.growpage as og
    sh = w.shape
    G = sh.group
    idx = torch.as_tensor(table, dtype=torch.long, device=w.k_cache.device)
    ks = []
    for u in unit_ids:
        layer, h = divmod(u, sh.num_kv_heads)
        keys = og.widen_bf16(w.k_cache[layer, idx, h].view(torch.int16).cpu().numpy().view(np.uint16))
        keys = keys.reshape(P * PAGE, -1)
        vals = og.widen_bf16(w.v_cache[layer, idx, h].view(torch.int16).cpu().numpy().view(np.uint16))
        vals = vals.reshape(P * PAGE, -1)
        t0 = time.perf_counter()
        res = og.unit_boundary(qt[layer][:, h * G:(h + 1) * G], keys, P, PAGE, 16, 0.99)
        keep = og.select_retained(res.s, P, PAGE, 16, 64)
        og.compact_unit(keys, keep)
        og.compact_unit(vals, keep)
        ks.append(time.perf_counter() - t0)
    return sum(ks)


def cpu_baseline(s, seconds: float):
    """The oracle as it stands on a bounded sample of the same event."""
    import oracle.growpage as og
    w = s.w
    sh = w.shape
    P = s.req.num_pages
    q = s._query()
    qc = q[:, 0].double().cpu().numpy()
    # summaries: the oracle's own EMA would need the whole history; the
    # sample times the boundary work (A2-A10) from the current summaries
    rng = np.random.default_rng(0)
    qbar = qc + 0.1 * rng.standard_normal(qc.shape)
    t0 = time.perf_counter()
    qt = og.summary_queries(qbar, qc, qc, s.req.pos, sh.rope_theta)
    prep = time.perf_counter() - t0
    done, spent = 0, prep
    order = list(range(s.units))
    while done < s.units and spent < seconds:
        spent += _oracle_units(w, s.req.pages, qt, order[done:done + 8], P)
        done += min(8, s.units - done)
    per_event = spent / done * s.units
    return {"value": 1.0 / per_event, "unit": "events/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} of {s.units} (layer, KV head) units of one {P}-page boundary event "
                      f"(demand, Eq. 10 selection, K/V gather; numpy fp64, BLAS threads up to the "
                      f"core count), scaled to one event"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 oracle, timed on the host cores."""
    if rank != 0:
        return None
    import oracle.growpage as og
    w = synth.make_workload("llama8b_single", device="cpu")
    sh = w.shape
    units = sh.num_layers * sh.num_kv_heads
    P = len(w.block_tables[0])
    sample_units = max(1, min(units, args.ref_units))
    rng = np.random.default_rng(0)
    times = []
    for step in range(args.warmup + args.steps):
        kind = (step // 2) % 2 == 0
        q = synth.query_step(w, [kind])
        qc = q[:, 0].double().numpy()
        qbar = qc + 0.1 * rng.standard_normal(qc.shape)
        t0 = time.perf_counter()
        qt = og.summary_queries(qbar, qc, qc, w.positions[0], sh.rope_theta)
        t = time.perf_counter() - t0
        ids = [(step * sample_units + i) % units for i in range(sample_units)]
        t += _oracle_units(w, w.block_tables[0], qt, ids, P)
        if step >= args.warmup:
            times.append(t * units / sample_units)
    per = sum(times) / len(times)
    value = 1.0 / per
    return {"metric": METRIC, "value": value, "unit": "events/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": "llama8b_single (as the GPU arm), oracle on "
                                   f"{sample_units} of {units} units per step, scaled"},
            "cpu_baseline": {"value": value, "unit": "events/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{sample_units} of {units} units per event, scaled"},
            "e2e": {"value": value, "unit": "events/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-units", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="llama8b_single",
                    choices=["llama8b_single", "batch64", "qwen3_8b", "stream256"])
    ap.add_argument("--policy", default="growpage", choices=["growpage", "fixed"])
    ap.add_argument("--decode-attention", action="store_true",
                    help="batch workloads: also time a decode step of attention over every cache")
    ap.add_argument("--async-overlap", action="store_true",
                    help="also time compaction on a side stream overlapped with decode steps")
    ap.add_argument("--overlap-intervals", type=int, default=8)
    ap.add_argument("--demand-metric", default="top_p", choices=["top_p", "entropy"],
                    help="working-set metric of the demand estimation (entropy: the Sec. 5.3 ablation)")
    ap.add_argument("--compaction", default="stable", choices=["stable", "fill"],
                    help="fill: the order-destroying hole-fill variant (reported separately)")
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
    if args.workload != "llama8b_single":
        if world > 1 or rank != 0:
            raise SystemExit("--workload other than the default runs on one GPU")
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        out = run_stream(args, dev) if args.workload == "stream256" else run_batch(args, dev)
        print(json.dumps(out), flush=True)
        return
    out = run_gpu(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
