"""Thin ctypes binding of the C ABI in include/growpage.h.

Argument marshalling only: every step of the hot path runs in the sm_103a
kernels of libgrowpage.so.  There is no fallback: if the library is missing
and cannot be built, ``load()`` raises.

Module-level functions carry the C names (``gp_create``, ``gp_boundary_demand``
...), take a context as first argument and raise ``GrowPageError`` on a
non-OK status.  Tensors are passed by device pointer; PyTorch only provides
device memory and streams.
"""

from __future__ import annotations

import ctypes as C
import struct
import os
from dataclasses import dataclass

import numpy as np

from . import _build_lib

GP_OK, GP_ERR_INVALID, GP_ERR_NO_PAGES, GP_ERR_NO_SLOTS = 0, 1, 2, 3
GP_ERR_CUDA, GP_ERR_TIMEOUT, GP_ERR_STATE, GP_ERR_UNSUPPORTED = 4, 5, 6, 7
GP_DTYPE_BF16, GP_DTYPE_F32 = 0, 1
GP_POLICY_GROWPAGE, GP_POLICY_FIXED, GP_POLICY_RANDOM, GP_POLICY_INVERSE, GP_POLICY_SHRINK = 0, 1, 2, 3, 4
GP_ACT_GROW, GP_ACT_COMPRESS, GP_ACT_SHRINK = 0, 1, 2
GP_METRIC_TOP_P, GP_METRIC_ENTROPY = 0, 1
GP_SCAN_AUTO, GP_SCAN_CUDA_CORE, GP_SCAN_TENSOR_CORE = 0, 1, 2
GP_SELECT_AUTO, GP_SELECT_SPECULATIVE, GP_SELECT_IN_COMPACTION = 0, 1, 2
GP_KERNEL_EMA, GP_KERNEL_PREP, GP_KERNEL_DEMAND, GP_KERNEL_COMPRESS, GP_KERNEL_ATTENTION = 0, 1, 2, 3, 4
GP_KERNEL_SELECT, GP_KERNEL_ENTROPY = 5, 6
KERNEL_NAMES = {0: "ema_update", 1: "prep_queries", 2: "boundary_demand", 3: "compress_hold",
                4: "decode_attention", 5: "select", 6: "entropy"}

EXPORTS = [
    "gp_config_default", "gp_create", "gp_destroy", "gp_last_error", "gp_status_string",
    "gp_page_alloc", "gp_page_ref", "gp_page_unref", "gp_page_refcount", "gp_free_page_count",
    "gp_slot_acquire", "gp_slot_release", "gp_update_summaries", "gp_boundary_demand",
    "gp_boundary_demand_noalloc",
    "gp_decide", "gp_grow_page", "gp_compress_hold", "gp_shrink", "gp_compress_fill", "gp_compact_kv",
    "gp_debug_demand_k", "gp_debug_entropy",
    "gp_debug_scores", "gp_debug_probs", "gp_debug_keep_mask", "gp_read_summaries",
    "gp_set_scan_kernel", "gp_set_timing", "gp_kernel_time", "gp_reset_timing", "gp_stats",
    "gp_debug_attention_plan",
    "gp_set_compaction_stream", "gp_wait_compaction", "gp_decode_attention",
    "gp_synchronize", "gp_debug_set_wait_limit", "gp_debug_fail_next_launch", "gp_set_selection_mode",
]


class GpConfig(C.Structure):
    _fields_ = [
        ("num_layers", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32), ("page_size", C.c_int32), ("kv_dtype", C.c_int32),
        ("q_dtype", C.c_int32), ("max_slots", C.c_int32), ("num_pages", C.c_int32),
        ("max_pages_per_req", C.c_int32), ("recent_window", C.c_int32), ("k_loc", C.c_int32),
        ("reserve_pages", C.c_int32), ("policy", C.c_int32),
        ("beta_s", C.c_double), ("beta_l", C.c_double), ("p", C.c_double), ("tau", C.c_double),
        ("rope_theta", C.c_double),
        ("random_compress", C.c_double), ("shrink_threshold", C.c_double),
        ("shrink_floor_pages", C.c_int32), ("random_seed", C.c_uint32),
        ("demand_metric", C.c_int32),
    ]


class GpRequest(C.Structure):
    _fields_ = [("slot", C.c_int32), ("num_pages", C.c_int32),
                ("block_table", C.POINTER(C.c_int32)), ("pos", C.c_int64)]


class GpDemand(C.Structure):
    _fields_ = [("sum_k_short", C.c_int64), ("sum_k_long", C.c_int64),
                ("num_candidates", C.c_int32), ("num_units", C.c_int32), ("delta", C.c_double),
                ("eff_short", C.c_double), ("eff_long", C.c_double)]


class GpAction(C.Structure):
    _fields_ = [("kind", C.c_int32), ("fallback", C.c_int32), ("forced", C.c_int32)]


class GpStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("demand_calls", "demand_requests", "grow", "compress",
                                          "fallback", "forced_grow", "cow_pages", "moved_rows",
                                          "shrink")]


class GrowPageError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


_LIB = None


def library_path() -> str:
    return _build_lib.LIB


def load(build_if_missing: bool = True):
    """Load libgrowpage.so (building it in-tree with nvcc if absent)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build_lib.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"native library {path} is missing; run __graft_entry__.build()")
        _build_lib.build()
    lib = C.CDLL(path)
    P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
    PI32 = C.POINTER(C.c_int32)
    sig = {
        "gp_config_default": (I32, [C.POINTER(GpConfig)]),
        "gp_create": (I32, [C.POINTER(GpConfig), P, P, P, C.POINTER(P)]),
        "gp_destroy": (I32, [P]),
        "gp_last_error": (C.c_char_p, [P]),
        "gp_status_string": (C.c_char_p, [I32]),
        "gp_page_alloc": (I32, [P, PI32]),
        "gp_page_ref": (I32, [P, I32]),
        "gp_page_unref": (I32, [P, I32]),
        "gp_page_refcount": (I32, [P, I32, PI32]),
        "gp_free_page_count": (I32, [P, PI32]),
        "gp_slot_acquire": (I32, [P, PI32]),
        "gp_slot_release": (I32, [P, I32]),
        "gp_update_summaries": (I32, [P, I32, P, P, P]),
        "gp_boundary_demand": (I32, [P, I32, C.POINTER(GpRequest), P, C.POINTER(GpDemand)]),
        "gp_boundary_demand_noalloc": (I32, [P, I32, C.POINTER(GpRequest), P, C.POINTER(GpDemand), P]),
        "gp_decide": (I32, [P, I32, C.POINTER(GpRequest), C.POINTER(GpDemand), C.POINTER(GpAction)]),
        "gp_grow_page": (I32, [P, C.POINTER(GpRequest)]),
        "gp_compress_hold": (I32, [P, I32, C.POINTER(GpRequest)]),
        "gp_shrink": (I32, [P, I32, C.POINTER(GpRequest)]),
        "gp_compress_fill": (I32, [P, I32, C.POINTER(GpRequest)]),
        "gp_compact_kv": (I32, [P, I32, C.POINTER(GpRequest), P]),
        "gp_debug_demand_k": (I32, [P, I32, P]),
        "gp_debug_entropy": (I32, [P, I32, P]),
        "gp_debug_scores": (I32, [P, I32, P]),
        "gp_debug_probs": (I32, [P, I32, P]),
        "gp_debug_keep_mask": (I32, [P, I32, P]),
        "gp_read_summaries": (I32, [P, I32, P]),
        "gp_set_scan_kernel": (I32, [P, I32]),
        "gp_debug_attention_plan": (I32, [P, I32, P, I32, I32, P, P, P]),
        "gp_set_timing": (I32, [P, I32]),
        "gp_kernel_time": (I32, [P, I32, C.POINTER(C.c_double), C.POINTER(I64)]),
        "gp_reset_timing": (I32, [P]),
        "gp_stats": (I32, [P, C.POINTER(GpStats)]),
        "gp_set_compaction_stream": (I32, [P, P]),
        "gp_wait_compaction": (I32, [P, P]),
        "gp_decode_attention": (I32, [P, I32, I32, C.POINTER(GpRequest), P, P, P, P]),
        "gp_synchronize": (I32, [P]),
        "gp_debug_set_wait_limit": (I32, [P, I32, I64]),
        "gp_debug_fail_next_launch": (I32, [P, I32]),
        "gp_set_selection_mode": (I32, [P, I32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(ctx, st: int):
    if st != GP_OK:
        lib = load()
        msg = lib.gp_last_error(ctx).decode() if ctx else lib.gp_status_string(st).decode()
        raise GrowPageError(st, msg or lib.gp_status_string(st).decode())


def _ptr(t) -> int:
    """Device (or host) address of a tensor / numpy array, or 0."""
    if t is None:
        return 0
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return int(t)


# ---------------------------------------------------------------------------
# requests
# ---------------------------------------------------------------------------

class Request:
    """A request as the scheduler holds it: slot, block table (host), position."""

    def __init__(self, slot: int, pages, pos: int, capacity: int):
        self.slot = int(slot)
        self.table = np.zeros(capacity, dtype=np.int32)
        pages = list(pages)
        self.table[:len(pages)] = pages
        self.num_pages = len(pages)
        self.pos = int(pos)

    @property
    def table(self):
        return self._table

    @table.setter
    def table(self, t):
        self._table = np.ascontiguousarray(t, dtype=np.int32)
        self._bt = self._table.ctypes.data  # the C side reads and extends it in place

    @property
    def pages(self):
        return self.table[:self.num_pages].tolist()


# gp_request as a numpy record, so that a call's requests are marshalled one
# field at a time instead of one ctypes attribute at a time
_REQ_DTYPE = np.dtype({"names": ["slot", "num_pages", "block_table", "pos"],
                       "formats": [np.int32, np.int32, np.uint64, np.int64],
                       "offsets": [GpRequest.slot.offset, GpRequest.num_pages.offset,
                                   GpRequest.block_table.offset, GpRequest.pos.offset],
                       "itemsize": C.sizeof(GpRequest)})


# gp_request packed field by field: {int32 slot, int32 num_pages, pointer
# block_table, int64 pos}, checked against the ctypes layout at import.
_REQ_PACK = struct.Struct("=iiQq")
assert (_REQ_PACK.size == C.sizeof(GpRequest) and GpRequest.slot.offset == 0 and GpRequest.num_pages.offset == 4
        and GpRequest.block_table.offset == 8 and GpRequest.pos.offset == 16), "gp_request layout"
_NUM_PAGES = struct.Struct("=i")


def _marshal(reqs):
    arr = (GpRequest * max(1, len(reqs)))()
    pack, size = _REQ_PACK.pack_into, _REQ_PACK.size
    for i, r in enumerate(reqs):
        pack(arr, i * size, r.slot, r.num_pages, r._bt, r.pos)
    return arr


def _unmarshal(arr, reqs):
    if len(reqs) <= 8:
        get, size = _NUM_PAGES.unpack_from, _REQ_PACK.size
        for i, r in enumerate(reqs):
            r.num_pages = get(arr, i * size + 4)[0]
    else:
        counts = np.frombuffer(arr, dtype=_REQ_DTYPE, count=len(reqs))["num_pages"].tolist()
        for r, p in zip(reqs, counts):
            r.num_pages = p


class _Demands(list):
    """gp_boundary_demand's results: gp_demand views into one ctypes array,
    which gp_decide passes on as it is while the list is unchanged."""

    def __init__(self, arr, n):
        super().__init__(arr[i] for i in range(n))
        self._arr = arr

    def __setitem__(self, i, v):
        self._arr = None
        super().__setitem__(i, v)

    def _whole(self, n):
        return self._arr if self._arr is not None and len(self) == n else None


# ---------------------------------------------------------------------------
# C-named wrappers
# ---------------------------------------------------------------------------

def gp_config_default(**overrides) -> GpConfig:
    cfg = GpConfig()
    _check(None, load().gp_config_default(C.byref(cfg)))
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def gp_create(cfg: GpConfig, k_cache=None, v_cache=None, stream=None):
    ctx = C.c_void_p()
    s = 0 if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    st = load().gp_create(C.byref(cfg), _ptr(k_cache) or None, _ptr(v_cache) or None, s or None, C.byref(ctx))
    _check(None, st)
    return ctx


def gp_destroy(ctx):
    _check(None, load().gp_destroy(ctx))


def gp_page_alloc(ctx) -> int:
    p = C.c_int32()
    _check(ctx, load().gp_page_alloc(ctx, C.byref(p)))
    return p.value


def gp_page_ref(ctx, page: int):
    _check(ctx, load().gp_page_ref(ctx, page))


def gp_page_unref(ctx, page: int):
    _check(ctx, load().gp_page_unref(ctx, page))


def gp_page_refcount(ctx, page: int) -> int:
    rc = C.c_int32()
    _check(ctx, load().gp_page_refcount(ctx, page, C.byref(rc)))
    return rc.value


def gp_free_page_count(ctx) -> int:
    n = C.c_int32()
    _check(ctx, load().gp_free_page_count(ctx, C.byref(n)))
    return n.value


def gp_slot_acquire(ctx) -> int:
    s = C.c_int32()
    _check(ctx, load().gp_slot_acquire(ctx, C.byref(s)))
    return s.value


def gp_slot_release(ctx, slot: int):
    _check(ctx, load().gp_slot_release(ctx, slot))


def gp_update_summaries(ctx, n: int, slots_dev, q_dev, first_dev):
    _check(ctx, load().gp_update_summaries(ctx, n, _ptr(slots_dev), _ptr(q_dev), _ptr(first_dev)))


def gp_boundary_demand(ctx, reqs, q_cur_dev):
    arr = _marshal(reqs)
    out = (GpDemand * max(1, len(reqs)))()
    _check(ctx, load().gp_boundary_demand(ctx, len(reqs), arr, _ptr(q_cur_dev), out))
    return _Demands(out, len(reqs))


def gp_boundary_demand_noalloc(ctx, reqs, q_cur_dev, k_units=None):
    """No-allocation variant; k_units (host int32 [n][L*Hkv][2]) is optional."""
    arr = _marshal(reqs)
    out = (GpDemand * max(1, len(reqs)))()
    _check(ctx, load().gp_boundary_demand_noalloc(ctx, len(reqs), arr, _ptr(q_cur_dev), out,
                                                  _ptr(k_units) or None))
    return [out[i] for i in range(len(reqs))]


def gp_decide(ctx, reqs, demand):
    arr = _marshal(reqs)
    dem = demand._whole(len(reqs)) if isinstance(demand, _Demands) else None
    if dem is None:
        dem = (GpDemand * max(1, len(reqs)))(*demand)
    out = (GpAction * max(1, len(reqs)))()
    _check(ctx, load().gp_decide(ctx, len(reqs), arr, dem, out))
    return [out[i] for i in range(len(reqs))]


def gp_grow_page(ctx, req: Request):
    if req.num_pages >= len(req.table):
        raise GrowPageError(GP_ERR_INVALID, "block table is full (Python capacity)")
    arr = _marshal([req])
    st = load().gp_grow_page(ctx, arr)
    _unmarshal(arr, [req])
    _check(ctx, st)


def gp_compress_hold(ctx, reqs):
    arr = _marshal(reqs)
    st = load().gp_compress_hold(ctx, len(reqs), arr)
    _unmarshal(arr, reqs)
    _check(ctx, st)


def gp_shrink(ctx, reqs):
    arr = _marshal(reqs)
    st = load().gp_shrink(ctx, len(reqs), arr)
    _unmarshal(arr, reqs)
    _check(ctx, st)


def gp_compress_fill(ctx, reqs):
    arr = _marshal(reqs)
    st = load().gp_compress_fill(ctx, len(reqs), arr)
    _unmarshal(arr, reqs)
    _check(ctx, st)


def _stream_ptr(stream):
    if stream is None:
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def gp_set_compaction_stream(ctx, stream):
    _check(ctx, load().gp_set_compaction_stream(ctx, _stream_ptr(stream)))


def gp_wait_compaction(ctx, stream=None):
    _check(ctx, load().gp_wait_compaction(ctx, _stream_ptr(stream)))


def gp_decode_attention(ctx, layer: int, reqs, num_tokens, q_dev, first_dev, out_dev):
    """One layer of decode attention with the summary update fused in.
    num_tokens: host int32 per request; q_dev [n][Hq][d]; out_dev fp32 [n][Hq][d]."""
    arr = _marshal(reqs)
    nt = np.ascontiguousarray(np.asarray(num_tokens, dtype=np.int32))
    _check(ctx, load().gp_decode_attention(ctx, layer, len(reqs), arr, nt.ctypes.data, _ptr(q_dev),
                                           _ptr(first_dev), _ptr(out_dev)))


def gp_compact_kv(ctx, reqs, keep_masks_dev):
    arr = _marshal(reqs)
    st = load().gp_compact_kv(ctx, len(reqs), arr, _ptr(keep_masks_dev))
    _unmarshal(arr, reqs)
    _check(ctx, st)


def gp_debug_demand_k(ctx, req_idx: int, units: int) -> np.ndarray:
    out = np.zeros((units, 2), dtype=np.int32)
    _check(ctx, load().gp_debug_demand_k(ctx, req_idx, out.ctypes.data))
    return out


def gp_debug_entropy(ctx, req_idx: int, units: int) -> np.ndarray:
    out = np.zeros((units, 2), dtype=np.float64)
    _check(ctx, load().gp_debug_entropy(ctx, req_idx, out.ctypes.data))
    return out


def gp_debug_scores(ctx, req_idx: int, units: int, ncmp: int) -> np.ndarray:
    out = np.zeros((units, ncmp), dtype=np.float32)
    _check(ctx, load().gp_debug_scores(ctx, req_idx, out.ctypes.data))
    return out


def gp_debug_probs(ctx, req_idx: int, units: int, ndem: int) -> np.ndarray:
    out = np.zeros((units, 2, ndem), dtype=np.float32)
    _check(ctx, load().gp_debug_probs(ctx, req_idx, out.ctypes.data))
    return out


def gp_debug_keep_mask(ctx, req_idx: int, units: int, num_pages: int, page_size: int = 256) -> np.ndarray:
    out = np.zeros((units, num_pages * page_size // 32), dtype=np.uint32)
    _check(ctx, load().gp_debug_keep_mask(ctx, req_idx, out.ctypes.data))
    return out


def gp_read_summaries(ctx, slot: int, L: int, hq: int, d: int) -> np.ndarray:
    out = np.zeros((L, 2, hq, d), dtype=np.float64)
    _check(ctx, load().gp_read_summaries(ctx, slot, out.ctypes.data))
    return out



def gp_debug_attention_plan(ctx, num_tokens, sms: int) -> np.ndarray:
    """The tensor-core attention kernel's work items for these token counts on
    `sms` SMs (host only): int32 [items][8] rows (request, KV head, piece,
    pieces, first page, tiles, first item of the pair, CTA)."""
    nt = np.ascontiguousarray(np.asarray(num_tokens, dtype=np.int32))
    n_items, n_ctas = C.c_int32(0), C.c_int32(0)
    lib = load()
    lib.gp_debug_attention_plan(ctx, len(nt), nt.ctypes.data, int(sms), 0, None, C.byref(n_items), C.byref(n_ctas))
    out = np.zeros((max(n_items.value, 1), 8), dtype=np.int32)
    _check(ctx, lib.gp_debug_attention_plan(ctx, len(nt), nt.ctypes.data, int(sms), out.shape[0], out.ctypes.data,
                                            C.byref(n_items), C.byref(n_ctas)))
    return out[:n_items.value]


def gp_set_scan_kernel(ctx, kind: int):
    _check(ctx, load().gp_set_scan_kernel(ctx, int(kind)))


def gp_set_selection_mode(ctx, mode: int):
    _check(ctx, load().gp_set_selection_mode(ctx, int(mode)))


def gp_set_timing(ctx, enabled: bool):
    _check(ctx, load().gp_set_timing(ctx, int(bool(enabled))))


def gp_kernel_time(ctx, kernel: int):
    ms, n = C.c_double(), C.c_int64()
    _check(ctx, load().gp_kernel_time(ctx, kernel, C.byref(ms), C.byref(n)))
    return ms.value, n.value


def gp_reset_timing(ctx):
    _check(ctx, load().gp_reset_timing(ctx))


def gp_synchronize(ctx):
    """Wait for all engine work; raise on device-side errors of earlier calls."""
    _check(ctx, load().gp_synchronize(ctx))


def gp_debug_set_wait_limit(ctx, kernel: int, cycles: int):
    _check(ctx, load().gp_debug_set_wait_limit(ctx, int(kernel), int(cycles)))


def gp_debug_fail_next_launch(ctx, kernel: int):
    _check(ctx, load().gp_debug_fail_next_launch(ctx, int(kernel)))


def gp_stats(ctx) -> dict:
    s = GpStats()
    _check(ctx, load().gp_stats(ctx, C.byref(s)))
    return {n: getattr(s, n) for n, _ in GpStats._fields_}


@dataclass
class Shape:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int

    @property
    def units(self) -> int:
        return self.num_layers * self.num_kv_heads


def unpack_mask(words: np.ndarray, n: int) -> np.ndarray:
    """uint32 keep-mask words -> bool[..., n] (bit i%32 of word i/32)."""
    w = np.asarray(words, dtype=np.uint32)
    bits = ((w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)
    return bits.reshape(*w.shape[:-1], -1)[..., :n]


def pack_mask(keep: np.ndarray) -> np.ndarray:
    """bool[..., n] (n a multiple of 32) -> uint32 words."""
    k = np.asarray(keep, dtype=bool)
    k = k.reshape(*k.shape[:-1], -1, 32).astype(np.uint32)
    return (k << np.arange(32, dtype=np.uint32)).sum(axis=-1).astype(np.uint32)
