// Host side of the GrowPage capacity-boundary engine: the C ABI declared in
// include/growpage.h.  Owns the page pool (refcounts, lowest-id-first free
// set), the summary slots, the device scratch and the orchestration of the
// sm_103a kernels.  Every device step runs in the kernels; this file only
// validates, plans, uploads descriptors and reads back results.
#include "growpage.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <tuple>
#include <unordered_set>
#include <vector>

#include "gp_internal.h"
#include "attn_kernels.h"
#include "gp_kernels.h"

namespace {

constexpr int kPage = 256;
constexpr int kMaxPagesPerReq = 256;

struct DevBuf {
  void* p = nullptr;
  size_t cap = 0;
};

struct DemandRec {
  int32_t slot = -1;
  int32_t num_pages = 0;
  std::vector<int32_t> pages;
  uint64_t gen = 0;
  int64_t score_off = 0;
  int64_t aval_off = 0;
  int64_t spec_off = -1;  // word offset of its speculative keep masks, -1 if none
};

struct CompressRec {
  bool spec = false;      // masks in the speculative buffer (at mask_off), else in `masks`
  int32_t num_pages = 0;
  int64_t mask_off = 0;
};

struct TimedEvent {
  int kernel;
  cudaEvent_t start, stop;
};

}  // namespace

struct gp_ctx {
  gp_config cfg{};
  bool host_only = true;
  void* k_cache = nullptr;
  void* v_cache = nullptr;
  cudaStream_t stream = nullptr;
  std::string err;

  // page pool (Sec. 4.2, App. E.2)
  std::vector<int32_t> refcnt;
  std::set<int32_t> free_pages;
  // summary slots (App. E.1)
  std::vector<uint8_t> slot_bound;
  std::vector<uint64_t> slot_gen;
  std::set<int32_t> free_slots;

  // device state
  double* pool = nullptr;          // [L][M][2][Hq][D]
  int* err_dev = nullptr;          // kernel error bits
  unsigned long long* moved_dev = nullptr;
  DevBuf upload, bt2, qt, bq, scores, aval, tickets, kout, ksum, masks, xstat, attn, spec_masks, ent;
  DevBuf upload_attn;              // decode attention's own descriptors (it may overlap a compaction)
  // speculative selection: the Eq. 10 keep masks of every request of the last
  // demand call, computed on an engine-owned stream while the host decides
  cudaStream_t sel_stream = nullptr;
  cudaEvent_t ev_dem = nullptr, ev_sel = nullptr;
  bool sel_pending = false;
  double* inv_freq = nullptr;      // [D/2] theta^(-2i/D) for RoPE
  CUtensorMap kmap;                // K cache as a 2-D bf16 tensor (tensor-core scan and attention)
  CUtensorMap vmap;                // V cache the same way (tensor-core attention)
  bool tc_ok = false;              // kmap is valid
  bool attn_tc_ok = false;         // kmap and vmap are valid
  int sms = 152;                   // SMs of the device
  int scan_kernel = GP_SCAN_AUTO;
  int select_mode = GP_SELECT_AUTO;
  int64_t spec_units_max = 4 * 152;  // AUTO: speculative selection up to this many units per call
  void* pinned = nullptr;
  size_t pinned_cap = 0;
  cudaEvent_t pinned_free = nullptr;  // recorded after the last async use of `pinned`
  void* readback = nullptr;           // pinned: a demand call's sums and error word
  size_t readback_cap = 0;
  // asynchronous compaction: a side stream, the event the side stream waits
  // for (engine stream state), and the event of the last compaction there
  cudaStream_t cstream = nullptr;
  cudaEvent_t ev_ready = nullptr, ev_done = nullptr;
  bool compaction_pending = false;
  std::unordered_set<int32_t> pending_pages;  // old and new pages of the pending compaction

  std::vector<DemandRec> last_demand;
  std::vector<CompressRec> last_compress;

  gp_stats_t stats{};
  int64_t decisions = 0;           // decisions taken so far (index of the RANDOM policy's draws)
  bool timing = false;
  std::vector<TimedEvent> timed;
  std::vector<cudaEvent_t> event_pool;
  double t_ms[GP_KERNEL_COUNT] = {};
  int64_t t_count[GP_KERNEL_COUNT] = {};
  // test hooks: the copy-wait limit of the selection / compaction launches,
  // and a launch to fail without running (-1: none)
  long long wait_limit_select = gp::kDefaultWaitLimit;
  long long wait_limit_compress = gp::kDefaultWaitLimit;
  int inject_fail = -1;
};

namespace {

gp_status fail(gp_ctx* c, gp_status st, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    c->err = buf;
  }
  return st;
}

#define GP_CUDA(ctx, call)                                                              \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail((ctx), GP_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

int elt_bytes(int dtype) { return dtype == GP_DTYPE_F32 ? 4 : 2; }

gp_status ensure(gp_ctx* c, DevBuf& b, size_t bytes) {
  if (bytes <= b.cap) return GP_OK;
  size_t cap = std::max(bytes, b.cap + b.cap / 2);
  cap = (cap + 255) & ~size_t(255);
  if (b.p) GP_CUDA(c, cudaFree(b.p));
  b.p = nullptr;
  b.cap = 0;
  GP_CUDA(c, cudaMalloc(&b.p, cap));
  b.cap = cap;
  return GP_OK;
}

gp_status ensure_pinned(gp_ctx* c, size_t bytes) {
  if (c->pinned_free) GP_CUDA(c, cudaEventSynchronize(c->pinned_free));
  if (bytes <= c->pinned_cap) return GP_OK;
  size_t cap = std::max(bytes, c->pinned_cap * 2);
  cap = (cap + 4095) & ~size_t(4095);
  if (c->pinned) GP_CUDA(c, cudaFreeHost(c->pinned));
  c->pinned = nullptr;
  c->pinned_cap = 0;
  GP_CUDA(c, cudaHostAlloc(&c->pinned, cap, cudaHostAllocDefault));
  c->pinned_cap = cap;
  return GP_OK;
}

// The pinned readback buffer; a demand call reads it only after
// synchronising the stream, so no copy into it is still in flight here.
gp_status ensure_readback(gp_ctx* c, size_t bytes) {
  if (bytes <= c->readback_cap) return GP_OK;
  size_t cap = std::max<size_t>(std::max(bytes, c->readback_cap * 2), 4096);
  cap = (cap + 4095) & ~size_t(4095);
  if (c->readback) GP_CUDA(c, cudaFreeHost(c->readback));
  c->readback = nullptr;
  c->readback_cap = 0;
  GP_CUDA(c, cudaHostAlloc(&c->readback, cap, cudaHostAllocDefault));
  c->readback_cap = cap;
  return GP_OK;
}

cudaEvent_t take_event(gp_ctx* c) {
  if (!c->event_pool.empty()) {
    cudaEvent_t e = c->event_pool.back();
    c->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Launch wrapper: brackets the launch with events when timing is on.
template <typename F>
gp_status timed_launch_on(gp_ctx* c, cudaStream_t s, int kernel, const char* name, F&& launch) {
  if (c->inject_fail == kernel) {  // test hook: fail as a launch failure would, without running
    c->inject_fail = -1;
    return fail(c, GP_ERR_CUDA, "%s launch failed: injected failure (test hook)", name);
  }
  cudaEvent_t a = nullptr, b = nullptr;
  if (c->timing) {
    a = take_event(c);
    b = take_event(c);
    cudaEventRecord(a, s);
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) return fail(c, GP_ERR_CUDA, "%s launch failed: %s", name, cudaGetErrorString(e));
  if (c->timing) {
    cudaEventRecord(b, s);
    c->timed.push_back({kernel, a, b});
  }
  return GP_OK;
}

template <typename F>
gp_status timed_launch(gp_ctx* c, int kernel, const char* name, F&& launch) {
  return timed_launch_on(c, c->stream, kernel, name, std::forward<F>(launch));
}

// Waits (host) for a speculative selection still running: it reads the
// importance cache and writes the speculative masks, which the next demand
// call rewrites.
gp_status join_select(gp_ctx* c) {
  if (c->sel_pending) {
    GP_CUDA(c, cudaEventSynchronize(c->ev_sel));
    c->sel_pending = false;
  }
  return GP_OK;
}

// Waits (host) for a compaction still running on the side stream: its K/V
// writes, its reads of the engine's scratch (tables, importance, masks) and
// its statistics must be done before the engine reuses, regrows or reads
// any of them.
gp_status join_compaction(gp_ctx* c) {
  if (c->compaction_pending) {
    GP_CUDA(c, cudaEventSynchronize(c->ev_done));
    c->compaction_pending = false;
    c->pending_pages.clear();
  }
  return GP_OK;
}

gp_status need_device(gp_ctx* c) {
  if (!c) return GP_ERR_INVALID;
  if (c->host_only) return fail(c, GP_ERR_STATE, "host-only context has no device caches");
  return GP_OK;
}

// Read and clear the kernels' error word (synchronises the stream).  A word
// holding only ERR_TIMEOUT (bounded waits gave up) is GP_ERR_TIMEOUT; any
// failed device-side check makes it GP_ERR_INVALID.
gp_status kernel_error_status(gp_ctx* c, int e);

gp_status check_kernel_errors(gp_ctx* c) {
  int e = 0;
  GP_CUDA(c, cudaMemcpyAsync(&e, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  return kernel_error_status(c, e);
}

// The status of an error word already read (the stream synchronised); a
// non-zero word is cleared on the device.
gp_status kernel_error_status(gp_ctx* c, int e) {
  if (e) {
    GP_CUDA(c, cudaMemsetAsync(c->err_dev, 0, sizeof(int), c->stream));
    GP_CUDA(c, cudaStreamSynchronize(c->stream));
    return fail(c, gp::status_of_kernel_error(e),
                "device-side error (bits 0x%x: 1 slot, 2 page, 4 keep mask count, 8 selection, 16 wait timed out)",
                e);
  }
  return GP_OK;
}

gp_status validate_request(gp_ctx* c, const gp_request& r, int idx, bool need_slot) {
  const gp_config& g = c->cfg;
  if (need_slot && (r.slot < 0 || r.slot >= g.max_slots || !c->slot_bound[r.slot]))
    return fail(c, GP_ERR_INVALID, "request %d: slot %d is not bound", idx, r.slot);
  if (r.num_pages < 1 || r.num_pages > g.max_pages_per_req)
    return fail(c, GP_ERR_INVALID, "request %d: num_pages %d outside [1, %d]", idx, r.num_pages,
                g.max_pages_per_req);
  if (!r.block_table) return fail(c, GP_ERR_INVALID, "request %d: null block table", idx);
  if (r.pos < 0) return fail(c, GP_ERR_INVALID, "request %d: negative position", idx);
  std::unordered_set<int32_t> seen;
  for (int j = 0; j < r.num_pages; ++j) {
    const int32_t pg = r.block_table[j];
    if (pg < 0 || pg >= g.num_pages || c->refcnt[pg] <= 0)
      return fail(c, GP_ERR_INVALID, "request %d: block %d holds page %d that is not allocated", idx, j, pg);
    if (!seen.insert(pg).second)
      return fail(c, GP_ERR_INVALID, "request %d: page %d appears twice in the block table", idx, pg);
  }
  return GP_OK;
}

int units_of(const gp_ctx* c) { return c->cfg.num_layers * c->cfg.num_kv_heads; }

// Tensor map of the K (or V) cache for the tensor-core kernels: a 2-D bf16 tensor of
// rows = L * num_pages * Hkv * b keys by d elements, copied in boxes of
// 64 elements x 128 keys with the 128-byte swizzle the MMA descriptors use.
// False (and the CUDA-core kernels are used) when the cache is not bf16, its
// base is not 16-byte aligned, or the row count does not fit a coordinate.
bool make_map(gp_ctx* c, void* cache, CUtensorMap* map) {
  const gp_config& g = c->cfg;
  if (g.kv_dtype != GP_DTYPE_BF16) return false;
  if (reinterpret_cast<uintptr_t>(cache) & 15u) return false;
  const uint64_t rows = (uint64_t)g.num_layers * (uint64_t)g.num_pages * (uint64_t)g.num_kv_heads * kPage;
  if (rows + 128 >= (1ull << 31)) return false;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  cuuint64_t dims[2] = {(cuuint64_t)g.head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)g.head_dim * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cache, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Work of the tensor-core attention kernel (persistent, one CTA per SM):
// every (request, KV head) pair's attended pages laid end to end and cut
// into one even range of W pages per SM; a CTA takes the items of its range
// -- whole pairs, and at most two pieces of pairs it shares with its
// neighbours, whose partials the last piece to finish merges.  A pair's
// first piece can be a single page at the end of a range, so W >= (longest
// pair - 1) / 63 keeps every pair within 64 pieces.  A pair with no attended
// token still gets an item (its summary update and zero output).  Even
// ranges balance equal pairs that a per-pair split cannot (16 requests of
// 128 pages over 152 SMs: 90.1 % of HBM with one item per SM of whole or
// halved pairs).  Fills everything but bt_off, slot and pos; cta_begin gets
// the first item of each CTA and the item count.
void attention_plan(int n, const int32_t* num_tokens, int Hkv, int sms, std::vector<gp::AttnItem>& items,
                    std::vector<int32_t>& cta_begin) {
  items.clear();
  cta_begin.clear();
  long long total_pages = 0;
  int max_npg = 0;
  for (int r = 0; r < n; ++r) {
    const int npg = (num_tokens[r] + kPage - 1) / kPage;
    total_pages += npg;
    max_npg = std::max(max_npg, npg);
  }
  const long long total = total_pages * Hkv;
  const long long W = std::max({1LL, (total + sms - 1) / sms, (long long)(max_npg + 61) / 63});
  long long room = W;  // pages left in the current CTA's range
  cta_begin.push_back(0);
  for (int r = 0; r < n; ++r) {
    const int npg = (num_tokens[r] + kPage - 1) / kPage;
    for (int h = 0; h < Hkv; ++h) {
      const int first = (int)items.size();
      int p0 = 0, split = 0;
      do {
        if (room == 0 && npg > p0) {  // the range is full: the next CTA's range starts here
          cta_begin.push_back((int32_t)items.size());
          room = W;
        }
        const int take = (int)std::min<long long>(npg - p0, room);
        const int span = std::min(num_tokens[r] - p0 * kPage, take * kPage);
        gp::AttnItem it{};
        it.r = r;
        it.h = h;
        it.split = split++;
        it.part_first = first;
        it.p0 = p0;
        it.T = span > 0 ? (span + 127) / 128 : 0;
        it.ntok = num_tokens[r];
        items.push_back(it);
        p0 += take;
        room -= take;
      } while (p0 < npg);
      for (size_t k = first; k < items.size(); ++k) items[k].nsp = split;
    }
  }
  cta_begin.push_back((int32_t)items.size());
}

}  // namespace

// The C linkage of every gp_* definition below comes from its declaration
// in growpage.h.

const char* gp_status_string(gp_status st) {
  switch (st) {
    case GP_OK: return "ok";
    case GP_ERR_INVALID: return "invalid argument";
    case GP_ERR_NO_PAGES: return "no free pages";
    case GP_ERR_NO_SLOTS: return "no free slots";
    case GP_ERR_CUDA: return "CUDA error";
    case GP_ERR_TIMEOUT: return "device wait timed out";
    case GP_ERR_STATE: return "invalid state";
    case GP_ERR_UNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

gp_status gp_config_default(gp_config* cfg) {
  if (!cfg) return GP_ERR_INVALID;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->page_size = kPage;
  cfg->kv_dtype = GP_DTYPE_BF16;
  cfg->q_dtype = GP_DTYPE_BF16;
  cfg->max_slots = 512;
  cfg->max_pages_per_req = 128;
  cfg->recent_window = 16;
  cfg->k_loc = 64;
  cfg->reserve_pages = 0;
  cfg->policy = GP_POLICY_GROWPAGE;
  cfg->beta_s = 0.9;
  cfg->beta_l = 0.999;
  cfg->p = 0.99;
  cfg->tau = 0.0;
  cfg->rope_theta = 10000.0;
  cfg->random_compress = 0.7;
  cfg->shrink_threshold = -0.005;
  cfg->shrink_floor_pages = 4;  // 1024 tokens
  cfg->random_seed = 0u;
  cfg->demand_metric = GP_METRIC_TOP_P;
  return GP_OK;
}

gp_status gp_create(const gp_config* cfg, void* k_cache, void* v_cache, void* stream, gp_ctx** out) {
  if (!cfg || !out) return GP_ERR_INVALID;
  *out = nullptr;
  const gp_config& g = *cfg;
  if (g.num_layers < 1 || g.num_q_heads < 1 || g.num_kv_heads < 1 || g.num_q_heads % g.num_kv_heads)
    return GP_ERR_INVALID;
  if (g.page_size != kPage) return GP_ERR_UNSUPPORTED;
  if (g.head_dim != 64 && g.head_dim != 128) return GP_ERR_UNSUPPORTED;
  const int G = g.num_q_heads / g.num_kv_heads;
  if (G != 2 && G != 4) return GP_ERR_UNSUPPORTED;
  if ((g.kv_dtype != GP_DTYPE_BF16 && g.kv_dtype != GP_DTYPE_F32) ||
      (g.q_dtype != GP_DTYPE_BF16 && g.q_dtype != GP_DTYPE_F32))
    return GP_ERR_INVALID;
  if (g.max_slots < 1 || g.num_pages < 1 || g.max_pages_per_req < 1) return GP_ERR_INVALID;
  if (g.max_pages_per_req > kMaxPagesPerReq) return GP_ERR_UNSUPPORTED;
  if (g.recent_window < 0 || g.recent_window >= kPage || g.k_loc < 0 || g.reserve_pages < 0)
    return GP_ERR_INVALID;
  if (g.policy < GP_POLICY_GROWPAGE || g.policy > GP_POLICY_SHRINK) return GP_ERR_INVALID;
  if (g.demand_metric != GP_METRIC_TOP_P && g.demand_metric != GP_METRIC_ENTROPY) return GP_ERR_INVALID;
  if (!(g.random_compress >= 0.0 && g.random_compress <= 1.0) || !std::isfinite(g.shrink_threshold) ||
      g.shrink_floor_pages < 2)
    return GP_ERR_INVALID;
  if (!(g.p > 0.0 && g.p < 1.0) || !(g.beta_s >= 0.0 && g.beta_s < 1.0) ||
      !(g.beta_l >= 0.0 && g.beta_l < 1.0) || !(g.rope_theta > 0.0) || !std::isfinite(g.tau))
    return GP_ERR_INVALID;
  if ((k_cache == nullptr) != (v_cache == nullptr)) return GP_ERR_INVALID;

  gp_ctx* c = new gp_ctx();
  c->cfg = g;
  c->host_only = (k_cache == nullptr);
  c->k_cache = k_cache;
  c->v_cache = v_cache;
  c->stream = static_cast<cudaStream_t>(stream);
  c->refcnt.assign(g.num_pages, 0);
  for (int i = 0; i < g.num_pages; ++i) c->free_pages.insert(i);
  c->slot_bound.assign(g.max_slots, 0);
  c->slot_gen.assign(g.max_slots, 0);
  for (int i = 0; i < g.max_slots; ++i) c->free_slots.insert(i);
  if (!c->host_only) {
    const size_t pool_bytes =
        sizeof(double) * (size_t)g.num_layers * g.max_slots * 2 * g.num_q_heads * g.head_dim;
    cudaError_t e = cudaMalloc((void**)&c->pool, pool_bytes);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->pool, 0, pool_bytes, c->stream);
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->err_dev, 64);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->err_dev, 0, 64, c->stream);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->pinned_free, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->sel_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_dem, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_sel, cudaEventDisableTiming);
    // RoPE inverse frequencies theta^(-2i/d), computed once in fp64
    std::vector<double> inv(g.head_dim / 2);
    for (int i = 0; i < g.head_dim / 2; ++i) inv[i] = std::pow(g.rope_theta, -2.0 * i / g.head_dim);
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->inv_freq, sizeof(double) * inv.size());
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(c->inv_freq, inv.data(), sizeof(double) * inv.size(), cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
      gp_destroy(c);
      return GP_ERR_CUDA;
    }
    c->moved_dev = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(c->err_dev) + 8);
    c->tc_ok = make_map(c, c->k_cache, &c->kmap);
    c->attn_tc_ok = c->tc_ok && make_map(c, c->v_cache, &c->vmap);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
      c->spec_units_max = 4 * (int64_t)sms;
      c->sms = sms;
    }
  }
  *out = c;
  return GP_OK;
}

gp_status gp_destroy(gp_ctx* c) {
  if (!c) return GP_ERR_INVALID;
  if (!c->host_only) {
    join_compaction(c);
    cudaStreamSynchronize(c->stream);
    if (c->sel_stream) {
      cudaStreamSynchronize(c->sel_stream);
      cudaStreamDestroy(c->sel_stream);
    }
    if (c->ev_dem) cudaEventDestroy(c->ev_dem);
    if (c->ev_sel) cudaEventDestroy(c->ev_sel);
    if (c->ev_ready) cudaEventDestroy(c->ev_ready);
    if (c->ev_done) cudaEventDestroy(c->ev_done);
    for (DevBuf* b : {&c->upload, &c->bt2, &c->qt, &c->bq, &c->scores, &c->aval, &c->tickets, &c->kout, &c->ksum, &c->ent,
                      &c->masks, &c->xstat, &c->attn, &c->spec_masks, &c->upload_attn})
      if (b->p) cudaFree(b->p);
    if (c->inv_freq) cudaFree(c->inv_freq);
    if (c->pool) cudaFree(c->pool);
    if (c->err_dev) cudaFree(c->err_dev);
    if (c->pinned) cudaFreeHost(c->pinned);
    if (c->readback) cudaFreeHost(c->readback);
    if (c->pinned_free) cudaEventDestroy(c->pinned_free);
    for (auto& t : c->timed) {
      cudaEventDestroy(t.start);
      cudaEventDestroy(t.stop);
    }
    for (auto e : c->event_pool) cudaEventDestroy(e);
  }
  delete c;
  return GP_OK;
}

const char* gp_last_error(const gp_ctx* c) { return c ? c->err.c_str() : "null context"; }

// ---- page pool ----------------------------------------------------------------

gp_status gp_page_alloc(gp_ctx* c, int32_t* page) {
  if (!c || !page) return GP_ERR_INVALID;
  if (c->free_pages.empty()) return fail(c, GP_ERR_NO_PAGES, "no free pages");
  const int32_t p = *c->free_pages.begin();
  c->free_pages.erase(c->free_pages.begin());
  c->refcnt[p] = 1;
  *page = p;
  return GP_OK;
}

gp_status gp_page_ref(gp_ctx* c, int32_t page) {
  if (!c) return GP_ERR_INVALID;
  if (page < 0 || page >= c->cfg.num_pages || c->refcnt[page] <= 0)
    return fail(c, GP_ERR_INVALID, "ref of page %d that is not allocated", page);
  ++c->refcnt[page];
  return GP_OK;
}

gp_status gp_page_unref(gp_ctx* c, int32_t page) {
  if (!c) return GP_ERR_INVALID;
  if (page < 0 || page >= c->cfg.num_pages || c->refcnt[page] <= 0)
    return fail(c, GP_ERR_INVALID, "unref of page %d that is not allocated", page);
  if (--c->refcnt[page] == 0) c->free_pages.insert(page);
  return GP_OK;
}

gp_status gp_page_refcount(const gp_ctx* c, int32_t page, int32_t* rc) {
  if (!c || !rc || page < 0 || page >= c->cfg.num_pages) return GP_ERR_INVALID;
  *rc = c->refcnt[page];
  return GP_OK;
}

gp_status gp_free_page_count(const gp_ctx* c, int32_t* n) {
  if (!c || !n) return GP_ERR_INVALID;
  *n = (int32_t)c->free_pages.size();
  return GP_OK;
}

// ---- slots --------------------------------------------------------------------

gp_status gp_slot_acquire(gp_ctx* c, int32_t* slot) {
  if (!c || !slot) return GP_ERR_INVALID;
  if (c->free_slots.empty()) return fail(c, GP_ERR_NO_SLOTS, "no free summary slots");
  const int32_t s = *c->free_slots.begin();
  c->free_slots.erase(c->free_slots.begin());
  c->slot_bound[s] = 1;
  ++c->slot_gen[s];
  *slot = s;
  return GP_OK;
}

gp_status gp_slot_release(gp_ctx* c, int32_t slot) {
  if (!c) return GP_ERR_INVALID;
  if (slot < 0 || slot >= c->cfg.max_slots || !c->slot_bound[slot])
    return fail(c, GP_ERR_INVALID, "release of slot %d that is not bound", slot);
  c->slot_bound[slot] = 0;
  ++c->slot_gen[slot];
  c->free_slots.insert(slot);
  return GP_OK;
}

// ---- hot path ---------------------------------------------------------------

gp_status gp_update_summaries(gp_ctx* c, int32_t n, const int32_t* slots_dev, const void* q_dev,
                              const uint8_t* first_dev) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if (n < 0 || n > c->cfg.max_slots) return fail(c, GP_ERR_INVALID, "n = %d outside [0, max_slots]", n);
  if (n == 0) return GP_OK;
  if (!slots_dev || !q_dev || !first_dev) return fail(c, GP_ERR_INVALID, "null device pointer");
  const gp_config& g = c->cfg;
  gp::EmaArgs a{};
  a.pool = c->pool;
  a.q = q_dev;
  a.q_f32 = g.q_dtype == GP_DTYPE_F32;
  a.slots = slots_dev;
  a.first = first_dev;
  a.n = n;
  a.L = g.num_layers;
  a.Hq = g.num_q_heads;
  a.D = g.head_dim;
  a.M = g.max_slots;
  a.beta_s = g.beta_s;
  a.beta_l = g.beta_l;
  a.err = c->err_dev;
  return timed_launch(c, GP_KERNEL_EMA, "ema_update", [&] { return gp::launch_ema(a, c->stream); });
}

namespace {

struct Staged {
  DevBuf* dev;   // the device mirror the descriptors are uploaded to
  gp::DevReq* reqs;
  int32_t* bt;
  int32_t* bt_new;
  int32_t* work;
  int32_t* part_base;
  int32_t* sel;  // requests of a demand call that get a speculative selection
  void* extra;   // a call's own table (decode attention: its work items)
  size_t bytes;
  size_t off_bt, off_bt_new, off_work, off_pb, off_sel, off_extra;
};

// Pinned layout [DevReq n][bt n*maxP][bt_new n*maxP][work n][part_base n+1]
// [sel n][extra bytes], mirrored in `dev` (the engine's upload buffer unless
// another is given).
gp_status stage(gp_ctx* c, int n, bool with_new, Staged* s, DevBuf* dev = nullptr, size_t extra = 0) {
  s->dev = dev ? dev : &c->upload;
  const int maxp = c->cfg.max_pages_per_req;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 255) & ~size_t(255); return r; };
  const size_t off_req = take(sizeof(gp::DevReq) * n);
  s->off_bt = take(sizeof(int32_t) * (size_t)n * maxp);
  s->off_bt_new = with_new ? take(sizeof(int32_t) * (size_t)n * maxp) : s->off_bt;
  s->off_work = take(sizeof(int32_t) * n);
  s->off_pb = take(sizeof(int32_t) * (n + 1));
  s->off_sel = take(sizeof(int32_t) * n);
  s->off_extra = take(extra);
  s->bytes = o;
  gp_status st = ensure_pinned(c, o);
  if (st != GP_OK) return st;
  st = ensure(c, *s->dev, o);
  if (st != GP_OK) return st;
  char* p = static_cast<char*>(c->pinned);
  s->reqs = reinterpret_cast<gp::DevReq*>(p + off_req);
  s->bt = reinterpret_cast<int32_t*>(p + s->off_bt);
  s->bt_new = reinterpret_cast<int32_t*>(p + s->off_bt_new);
  s->work = reinterpret_cast<int32_t*>(p + s->off_work);
  s->part_base = reinterpret_cast<int32_t*>(p + s->off_pb);
  s->sel = reinterpret_cast<int32_t*>(p + s->off_sel);
  s->extra = p + s->off_extra;
  return GP_OK;
}

gp_status upload(gp_ctx* c, const Staged& s) {
  GP_CUDA(c, cudaMemcpyAsync(s.dev->p, c->pinned, s.bytes, cudaMemcpyHostToDevice, c->stream));
  GP_CUDA(c, cudaEventRecord(c->pinned_free, c->stream));
  return GP_OK;
}

template <typename T>
T* dev_at(const Staged& s, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(s.dev->p) + off);
}

}  // namespace

gp_status gp_boundary_demand(gp_ctx* c, int32_t n, const gp_request* reqs, const void* q_cur_dev,
                             gp_demand* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if ((st = join_select(c)) != GP_OK) return st;
  if (n < 0 || n > c->cfg.max_slots) return fail(c, GP_ERR_INVALID, "n = %d outside [0, max_slots]", n);
  if (n == 0) return GP_OK;
  if (!reqs || !out || !q_cur_dev) return fail(c, GP_ERR_INVALID, "null argument");
  const gp_config& g = c->cfg;
  std::unordered_set<int32_t> slots;
  for (int r = 0; r < n; ++r) {
    st = validate_request(c, reqs[r], r, true);
    if (st != GP_OK) return st;
    if (!slots.insert(reqs[r].slot).second)
      return fail(c, GP_ERR_INVALID, "slot %d appears twice in one call", reqs[r].slot);
  }
  const int units = units_of(c);
  const int G = g.num_q_heads / g.num_kv_heads;
  const int rows = 2 * G;
  const int maxp = g.max_pages_per_req;

  // offsets of the importance cache and the a-values
  std::vector<int64_t> score_off(n), aval_off(n);
  int64_t score_total = 0, aval_total = 0;
  for (int r = 0; r < n; ++r) {
    const int P = reqs[r].num_pages;
    score_off[r] = score_total;
    score_total += (int64_t)units * (P * kPage - g.recent_window);
    aval_off[r] = aval_total;
    aval_total += (int64_t)units * 2 * (P - 1) * kPage;
  }
  // Eq. 10 selection: speculatively, right after the demand kernels on the
  // selection stream, where it hides behind the host's decision when the call
  // is small; for calls of many units, inside the compaction launch, where
  // the copies of other units' CTAs keep HBM busy while a CTA selects.
  int64_t cand_units = 0;
  for (int r = 0; r < n; ++r)
    if (reqs[r].num_pages >= 2) cand_units += units;
  const bool speculate = c->select_mode == GP_SELECT_SPECULATIVE ||
                         (c->select_mode == GP_SELECT_AUTO && cand_units <= c->spec_units_max);
  // speculative keep masks: every request that Compress & Hold could take
  std::vector<int64_t> spec_off(n, -1);
  int64_t spec_total = 0;
  for (int r = 0; r < n; ++r) {
    if (!speculate || reqs[r].num_pages < 2) continue;
    spec_off[r] = spec_total;
    spec_total += (int64_t)units * (reqs[r].num_pages * kPage / 32);
  }
  if ((st = ensure(c, c->spec_masks, sizeof(uint32_t) * (size_t)std::max<int64_t>(spec_total, 1))) != GP_OK)
    return st;
  Staged s{};
  st = stage(c, n, false, &s);
  if (st != GP_OK) return st;
  if ((st = ensure(c, c->qt, sizeof(float) * (size_t)n * units * rows * g.head_dim)) != GP_OK) return st;
  if ((st = ensure(c, c->bq, gp::bq_bytes(g.head_dim, G) * (size_t)n * units)) != GP_OK) return st;
  if ((st = ensure(c, c->scores, sizeof(float) * (size_t)std::max<int64_t>(score_total, 1))) != GP_OK) return st;
  if ((st = ensure(c, c->aval, sizeof(float) * (size_t)std::max<int64_t>(aval_total, 1))) != GP_OK) return st;
  // tickets [n][units] then the tensor-core scan's statistics counts [n][units]
  if ((st = ensure(c, c->tickets, sizeof(unsigned) * 2 * (size_t)n * units)) != GP_OK) return st;
  if ((st = ensure(c, c->xstat, sizeof(float2) * (size_t)n * units * gp::TC_MAX_PARTS * 16)) != GP_OK) return st;
  if ((st = ensure(c, c->kout, sizeof(int32_t) * (size_t)n * units * 2)) != GP_OK) return st;
  if ((st = ensure(c, c->ksum, sizeof(unsigned long long) * (size_t)n * 2)) != GP_OK) return st;

  // work: the tensor-core requests first (one launch, split into parts),
  // then the CUDA-core requests in buckets of equal cluster size C (one
  // launch each; a bucket's ppc bounds the pages any CTA of it scores)
  const bool tc = c->tc_ok && c->scan_kernel != GP_SCAN_CUDA_CORE;
  std::vector<int32_t> tc_work;
  std::map<int, std::vector<int32_t>> buckets;
  std::map<int, int> bucket_ppc;
  for (int r = 0; r < n; ++r) {
    const gp::DemandPlan pl = gp::demand_plan(reqs[r].num_pages, tc);
    if (c->scan_kernel == GP_SCAN_TENSOR_CORE && pl.variant != gp::DEMAND_TC)
      return fail(c, GP_ERR_UNSUPPORTED, "request %d: the tensor-core scan needs a bf16 cache and at most %d pages",
                  r, gp::TC_MAX_PAGES);
    if (pl.variant == gp::DEMAND_TC) {
      tc_work.push_back(r);
    } else {
      buckets[pl.C].push_back(r);
      int& mp = bucket_ppc[pl.C];
      mp = std::max(mp, pl.ppc);
    }
  }
  for (int r = 0; r < n; ++r) {
    gp::DevReq& d = s.reqs[r];
    d.num_pages = reqs[r].num_pages;
    d.slot = reqs[r].slot;
    d.pos = reqs[r].pos;
    d.score_off = score_off[r];
    d.aval_off = aval_off[r];
    d.mask_off = std::max<int64_t>(spec_off[r], 0);
    d.bt_off = r * maxp;
    d.pad = 0;
    std::memcpy(s.bt + (size_t)r * maxp, reqs[r].block_table, sizeof(int32_t) * reqs[r].num_pages);
  }
  struct Launch {
    int variant, C, ppc, first, count;
  };
  std::vector<Launch> launches;
  int wpos = 0;
  int n_parts = 0;
  s.part_base[0] = 0;
  if (!tc_work.empty()) {
    launches.push_back({gp::DEMAND_TC, 1, gp::TC_MAX_PPC, 0, (int)tc_work.size()});
    for (int32_t r : tc_work) {
      s.work[wpos++] = r;
      n_parts += units * gp::tc_parts(reqs[r].num_pages);
      s.part_base[wpos] = n_parts;
    }
  }
  for (auto it = buckets.rbegin(); it != buckets.rend(); ++it) {  // largest clusters first
    launches.push_back({gp::DEMAND_FFMA, it->first, bucket_ppc[it->first], wpos, (int)it->second.size()});
    for (int32_t r : it->second) s.work[wpos++] = r;
  }
  int n_sel = 0;
  for (int r = 0; r < n; ++r)
    if (spec_off[r] >= 0) s.sel[n_sel++] = r;
  if ((st = upload(c, s)) != GP_OK) return st;

  gp::PrepArgs pa{};
  pa.pool = c->pool;
  pa.q = q_cur_dev;
  pa.q_f32 = g.q_dtype == GP_DTYPE_F32;
  pa.reqs = dev_at<gp::DevReq>(s, 0);
  pa.n = n;
  pa.L = g.num_layers;
  pa.Hq = g.num_q_heads;
  pa.Hkv = g.num_kv_heads;
  pa.D = g.head_dim;
  pa.M = g.max_slots;
  pa.inv_freq = c->inv_freq;
  pa.qt = static_cast<float*>(c->qt.p);
  pa.bq = static_cast<unsigned char*>(c->bq.p);
  pa.err = c->err_dev;
  pa.zero32 = static_cast<unsigned*>(c->tickets.p);   // tickets and statistics counts
  pa.n_zero32 = 2 * (size_t)n * units;
  pa.zero64 = static_cast<unsigned long long*>(c->ksum.p);
  pa.n_zero64 = n * 2;
  st = timed_launch(c, GP_KERNEL_PREP, "prep_queries", [&] { return gp::launch_prep(pa, c->stream); });
  if (st != GP_OK) return st;

  for (const Launch& l : launches) {
    gp::DemandArgs da{};
    da.kmap = c->kmap;
    da.variant = l.variant;
    da.k_cache = c->k_cache;
    da.kv_f32 = g.kv_dtype == GP_DTYPE_F32;
    da.num_pages_total = g.num_pages;
    da.L = g.num_layers;
    da.Hkv = g.num_kv_heads;
    da.D = g.head_dim;
    da.G = G;
    da.b = kPage;
    da.R = g.recent_window;
    da.pfix = gp::coverage_fraction(g.p);
    da.qt = pa.qt;
    da.bq = pa.bq;
    da.reqs = pa.reqs;
    da.bt = dev_at<int32_t>(s, s.off_bt);
    da.work = dev_at<int32_t>(s, s.off_work) + l.first;
    da.n_work = l.count;
    da.C = l.C;
    da.ppc = l.ppc;
    da.part_base = dev_at<int32_t>(s, s.off_pb);
    da.n_parts = n_parts;
    da.xstat = static_cast<float2*>(c->xstat.p);
    da.xcount = static_cast<unsigned*>(c->tickets.p) + (size_t)n * units;
    da.scores = static_cast<float*>(c->scores.p);
    da.aval = static_cast<float*>(c->aval.p);
    da.tickets = static_cast<unsigned*>(c->tickets.p);
    da.kout = static_cast<int32_t*>(c->kout.p);
    da.ksum = static_cast<unsigned long long*>(c->ksum.p);
    da.err = c->err_dev;
    st = timed_launch(c, GP_KERNEL_DEMAND, "boundary_demand", [&] { return gp::launch_demand(da, c->stream); });
    if (st != GP_OK) return st;
  }
  // Speculative selection: the Eq. 10 keep masks of every request that could
  // be compressed, on the engine's selection stream, while the host reads
  // the sums and decides.  A Compress & Hold of these requests then only
  // moves rows.
  if (n_sel > 0) {
    GP_CUDA(c, cudaEventRecord(c->ev_dem, c->stream));
    GP_CUDA(c, cudaStreamWaitEvent(c->sel_stream, c->ev_dem, 0));
    gp::CompressArgs ca{};
    ca.k_cache = c->k_cache;
    ca.v_cache = c->v_cache;
    ca.num_pages_total = g.num_pages;
    ca.L = g.num_layers;
    ca.Hkv = g.num_kv_heads;
    ca.D = g.head_dim;
    ca.elt = elt_bytes(g.kv_dtype);
    ca.b = kPage;
    ca.R = g.recent_window;
    ca.k_loc = g.k_loc;
    ca.drop = 1;
    ca.fill = 0;
    ca.select_only = 1;
    ca.reqs = pa.reqs;
    ca.old_bt = dev_at<int32_t>(s, s.off_bt);
    ca.new_bt = ca.old_bt;
    ca.scores = static_cast<const float*>(c->scores.p);
    ca.keep_in = nullptr;
    ca.keep_out = static_cast<uint32_t*>(c->spec_masks.p);
    ca.work = dev_at<int32_t>(s, s.off_sel);
    ca.n_work = n_sel;
    ca.moved = c->moved_dev;
    ca.err = c->err_dev;
    ca.wait_limit = c->wait_limit_select;
    st = timed_launch_on(c, c->sel_stream, GP_KERNEL_SELECT, "select",
                         [&] { return gp::launch_compress(ca, c->sel_stream); });
    if (st != GP_OK) return st;
    GP_CUDA(c, cudaEventRecord(c->ev_sel, c->sel_stream));
    c->sel_pending = true;
  }
  // the entropy metric (Sec. 5.3 ablation): exp(H(a^x)) per unit from the a-values
  const bool entropy = g.demand_metric == GP_METRIC_ENTROPY;
  std::vector<double> eff(entropy ? (size_t)n * units * 2 : 0);
  if (entropy) {
    if ((st = ensure(c, c->ent, sizeof(double) * eff.size())) != GP_OK) return st;
    gp::EntropyArgs ea{};
    ea.reqs = pa.reqs;
    ea.aval = static_cast<const float*>(c->aval.p);
    ea.n = n;
    ea.units = units;
    ea.b = kPage;
    ea.out = static_cast<double*>(c->ent.p);
    st = timed_launch(c, GP_KERNEL_ENTROPY, "entropy", [&] { return gp::launch_entropy(ea, c->stream); });
    if (st != GP_OK) return st;
    GP_CUDA(c, cudaMemcpyAsync(eff.data(), c->ent.p, sizeof(double) * eff.size(), cudaMemcpyDeviceToHost,
                               c->stream));
  }
  // the sums and the error word in one pinned buffer, read after one
  // synchronisation
  const size_t sum_bytes = sizeof(unsigned long long) * (size_t)n * 2;
  if ((st = ensure_readback(c, sum_bytes + 16)) != GP_OK) return st;
  const unsigned long long* sums = static_cast<const unsigned long long*>(c->readback);
  int* err_host = reinterpret_cast<int*>(static_cast<char*>(c->readback) + sum_bytes);
  GP_CUDA(c, cudaMemcpyAsync(c->readback, c->ksum.p, sum_bytes, cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaMemcpyAsync(err_host, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  if ((st = kernel_error_status(c, *err_host)) != GP_OK) return st;

  c->last_demand.assign(n, DemandRec{});
  for (int r = 0; r < n; ++r) {
    const int P = reqs[r].num_pages;
    gp_demand& o = out[r];
    o.sum_k_short = (int64_t)sums[2 * r];
    o.sum_k_long = (int64_t)sums[2 * r + 1];
    o.num_candidates = (P - 1) * kPage;
    o.num_units = units;
    o.delta = o.num_candidates > 0
                  ? (double)(o.sum_k_short - o.sum_k_long) / ((double)o.num_candidates * units)
                  : 0.0;
    o.eff_short = 0.0;
    o.eff_long = 0.0;
    if (entropy) {
      for (int u = 0; u < units; ++u) {  // unit order: the same sum on every call
        o.eff_short += eff[((size_t)r * units + u) * 2];
        o.eff_long += eff[((size_t)r * units + u) * 2 + 1];
      }
      o.delta = o.num_candidates > 0 ? (o.eff_short - o.eff_long) / ((double)o.num_candidates * units) : 0.0;
    }
    DemandRec& rec = c->last_demand[r];
    rec.slot = reqs[r].slot;
    rec.num_pages = P;
    rec.pages.assign(reqs[r].block_table, reqs[r].block_table + P);
    rec.gen = c->slot_gen[reqs[r].slot];
    rec.score_off = score_off[r];
    rec.aval_off = aval_off[r];
    rec.spec_off = spec_off[r];
  }
  c->stats.demand_calls += 1;
  c->stats.demand_requests += n;
  return GP_OK;
}

namespace {

// SplitMix64 output function (Steele, Lea and Flood, OOPSLA 2014): the
// state x advanced by the golden-ratio increment, then mixed.
uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Uniform draw in [0, 1) of the k-th decision of a context.
double policy_draw(uint32_t seed, int64_t k) {
  const uint64_t v = splitmix64(((uint64_t)seed << 32) + (uint64_t)k);
  return (double)(v >> 11) * (1.0 / 9007199254740992.0);  // 2^-53
}

}  // namespace

gp_status gp_decide(gp_ctx* c, int32_t n, const gp_request* reqs, const gp_demand* demand, gp_action* out) {
  if (!c) return GP_ERR_INVALID;
  if (n < 0) return fail(c, GP_ERR_INVALID, "negative n");
  if (n > 0 && (!reqs || !demand || !out)) return fail(c, GP_ERR_INVALID, "null argument");
  const gp_config& g = c->cfg;
  for (int r = 0; r < n; ++r)
    if (reqs[r].num_pages < 1) return fail(c, GP_ERR_INVALID, "request %d: num_pages %d", r, reqs[r].num_pages);
  int64_t free_now = (int64_t)c->free_pages.size();
  int64_t granted = 0;
  for (int r = 0; r < n; ++r) {
    const int P = reqs[r].num_pages;
    gp_action a{GP_ACT_COMPRESS, 0, 0};
    const int64_t k = c->decisions++;
    if (P == 1) {
      a.kind = GP_ACT_GROW;
      a.forced = 1;
    } else {
      const double units = (double)demand[r].num_units;
      const double cand = (double)demand[r].num_candidates;
      const int64_t diff = demand[r].sum_k_short - demand[r].sum_k_long;
      const bool entropy = g.demand_metric == GP_METRIC_ENTROPY;
      const double delta = entropy ? (demand[r].eff_short - demand[r].eff_long) / (cand * units)
                                   : (double)diff / (cand * units);
      // Delta > tau; for D_p and tau = 0 the exact integer test
      const bool above_tau = (g.tau == 0.0 && !entropy) ? diff > 0 : delta > g.tau;
      bool want = false, shrink = false;
      switch (g.policy) {
        case GP_POLICY_GROWPAGE: want = above_tau; break;
        case GP_POLICY_FIXED: want = false; break;
        case GP_POLICY_RANDOM: want = !(policy_draw(g.random_seed, k) < g.random_compress); break;
        case GP_POLICY_INVERSE: want = !above_tau; break;
        case GP_POLICY_SHRINK:
          want = above_tau;
          shrink = !want && delta < g.shrink_threshold && P > g.shrink_floor_pages;
          break;
        default: break;
      }
      if (want) {
        if (free_now - granted > (int64_t)g.reserve_pages) {
          a.kind = GP_ACT_GROW;
          ++granted;
        } else {
          a.kind = GP_ACT_COMPRESS;
          a.fallback = 1;
        }
      } else if (shrink) {
        a.kind = GP_ACT_SHRINK;
      }
    }
    out[r] = a;
    if (a.kind == GP_ACT_GROW) {
      c->stats.grow += 1;
      if (a.forced) c->stats.forced_grow += 1;
    } else if (a.kind == GP_ACT_SHRINK) {
      c->stats.shrink += 1;
    } else {
      c->stats.compress += 1;
      if (a.fallback) c->stats.fallback += 1;
    }
  }
  return GP_OK;
}

gp_status gp_grow_page(gp_ctx* c, gp_request* req) {
  if (!c || !req) return GP_ERR_INVALID;
  if (!req->block_table) return fail(c, GP_ERR_INVALID, "null block table");
  if (req->num_pages < 0 || req->num_pages >= c->cfg.max_pages_per_req)
    return fail(c, GP_ERR_INVALID, "block table is full (%d pages)", req->num_pages);
  int32_t page = -1;
  gp_status st = gp_page_alloc(c, &page);
  if (st != GP_OK) return st;
  req->block_table[req->num_pages] = page;
  req->num_pages += 1;
  if (req->slot >= 0 && req->slot < c->cfg.max_slots) ++c->slot_gen[req->slot];
  return GP_OK;
}

namespace {

// Shared path of gp_compress_hold (keep_in == null) and gp_compact_kv.
// drop: pages' worth of history dropped per (layer, KV head): 1 for Compress &
// Hold, 2 for Shrink (which then returns the emptied last page).
// fill: hole-fill compaction (order-destroying) instead of the stable one.
gp_status compress_common(gp_ctx* c, int32_t n, gp_request* reqs, const uint32_t* keep_in, int drop, int fill = 0) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  // the speculative selection reads the upload buffer this call rewrites
  if ((st = join_select(c)) != GP_OK) return st;
  if (n < 0 || n > c->cfg.max_slots) return fail(c, GP_ERR_INVALID, "n = %d outside [0, max_slots]", n);
  if (n == 0) return GP_OK;
  if (!reqs) return fail(c, GP_ERR_INVALID, "null requests");
  const gp_config& g = c->cfg;
  const int units = units_of(c);
  const int maxp = g.max_pages_per_req;
  std::vector<int64_t> score_off(n, 0), spec_off(n, -1);
  std::unordered_set<int32_t> slots;
  for (int r = 0; r < n; ++r) {
    st = validate_request(c, reqs[r], r, keep_in == nullptr);
    if (st != GP_OK) return st;
    if (reqs[r].num_pages < drop + 1)
      return fail(c, GP_ERR_INVALID, "request %d: %s needs at least %d pages", r,
                  drop == 1 ? "Compress & Hold" : "Shrink", drop + 1);
    if (keep_in == nullptr) {
      if (!slots.insert(reqs[r].slot).second)
        return fail(c, GP_ERR_INVALID, "slot %d appears twice in one call", reqs[r].slot);
      const DemandRec* rec = nullptr;
      for (const auto& d : c->last_demand)
        if (d.slot == reqs[r].slot) rec = &d;
      if (!rec || rec->gen != c->slot_gen[reqs[r].slot] || rec->num_pages != reqs[r].num_pages ||
          !std::equal(rec->pages.begin(), rec->pages.end(), reqs[r].block_table))
        return fail(c, GP_ERR_STATE,
                    "request %d: no gp_boundary_demand result for its current pages (call it first)", r);
      score_off[r] = rec->score_off;
      spec_off[r] = rec->spec_off;
    }
  }
  // the speculative keep masks of the last demand call serve Compress & Hold
  // (stable or hole fill) when every request has them; Shrink selects anew
  bool spec = keep_in == nullptr && drop == 1;
  for (int r = 0; r < n && spec; ++r) spec = spec_off[r] >= 0;
  // copy-on-write plan (App. E.2): every shared page gets a fresh target page
  size_t need = 0;
  for (int r = 0; r < n; ++r)
    for (int j = 0; j < reqs[r].num_pages; ++j)
      if (c->refcnt[reqs[r].block_table[j]] > 1) ++need;
  if (need > c->free_pages.size())
    return fail(c, GP_ERR_NO_PAGES, "copy-on-write needs %zu fresh pages, %zu free", need,
                c->free_pages.size());

  Staged s{};
  if ((st = stage(c, n, true, &s)) != GP_OK) return st;
  int64_t mask_total = 0;
  std::vector<int64_t> mask_off(n);
  for (int r = 0; r < n; ++r) {
    mask_off[r] = mask_total;
    mask_total += (int64_t)units * (reqs[r].num_pages * kPage / 32);
  }
  if ((st = ensure(c, c->masks, sizeof(uint32_t) * (size_t)mask_total)) != GP_OK) return st;

  // allocate the CoW targets (cannot fail now), lowest id first, ascending logical order
  std::vector<std::vector<int32_t>> replaced(n);
  for (int r = 0; r < n; ++r) {
    gp::DevReq& d = s.reqs[r];
    const int P = reqs[r].num_pages;
    d.num_pages = P;
    d.slot = reqs[r].slot;
    d.pos = reqs[r].pos;
    d.score_off = score_off[r];
    d.aval_off = 0;
    d.mask_off = spec ? spec_off[r] : mask_off[r];
    d.bt_off = r * maxp;
    d.pad = 0;
    for (int j = 0; j < P; ++j) {
      const int32_t pg = reqs[r].block_table[j];
      s.bt[(size_t)r * maxp + j] = pg;
      int32_t tgt = pg;
      if (c->refcnt[pg] > 1) {
        gp_page_alloc(c, &tgt);
        replaced[r].push_back(pg);
      }
      s.bt_new[(size_t)r * maxp + j] = tgt;
    }
    s.work[r] = r;
  }
  if ((st = upload(c, s)) != GP_OK) return st;

  gp::CompressArgs ca{};
  ca.k_cache = c->k_cache;
  ca.v_cache = c->v_cache;
  ca.num_pages_total = g.num_pages;
  ca.L = g.num_layers;
  ca.Hkv = g.num_kv_heads;
  ca.D = g.head_dim;
  ca.elt = elt_bytes(g.kv_dtype);
  ca.b = kPage;
  ca.R = g.recent_window;
  ca.k_loc = g.k_loc;
  ca.drop = drop;
  ca.fill = fill;
  ca.reqs = dev_at<gp::DevReq>(s, 0);
  ca.old_bt = dev_at<int32_t>(s, s.off_bt);
  ca.new_bt = dev_at<int32_t>(s, s.off_bt_new);
  ca.scores = static_cast<const float*>(c->scores.p);
  ca.keep_in = spec ? static_cast<const uint32_t*>(c->spec_masks.p) : keep_in;
  ca.keep_out = spec ? nullptr : static_cast<uint32_t*>(c->masks.p);
  ca.work = dev_at<int32_t>(s, s.off_work);
  ca.n_work = n;
  ca.moved = c->moved_dev;
  ca.err = c->err_dev;
  ca.wait_limit = c->wait_limit_compress;
  // on the side stream (if any), after everything the engine stream holds
  cudaStream_t ks = c->stream;
  if (c->cstream) {
    GP_CUDA(c, cudaEventRecord(c->ev_ready, c->stream));
    GP_CUDA(c, cudaStreamWaitEvent(c->cstream, c->ev_ready, 0));
    ks = c->cstream;
  }
  if (spec) GP_CUDA(c, cudaStreamWaitEvent(ks, c->ev_sel, 0));  // the speculative masks are written (joined above)
  st = timed_launch_on(c, ks, GP_KERNEL_COMPRESS, "compress_hold", [&] { return gp::launch_compress(ca, ks); });
  if (st == GP_OK && c->cstream) {
    GP_CUDA(c, cudaEventRecord(c->ev_done, c->cstream));
    c->compaction_pending = true;
    c->pending_pages.clear();
    for (int r = 0; r < n; ++r)
      for (int j = 0; j < reqs[r].num_pages; ++j) {
        c->pending_pages.insert(s.bt[(size_t)r * maxp + j]);
        c->pending_pages.insert(s.bt_new[(size_t)r * maxp + j]);
      }
  }
  if (st != GP_OK) {
    // roll back the page allocations
    for (int r = 0; r < n; ++r)
      for (int j = 0; j < reqs[r].num_pages; ++j) {
        const int32_t t = s.bt_new[(size_t)r * maxp + j];
        if (t != reqs[r].block_table[j]) gp_page_unref(c, t);
      }
    return st;
  }
  // host bookkeeping: new tables, drop the references to replaced shared pages
  c->last_compress.assign(n, CompressRec{});
  for (int r = 0; r < n; ++r) {
    const int P = reqs[r].num_pages;
    for (int j = 0; j < P; ++j) reqs[r].block_table[j] = s.bt_new[(size_t)r * maxp + j];
    for (int32_t pg : replaced[r]) gp_page_unref(c, pg);
    c->stats.cow_pages += (int64_t)replaced[r].size();
    if (drop == 2) {
      // Shrink: the emptied last page goes back to the pool
      gp_page_unref(c, reqs[r].block_table[P - 1]);
      reqs[r].num_pages = P - 1;
    }
    if (reqs[r].slot >= 0 && reqs[r].slot < g.max_slots) ++c->slot_gen[reqs[r].slot];
    c->last_compress[r].num_pages = P;
    c->last_compress[r].mask_off = spec ? spec_off[r] : mask_off[r];
    c->last_compress[r].spec = spec;
  }
  return GP_OK;
}

}  // namespace

gp_status gp_compress_hold(gp_ctx* c, int32_t n, gp_request* reqs) { return compress_common(c, n, reqs, nullptr, 1); }

gp_status gp_shrink(gp_ctx* c, int32_t n, gp_request* reqs) { return compress_common(c, n, reqs, nullptr, 2); }

gp_status gp_compress_fill(gp_ctx* c, int32_t n, gp_request* reqs) {
  return compress_common(c, n, reqs, nullptr, 1, 1);
}

gp_status gp_compact_kv(gp_ctx* c, int32_t n, gp_request* reqs, const uint32_t* keep_masks_dev) {
  if (!c) return GP_ERR_INVALID;
  if (n > 0 && !keep_masks_dev) return fail(c, GP_ERR_INVALID, "null keep masks");
  return compress_common(c, n, reqs, keep_masks_dev, 1);
}

// ---- inspection --------------------------------------------------------------

gp_status gp_debug_demand_k(gp_ctx* c, int32_t req_idx, int32_t* k_out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (!k_out || req_idx < 0 || req_idx >= (int)c->last_demand.size())
    return fail(c, GP_ERR_INVALID, "no demand result %d", req_idx);
  const int units = units_of(c);
  GP_CUDA(c, cudaMemcpyAsync(k_out, static_cast<int32_t*>(c->kout.p) + (size_t)req_idx * units * 2,
                             sizeof(int32_t) * units * 2, cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  return GP_OK;
}

gp_status gp_debug_entropy(gp_ctx* c, int32_t req_idx, double* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (c->cfg.demand_metric != GP_METRIC_ENTROPY) return fail(c, GP_ERR_STATE, "the demand metric is not ENTROPY");
  if (!out || req_idx < 0 || req_idx >= (int)c->last_demand.size())
    return fail(c, GP_ERR_INVALID, "no demand result %d", req_idx);
  const int units = units_of(c);
  GP_CUDA(c, cudaMemcpyAsync(out, static_cast<double*>(c->ent.p) + (size_t)req_idx * units * 2,
                             sizeof(double) * units * 2, cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  return GP_OK;
}

gp_status gp_debug_scores(gp_ctx* c, int32_t req_idx, float* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (!out || req_idx < 0 || req_idx >= (int)c->last_demand.size())
    return fail(c, GP_ERR_INVALID, "no demand result %d", req_idx);
  const DemandRec& rec = c->last_demand[req_idx];
  const size_t count = (size_t)units_of(c) * (rec.num_pages * kPage - c->cfg.recent_window);
  GP_CUDA(c, cudaMemcpyAsync(out, static_cast<float*>(c->scores.p) + rec.score_off, sizeof(float) * count,
                             cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  return GP_OK;
}

gp_status gp_debug_probs(gp_ctx* c, int32_t req_idx, float* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (!out || req_idx < 0 || req_idx >= (int)c->last_demand.size())
    return fail(c, GP_ERR_INVALID, "no demand result %d", req_idx);
  const DemandRec& rec = c->last_demand[req_idx];
  const size_t count = (size_t)units_of(c) * 2 * (rec.num_pages - 1) * kPage;
  if (count == 0) return GP_OK;
  GP_CUDA(c, cudaMemcpyAsync(out, static_cast<float*>(c->aval.p) + rec.aval_off, sizeof(float) * count,
                             cudaMemcpyDeviceToHost, c->stream));
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  return GP_OK;
}

gp_status gp_debug_keep_mask(gp_ctx* c, int32_t req_idx, uint32_t* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (!out || req_idx < 0 || req_idx >= (int)c->last_compress.size())
    return fail(c, GP_ERR_INVALID, "no compress result %d", req_idx);
  const CompressRec& rec = c->last_compress[req_idx];
  const size_t count = (size_t)units_of(c) * (rec.num_pages * kPage / 32);
  const uint32_t* src = static_cast<const uint32_t*>(rec.spec ? c->spec_masks.p : c->masks.p);
  GP_CUDA(c, cudaMemcpyAsync(out, src + rec.mask_off, sizeof(uint32_t) * count, cudaMemcpyDeviceToHost, c->stream));
  return check_kernel_errors(c);
}

gp_status gp_read_summaries(gp_ctx* c, int32_t slot, double* out) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  const gp_config& g = c->cfg;
  if (!out || slot < 0 || slot >= g.max_slots) return fail(c, GP_ERR_INVALID, "bad slot %d", slot);
  const size_t row = sizeof(double) * 2 * g.num_q_heads * g.head_dim;
  GP_CUDA(c, cudaMemcpy2DAsync(out, row, reinterpret_cast<char*>(c->pool) + row * slot, row * g.max_slots, row,
                               g.num_layers, cudaMemcpyDeviceToHost, c->stream));
  return check_kernel_errors(c);
}

gp_status gp_set_scan_kernel(gp_ctx* c, int32_t kind) {
  if (!c) return GP_ERR_INVALID;
  if (kind != GP_SCAN_AUTO && kind != GP_SCAN_CUDA_CORE && kind != GP_SCAN_TENSOR_CORE)
    return fail(c, GP_ERR_INVALID, "unknown scan kernel %d", kind);
  if (kind == GP_SCAN_TENSOR_CORE && !c->host_only && !c->tc_ok)
    return fail(c, GP_ERR_UNSUPPORTED, "the tensor-core scan needs a 16-byte aligned bf16 K cache");
  c->scan_kernel = kind;
  return GP_OK;
}

gp_status gp_set_selection_mode(gp_ctx* c, int32_t mode) {
  if (!c) return GP_ERR_INVALID;
  if (mode != GP_SELECT_AUTO && mode != GP_SELECT_SPECULATIVE && mode != GP_SELECT_IN_COMPACTION)
    return fail(c, GP_ERR_INVALID, "unknown selection mode %d", mode);
  c->select_mode = mode;
  return GP_OK;
}

gp_status gp_set_timing(gp_ctx* c, int32_t enabled) {
  if (!c) return GP_ERR_INVALID;
  c->timing = enabled != 0;
  return GP_OK;
}

static gp_status resolve_timing(gp_ctx* c) {
  if (c->timed.empty()) return GP_OK;
  GP_CUDA(c, cudaStreamSynchronize(c->stream));
  for (auto& t : c->timed) {
    float ms = 0.f;
    GP_CUDA(c, cudaEventElapsedTime(&ms, t.start, t.stop));
    c->t_ms[t.kernel] += ms;
    c->t_count[t.kernel] += 1;
    c->event_pool.push_back(t.start);
    c->event_pool.push_back(t.stop);
  }
  c->timed.clear();
  return GP_OK;
}

gp_status gp_kernel_time(gp_ctx* c, int32_t kernel, double* ms, int64_t* launches) {
  if (!c || kernel < 0 || kernel >= GP_KERNEL_COUNT || !ms || !launches) return GP_ERR_INVALID;
  gp_status st = resolve_timing(c);
  if (st != GP_OK) return st;
  *ms = c->t_ms[kernel];
  *launches = c->t_count[kernel];
  return GP_OK;
}

gp_status gp_reset_timing(gp_ctx* c) {
  if (!c) return GP_ERR_INVALID;
  gp_status st = resolve_timing(c);
  if (st != GP_OK) return st;
  for (int k = 0; k < GP_KERNEL_COUNT; ++k) {
    c->t_ms[k] = 0.0;
    c->t_count[k] = 0;
  }
  return GP_OK;
}

gp_status gp_synchronize(gp_ctx* c) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if ((st = join_select(c)) != GP_OK) return st;
  return check_kernel_errors(c);  // synchronises the engine stream
}

gp_status gp_debug_attention_plan(gp_ctx* c, int32_t n, const int32_t* num_tokens, int32_t sms, int32_t max_items,
                                  int32_t* items_out, int32_t* n_items, int32_t* n_ctas) {
  if (!c) return GP_ERR_INVALID;
  if (n < 0 || sms < 1 || max_items < 0 || !n_items || !n_ctas || (n > 0 && !num_tokens))
    return fail(c, GP_ERR_INVALID, "gp_debug_attention_plan: bad arguments");
  for (int r = 0; r < n; ++r)
    if (num_tokens[r] < 0 || num_tokens[r] > c->cfg.max_pages_per_req * kPage)
      return fail(c, GP_ERR_INVALID, "request %d: num_tokens %d outside [0, %d]", r, num_tokens[r],
                  c->cfg.max_pages_per_req * kPage);
  std::vector<gp::AttnItem> items;
  std::vector<int32_t> cta_begin;
  attention_plan(n, num_tokens, c->cfg.num_kv_heads, sms, items, cta_begin);
  *n_items = (int32_t)items.size();
  *n_ctas = (int32_t)cta_begin.size() - 1;
  if ((int64_t)items.size() > max_items)
    return fail(c, GP_ERR_INVALID, "gp_debug_attention_plan: %zu items, room for %d", items.size(), max_items);
  for (int cta = 0; cta + 1 < (int)cta_begin.size(); ++cta)
    for (int k = cta_begin[cta]; k < cta_begin[cta + 1]; ++k) {
      const gp::AttnItem& it = items[k];
      int32_t* o = items_out + (size_t)k * 8;
      o[0] = it.r;
      o[1] = it.h;
      o[2] = it.split;
      o[3] = it.nsp;
      o[4] = it.p0;
      o[5] = it.T;
      o[6] = it.part_first;
      o[7] = cta;
    }
  return GP_OK;
}

gp_status gp_debug_set_wait_limit(gp_ctx* c, int32_t kernel, int64_t cycles) {
  if (!c) return GP_ERR_INVALID;
  const long long v = cycles >= 0 ? (long long)cycles : gp::kDefaultWaitLimit;
  if (kernel == GP_KERNEL_COMPRESS) {
    c->wait_limit_compress = v;
  } else if (kernel == GP_KERNEL_SELECT) {
    c->wait_limit_select = v;
  } else {
    return fail(c, GP_ERR_UNSUPPORTED, "kernel %d has no settable wait limit", kernel);
  }
  return GP_OK;
}

gp_status gp_debug_fail_next_launch(gp_ctx* c, int32_t kernel) {
  if (!c) return GP_ERR_INVALID;
  if (kernel < -1 || kernel >= GP_KERNEL_COUNT) return fail(c, GP_ERR_INVALID, "unknown kernel %d", kernel);
  c->inject_fail = kernel;
  return GP_OK;
}

gp_status gp_stats(const gp_ctx* c, gp_stats_t* out) {
  if (!c || !out) return GP_ERR_INVALID;
  *out = c->stats;
  if (!c->host_only) {
    if (c->compaction_pending && cudaEventSynchronize(c->ev_done) != cudaSuccess) return GP_ERR_CUDA;
    unsigned long long moved = 0;
    if (cudaMemcpyAsync(&moved, c->moved_dev, sizeof(moved), cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
        cudaStreamSynchronize(c->stream) != cudaSuccess)
      return GP_ERR_CUDA;
    out->moved_rows = (int64_t)moved;
  }
  return GP_OK;
}


// ---- decode attention with the summary update fused in --------------------------

gp_status gp_decode_attention(gp_ctx* c, int32_t layer, int32_t n, const gp_request* reqs,
                              const int32_t* num_tokens, const void* q_dev, const uint8_t* first_dev,
                              float* out_dev) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  const gp_config& g = c->cfg;
  if (layer < 0 || layer >= g.num_layers) return fail(c, GP_ERR_INVALID, "layer %d", layer);
  if (n < 0 || n > g.max_slots) return fail(c, GP_ERR_INVALID, "n = %d outside [0, max_slots]", n);
  if (n == 0) return GP_OK;
  if (!reqs || !num_tokens || !q_dev || !first_dev || !out_dev) return fail(c, GP_ERR_INVALID, "null argument");
  std::unordered_set<int32_t> slots;
  for (int r = 0; r < n; ++r) {
    if ((st = validate_request(c, reqs[r], r, true)) != GP_OK) return st;
    if (!slots.insert(reqs[r].slot).second) return fail(c, GP_ERR_INVALID, "slot %d appears twice", reqs[r].slot);
    if (num_tokens[r] < 0 || num_tokens[r] > reqs[r].num_pages * kPage)
      return fail(c, GP_ERR_INVALID, "request %d: num_tokens %d outside [0, %d]", r, num_tokens[r],
                  reqs[r].num_pages * kPage);
  }
  // A compaction pending on the side stream (App. E.3) runs on: this call
  // waits for it on the device only if one of its requests holds a page the
  // compaction reads or writes.  The call uploads its descriptors to its own
  // buffer, so neither the compaction nor the speculative selection, which
  // read the engine's upload buffer, is disturbed.
  bool overlap = false;
  if (c->compaction_pending)
    for (int r = 0; r < n && !overlap; ++r)
      for (int j = 0; j < reqs[r].num_pages && !overlap; ++j)
        overlap = c->pending_pages.count(reqs[r].block_table[j]) != 0;
  const int G = g.num_q_heads / g.num_kv_heads;
  // The tensor-core kernel takes bf16 caches with d = 128 and G = 2 or 4
  // (AUTO and TENSOR_CORE); the CUDA-core kernel everything else.
  const bool tc = c->attn_tc_ok && c->scan_kernel != GP_SCAN_CUDA_CORE && gp::attention_tc_shape(g.head_dim, G);
  if (c->scan_kernel == GP_SCAN_TENSOR_CORE && !tc)
    return fail(c, GP_ERR_UNSUPPORTED, "the tensor-core attention kernel cannot take this cache or shape");
  if (overlap) GP_CUDA(c, cudaStreamWaitEvent(c->stream, c->ev_done, 0));
  const int maxp = g.max_pages_per_req;
  const int Hkv = g.num_kv_heads;
  std::vector<int> npg(n), order(n), nsp(n);
  long long total_pages = 0;
  for (int r = 0; r < n; ++r) {
    npg[r] = (num_tokens[r] + kPage - 1) / kPage;
    total_pages += npg[r];
    order[r] = r;
  }
  std::vector<gp::AttnItem> items;
  std::vector<int32_t> cta_begin;
  if (tc) {
    attention_plan(n, num_tokens, Hkv, c->sms, items, cta_begin);
    for (gp::AttnItem& it : items) {
      it.bt_off = it.r * maxp;
      it.slot = reqs[it.r].slot;
      it.pos = reqs[it.r].pos;
    }
  }
  // The CUDA-core kernel runs one CTA per item: splits of about `chunk`
  // attended pages per pair, longest requests first, for about six waves of
  // two CTAs per SM (2, 3, 6, 12 waves gave 69.5, 71.6, 74.0, 73.3 % of HBM
  // on a 64-request decode step).
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return npg[x] > npg[y]; });
  const long long target_ctas = 6LL * 2 * c->sms;
  const long long chunk = std::max(1LL, (total_pages * Hkv + target_ctas - 1) / target_ctas);
  long long n_ctas = 0;
  for (int r = 0; r < n; ++r) {
    nsp[r] = (int)std::max(1LL, std::min(64LL, (npg[r] + chunk - 1) / chunk));
    n_ctas += (long long)nsp[r] * Hkv;
  }
  if (tc) n_ctas = (long long)items.size();
  const size_t part_floats = (size_t)n_ctas * G * (g.head_dim + 2);
  const size_t tick_off = (part_floats * sizeof(float) + 255) & ~size_t(255);
  if ((st = ensure(c, c->attn, tick_off + sizeof(unsigned) * (size_t)n * Hkv)) != GP_OK) return st;
  const size_t items_bytes = sizeof(gp::AttnItem) * items.size();
  Staged s{};
  if ((st = stage(c, n, false, &s, &c->upload_attn, items_bytes + sizeof(int32_t) * cta_begin.size())) != GP_OK)
    return st;
  s.part_base[0] = 0;
  for (int i = 0; i < n; ++i) {
    s.sel[i] = order[i];
    s.part_base[i + 1] = s.part_base[i] + nsp[order[i]] * Hkv;
  }
  if (tc) {
    std::memcpy(s.extra, items.data(), items_bytes);
    std::memcpy(static_cast<char*>(s.extra) + items_bytes, cta_begin.data(), sizeof(int32_t) * cta_begin.size());
  }
  for (int r = 0; r < n; ++r) {
    gp::DevReq& d = s.reqs[r];
    d.num_pages = reqs[r].num_pages;
    d.slot = reqs[r].slot;
    d.pos = reqs[r].pos;
    d.score_off = 0;
    d.aval_off = 0;
    d.mask_off = 0;
    d.bt_off = r * maxp;
    d.pad = 0;
    std::memcpy(s.bt + (size_t)r * maxp, reqs[r].block_table, sizeof(int32_t) * reqs[r].num_pages);
    s.work[r] = num_tokens[r];  // the staged work array carries the token counts here
  }
  if ((st = upload(c, s)) != GP_OK) return st;
  char* base = static_cast<char*>(c->attn.p);
  GP_CUDA(c, cudaMemsetAsync(base + tick_off, 0, sizeof(unsigned) * (size_t)n * g.num_kv_heads, c->stream));
  gp::AttnArgs a{};
  a.tc = tc ? 1 : 0;
  if (tc) {
    a.kmap = c->kmap;
    a.vmap = c->vmap;
  }
  a.k_cache = c->k_cache;
  a.v_cache = c->v_cache;
  a.kv_f32 = g.kv_dtype == GP_DTYPE_F32;
  a.num_pages_total = g.num_pages;
  a.layer = layer;
  a.Hq = g.num_q_heads;
  a.Hkv = g.num_kv_heads;
  a.D = g.head_dim;
  a.G = G;
  a.M = g.max_slots;
  a.reqs = dev_at<gp::DevReq>(s, 0);
  a.bt = dev_at<int32_t>(s, s.off_bt);
  a.ntok = dev_at<int32_t>(s, s.off_work);
  a.q = q_dev;
  a.q_f32 = g.q_dtype == GP_DTYPE_F32;
  a.first = first_dev;
  a.pool = c->pool;
  a.beta_s = g.beta_s;
  a.beta_l = g.beta_l;
  a.inv_freq = c->inv_freq;
  a.out = out_dev;
  a.part = reinterpret_cast<float*>(base);
  a.tickets = reinterpret_cast<unsigned*>(base + tick_off);
  a.split_base = dev_at<int32_t>(s, s.off_pb);
  a.order = dev_at<int32_t>(s, s.off_sel);
  a.n = n;
  a.n_ctas = (int)n_ctas;
  a.grid = tc ? (int)cta_begin.size() - 1 : 0;
  a.items = tc ? dev_at<gp::AttnItem>(s, s.off_extra) : nullptr;
  a.cta_begin = tc ? dev_at<int32_t>(s, s.off_extra + items_bytes) : nullptr;
  a.err = c->err_dev;
  return timed_launch(c, GP_KERNEL_ATTENTION, "decode_attention",
                      [&] { return gp::launch_decode_attention(a, c->stream); });
}

// ---- asynchronous compaction (side stream) ------------------------------------

gp_status gp_set_compaction_stream(gp_ctx* c, void* stream) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if ((st = join_compaction(c)) != GP_OK) return st;
  if (stream && (!c->ev_ready || !c->ev_done)) {
    GP_CUDA(c, cudaEventCreateWithFlags(&c->ev_ready, cudaEventDisableTiming));
    GP_CUDA(c, cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming));
  }
  c->cstream = static_cast<cudaStream_t>(stream);
  return GP_OK;
}

gp_status gp_wait_compaction(gp_ctx* c, void* stream) {
  gp_status st = need_device(c);
  if (st != GP_OK) return st;
  if (c->ev_done) GP_CUDA(c, cudaStreamWaitEvent(stream ? static_cast<cudaStream_t>(stream) : c->stream, c->ev_done, 0));
  return GP_OK;
}

// ---- read-only view for other translation units (gp_internal.h) ------------

namespace gp {

gp_status ctx_join_compaction(gp_ctx* c) { return c ? join_compaction(c) : GP_ERR_INVALID; }

gp_status ctx_join_select(gp_ctx* c) { return c ? join_select(c) : GP_ERR_INVALID; }

gp_status status_of_kernel_error(int bits) {
  if (bits == 0) return GP_OK;
  return (bits & ~ERR_TIMEOUT) == 0 ? GP_ERR_TIMEOUT : GP_ERR_INVALID;
}

void ctx_forget_demand(gp_ctx* c, int slot) {
  if (!c) return;
  for (auto& d : c->last_demand)
    if (d.slot == slot) d.slot = -1;
}

bool ctx_view(const gp_ctx* c, CtxView* out) {
  if (!c || !out) return false;
  out->cfg = &c->cfg;
  out->k_cache = c->k_cache;
  out->v_cache = c->v_cache;
  out->pool = c->pool;
  out->stream = c->stream;
  out->err_dev = c->err_dev;
  out->host_only = c->host_only;
  out->inv_freq = c->inv_freq;
  out->kmap = &c->kmap;
  out->tc_ok = c->tc_ok && c->scan_kernel != GP_SCAN_CUDA_CORE;
  out->scan_kernel = c->scan_kernel;
  return true;
}

bool ctx_slot_bound(const gp_ctx* c, int slot) {
  return c && slot >= 0 && slot < c->cfg.max_slots && c->slot_bound[slot];
}

gp_status ctx_fail(gp_ctx* c, gp_status st, const char* msg) { return fail(c, st, "%s", msg); }

}  // namespace gp
