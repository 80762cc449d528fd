// gp_boundary_demand_noalloc: the demand estimation of gp_boundary_demand for
// callers that must not allocate memory.
//
// A serving process that reserves all of its GPU memory up front (so that no
// request can fail mid-flight on an out-of-memory error, and no cudaMalloc /
// cudaFree stalls the device with an implicit synchronisation) cannot let a
// library grow scratch buffers on demand.  This entry point therefore uses
// only the file-scope device array below for every temporary it needs: the
// request descriptors and block tables, the calibrated summaries and their
// tensor-core operands, the importance values, the a-values and arrival
// tickets of the D_p select, the partial softmax statistics of the
// tensor-core scan, the per-(layer, KV head) D_p and their sums.
// It calls no cudaMalloc, cudaFree, cudaHostAlloc or other allocating routine;
// host-side staging lives in fixed file-scope arrays.  Inputs (the caches,
// the summaries in the engine's pool, the current queries) and outputs (the
// gp_demand results, and optionally the per-unit D_p values) are the
// caller's.
//
// The array is GP_NOALLOC_SCRATCH_BYTES (64 MiB) and every GPU that loads the
// library holds it until the process exits.  Every call shares it (and the
// host staging arrays): calls whose work overlaps on the GPU, or that run on
// several host threads at once, race.  It keeps the last call's contents;
// the D_p sums, tickets and counts that must start at zero are cleared by
// each call.
//
// Set-up: on the first call on a device (with that device current) the
// array's device address is looked up once with cudaGetSymbolAddress and
// cached.  Make that first call before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

#include "gp_internal.h"
#include "gp_kernels.h"
#include "growpage.h"

#define GP_NOALLOC_SCRATCH_BYTES (64ull << 20)
#define GP_NOALLOC_MAX_REQ 512
#define GP_NOALLOC_MAX_DEVICES 64
#define GP_NOALLOC_MAX_PAGES_BITS (1u << 22)   // page ids checked for duplicates

static __device__ __align__(256) unsigned char gp_noalloc_scratch[GP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kPage = 256;

unsigned char* g_scratch_addr[GP_NOALLOC_MAX_DEVICES] = {};
gp::DevReq g_reqs[GP_NOALLOC_MAX_REQ];
int32_t g_work[GP_NOALLOC_MAX_REQ];
int32_t g_part_base[GP_NOALLOC_MAX_REQ + 1];
unsigned long long g_sums[2 * GP_NOALLOC_MAX_REQ];
uint32_t g_seen[GP_NOALLOC_MAX_PAGES_BITS / 32];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

gp_status fail(gp_ctx* c, gp_status st, const char* fmt, long long a = 0, long long b = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b);
  return gp::ctx_fail(c, st, buf);
}

gp_status cuda_fail(gp_ctx* c, const char* what, cudaError_t e) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s failed: %s", what, cudaGetErrorString(e));
  return gp::ctx_fail(c, GP_ERR_CUDA, buf);
}

}  // namespace

gp_status gp_boundary_demand_noalloc(gp_ctx* c, int32_t n, const gp_request* reqs, const void* q_cur_dev,
                                     gp_demand* out, int32_t* k_units) {
  gp::CtxView v{};
  if (!gp::ctx_view(c, &v)) return GP_ERR_INVALID;
  if (v.host_only) return fail(c, GP_ERR_STATE, "host-only context has no device caches");
  const gp_config& g = *v.cfg;
  if (n < 0 || n > g.max_slots || n > GP_NOALLOC_MAX_REQ)
    return fail(c, GP_ERR_INVALID, "n = %lld outside [0, %lld]", n,
                g.max_slots < GP_NOALLOC_MAX_REQ ? g.max_slots : GP_NOALLOC_MAX_REQ);
  if (n == 0) return GP_OK;
  if (!reqs || !out || !q_cur_dev) return fail(c, GP_ERR_INVALID, "null argument");
  if (g.demand_metric != GP_METRIC_TOP_P)
    return fail(c, GP_ERR_UNSUPPORTED, "the entropy metric needs gp_boundary_demand");
  if (g.num_pages > (int)GP_NOALLOC_MAX_PAGES_BITS)
    return fail(c, GP_ERR_UNSUPPORTED, "more than %lld pages", GP_NOALLOC_MAX_PAGES_BITS);

  // ---- validation (no heap: a static bitmap finds repeated pages) ----------
  for (int r = 0; r < n; ++r) {
    const gp_request& q = reqs[r];
    if (!gp::ctx_slot_bound(c, q.slot)) return fail(c, GP_ERR_INVALID, "request %lld: slot %lld is not bound", r, q.slot);
    for (int r2 = 0; r2 < r; ++r2)
      if (reqs[r2].slot == q.slot) return fail(c, GP_ERR_INVALID, "slot %lld appears twice in one call", q.slot);
    if (q.num_pages < 1 || q.num_pages > g.max_pages_per_req)
      return fail(c, GP_ERR_INVALID, "request %lld: num_pages %lld out of range", r, q.num_pages);
    if (!q.block_table || q.pos < 0) return fail(c, GP_ERR_INVALID, "request %lld: null block table or negative position", r);
    gp_status bad = GP_OK;
    int j = 0;
    for (; j < q.num_pages; ++j) {
      const int32_t pg = q.block_table[j];
      int32_t rc = 0;
      if (pg < 0 || pg >= g.num_pages || gp_page_refcount(c, pg, &rc) != GP_OK || rc <= 0) {
        bad = fail(c, GP_ERR_INVALID, "request %lld: page %lld is not allocated", r, pg);
        break;
      }
      if (g_seen[pg >> 5] & (1u << (pg & 31))) {
        bad = fail(c, GP_ERR_INVALID, "request %lld: page %lld appears twice", r, pg);
        break;
      }
      g_seen[pg >> 5] |= 1u << (pg & 31);
    }
    for (int k = 0; k < j; ++k) g_seen[q.block_table[k] >> 5] &= ~(1u << (q.block_table[k] & 31));
    if (bad != GP_OK) return bad;
  }

  {
    // a compaction still running on a side stream writes K/V this call reads;
    // a speculative selection of an earlier gp_boundary_demand may still write
    // the kernel error word this call reads and clears
    gp_status js = gp::ctx_join_compaction(c);
    if (js == GP_OK) js = gp::ctx_join_select(c);
    if (js != GP_OK) return js;
  }

  // ---- scratch layout and its limit ------------------------------------------
  const int units = g.num_layers * g.num_kv_heads;
  const int G = g.num_q_heads / g.num_kv_heads;
  const int maxp = g.max_pages_per_req;
  size_t o = 0;
  const size_t off_req = o;   o = align256(o + sizeof(gp::DevReq) * n);
  const size_t off_bt = o;    o = align256(o + sizeof(int32_t) * (size_t)n * maxp);
  const size_t off_work = o;  o = align256(o + sizeof(int32_t) * n);
  const size_t off_pb = o;    o = align256(o + sizeof(int32_t) * (n + 1));
  const size_t off_xs = o;    o = align256(o + sizeof(float2) * (size_t)n * units * gp::TC_MAX_PARTS * 16);
  const size_t off_qt = o;    o = align256(o + sizeof(float) * (size_t)n * units * 2 * G * g.head_dim);
  const size_t off_bq = o;    o = align256(o + gp::bq_bytes(g.head_dim, G) * (size_t)n * units);
  const size_t off_kout = o;  o = align256(o + sizeof(int32_t) * (size_t)n * units * 2);
  const size_t off_ksum = o;  o = align256(o + sizeof(unsigned long long) * (size_t)n * 2);
  const size_t off_tk = o;    o = align256(o + sizeof(unsigned) * 2 * (size_t)n * units);  // tickets, counts
  // one float region: per request its importance values, then its a-values,
  // each starting on a 256-byte boundary (the D_p select reads a unit's
  // a-values with 16-byte loads and bulk copies; every unit's a-values span a
  // multiple of 256 floats, so aligning the request's start aligns them all)
  const size_t off_sc = o;
  for (int r = 0; r < n; ++r) {
    g_reqs[r].num_pages = reqs[r].num_pages;
    g_reqs[r].slot = reqs[r].slot;
    g_reqs[r].pos = reqs[r].pos;
    g_reqs[r].score_off = (int64_t)((o - off_sc) / sizeof(float));
    o = align256(o + sizeof(float) * (size_t)units * (reqs[r].num_pages * kPage - g.recent_window));
    g_reqs[r].aval_off = (int64_t)((o - off_sc) / sizeof(float));
    if ((g_reqs[r].aval_off * sizeof(float)) % 16 != 0)
      return fail(c, GP_ERR_INVALID, "request %lld: a-value offset %lld is not 16-byte aligned", r,
                  g_reqs[r].aval_off);
    o = align256(o + sizeof(float) * (size_t)units * 2 * (reqs[r].num_pages - 1) * kPage);
    g_reqs[r].mask_off = 0;
    g_reqs[r].bt_off = r * maxp;
    g_reqs[r].pad = 0;
  }
  if (o > GP_NOALLOC_SCRATCH_BYTES)
    return fail(c, GP_ERR_INVALID,
                "this call needs %lld bytes of scratch; the static scratch of gp_boundary_demand_noalloc "
                "holds %lld (use gp_boundary_demand, or fewer / shorter requests per call)",
                (long long)o, (long long)GP_NOALLOC_SCRATCH_BYTES);

  // ---- one-time set-up per device: the array's device address --------------
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(c, "cudaGetDevice", e);
  if (dev < 0 || dev >= GP_NOALLOC_MAX_DEVICES) return fail(c, GP_ERR_UNSUPPORTED, "device ordinal %lld", dev);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, gp_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(c, "cudaGetSymbolAddress", e);
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  unsigned char* base = g_scratch_addr[dev];

  // ---- work, as gp_boundary_demand forms it: the tensor-core requests first
  // (one launch, split into parts), then the CUDA-core requests in buckets of
  // equal cluster size C; a bucket's ppc bounds the pages any CTA scores.
  int bucket_count[17] = {};
  int bucket_ppc[17] = {};
  int n_tc = 0;
  for (int r = 0; r < n; ++r) {
    const gp::DemandPlan pl = gp::demand_plan(reqs[r].num_pages, v.tc_ok);
    if (v.scan_kernel == GP_SCAN_TENSOR_CORE && pl.variant != gp::DEMAND_TC)
      return fail(c, GP_ERR_UNSUPPORTED, "request %lld: the tensor-core scan cannot serve it", r);
    if (pl.variant == gp::DEMAND_TC) {
      ++n_tc;
      continue;
    }
    if (pl.C < 1 || pl.C > 16) return fail(c, GP_ERR_UNSUPPORTED, "request %lld: cluster size %lld", r, pl.C);
    bucket_count[pl.C] += 1;
    if (pl.ppc > bucket_ppc[pl.C]) bucket_ppc[pl.C] = pl.ppc;
  }
  int bucket_start[17];
  int pos = n_tc;
  for (int C = 16; C >= 1; --C) {
    bucket_start[C] = pos;
    pos += bucket_count[C];
  }
  int fill[17];
  memcpy(fill, bucket_start, sizeof(fill));
  int tc_pos = 0, n_parts = 0;
  g_part_base[0] = 0;
  for (int r = 0; r < n; ++r) {
    const gp::DemandPlan pl = gp::demand_plan(reqs[r].num_pages, v.tc_ok);
    if (pl.variant == gp::DEMAND_TC) {
      g_work[tc_pos++] = r;
      n_parts += units * gp::tc_parts(reqs[r].num_pages);
      g_part_base[tc_pos] = n_parts;
    } else {
      g_work[fill[pl.C]++] = r;
    }
  }

  // ---- uploads (from the caller's / static host memory; no staging buffers) --
  cudaStream_t s = v.stream;
  e = cudaMemcpyAsync(base + off_req, g_reqs, sizeof(gp::DevReq) * n, cudaMemcpyHostToDevice, s);
  for (int r = 0; r < n && e == cudaSuccess; ++r)
    e = cudaMemcpyAsync(base + off_bt + sizeof(int32_t) * (size_t)r * maxp, reqs[r].block_table,
                        sizeof(int32_t) * reqs[r].num_pages, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + off_work, g_work, sizeof(int32_t) * n, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + off_pb, g_part_base, sizeof(int32_t) * (n_tc + 1), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(c, "upload", e);

  gp::PrepArgs pa{};
  pa.pool = v.pool;
  pa.q = q_cur_dev;
  pa.q_f32 = g.q_dtype == GP_DTYPE_F32;
  pa.reqs = reinterpret_cast<const gp::DevReq*>(base + off_req);
  pa.n = n;
  pa.L = g.num_layers;
  pa.Hq = g.num_q_heads;
  pa.Hkv = g.num_kv_heads;
  pa.D = g.head_dim;
  pa.M = g.max_slots;
  pa.inv_freq = v.inv_freq;
  pa.qt = reinterpret_cast<float*>(base + off_qt);
  pa.bq = base + off_bq;
  pa.err = v.err_dev;
  pa.zero32 = reinterpret_cast<unsigned*>(base + off_tk);  // tickets and statistics counts
  pa.n_zero32 = 2 * (size_t)n * units;
  pa.zero64 = reinterpret_cast<unsigned long long*>(base + off_ksum);
  pa.n_zero64 = n * 2;
  e = gp::launch_prep(pa, s);
  if (e != cudaSuccess) return cuda_fail(c, "prep_queries launch", e);

  for (int k = 0; k <= 16; ++k) {
    // k = 0: the tensor-core launch; k = C: the CUDA-core bucket of cluster size C
    const int C = k == 0 ? 1 : 17 - k;
    const int count = k == 0 ? n_tc : bucket_count[C];
    if (!count) continue;
    const int var = k == 0 ? gp::DEMAND_TC : gp::DEMAND_FFMA;
    gp::DemandArgs da{};
    if (var == gp::DEMAND_TC) da.kmap = *v.kmap;
    da.variant = var;
    da.k_cache = v.k_cache;
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
    da.bt = reinterpret_cast<const int32_t*>(base + off_bt);
    da.work = reinterpret_cast<const int32_t*>(base + off_work) + (k == 0 ? 0 : bucket_start[C]);
    da.n_work = count;
    da.C = C;
    da.ppc = k == 0 ? gp::TC_MAX_PPC : bucket_ppc[C];
    da.part_base = reinterpret_cast<const int32_t*>(base + off_pb);
    da.n_parts = n_parts;
    da.xstat = reinterpret_cast<float2*>(base + off_xs);
    da.xcount = reinterpret_cast<unsigned*>(base + off_tk) + (size_t)n * units;
    da.scores = reinterpret_cast<float*>(base + off_sc);
    da.aval = reinterpret_cast<float*>(base + off_sc);
    da.tickets = reinterpret_cast<unsigned*>(base + off_tk);
    da.kout = reinterpret_cast<int32_t*>(base + off_kout);
    da.ksum = reinterpret_cast<unsigned long long*>(base + off_ksum);
    da.err = v.err_dev;
    e = gp::launch_demand(da, s);
    if (e != cudaSuccess) return cuda_fail(c, "boundary_demand launch", e);
  }

  // ---- results -------------------------------------------------------------
  int kerr = 0;
  e = cudaMemcpyAsync(g_sums, base + off_ksum, sizeof(unsigned long long) * n * 2, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && k_units)
    e = cudaMemcpyAsync(k_units, base + off_kout, sizeof(int32_t) * (size_t)n * units * 2,
                        cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&kerr, v.err_dev, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(c, "result copy", e);
  if (kerr) {
    e = cudaMemsetAsync(v.err_dev, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(c, "error word reset", e);
    return fail(c, gp::status_of_kernel_error(kerr),
                "device-side error (bits 0x%llx: 1 slot, 2 page, 16 wait timed out)", kerr);
  }
  // the allocating entry point's importance cache for these slots now
  // predates their current queries: a Compress & Hold needs a new
  // gp_boundary_demand (GP_ERR_STATE until then)
  for (int r = 0; r < n; ++r) gp::ctx_forget_demand(c, reqs[r].slot);
  for (int r = 0; r < n; ++r) {
    const int P = reqs[r].num_pages;
    out[r].sum_k_short = (int64_t)g_sums[2 * r];
    out[r].sum_k_long = (int64_t)g_sums[2 * r + 1];
    out[r].num_candidates = (P - 1) * kPage;
    out[r].num_units = units;
    out[r].delta = out[r].num_candidates > 0
                       ? (double)(out[r].sum_k_short - out[r].sum_k_long) /
                             ((double)out[r].num_candidates * units)
                       : 0.0;
    out[r].eff_short = 0.0;
    out[r].eff_long = 0.0;
  }
  return GP_OK;
}
