// Internal interface between the host engine (growpage.cpp) and the sm_103a
// kernels.  Plain structs of device pointers and sizes; no torch types.
#pragma once

#include <cmath>
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace gp {

// Per-request descriptor uploaded for one hot-path call.
struct DevReq {
  int32_t num_pages;   // P
  int32_t slot;        // summary-pool row
  int64_t pos;         // current decode position (RoPE)
  int64_t score_off;   // float offset of the request's importance cache
  int64_t aval_off;    // float offset of its a-values [units][2][(P-1) b]
  int64_t mask_off;    // word offset of its keep masks
  int32_t bt_off;      // offset of its block table in the packed table array
  int32_t pad;
};

// Error bits written by kernels (atomicOr into a device word).
enum : int {
  ERR_BAD_SLOT = 1,
  ERR_BAD_PAGE = 2,
  ERR_BAD_MASK = 4,
  ERR_BAD_COUNT = 8,
  ERR_TIMEOUT = 16,
};

// ---- A1: EMA update -------------------------------------------------------
struct EmaArgs {
  double* pool;            // [L][M][2][Hq][D]
  const void* q;           // [L][n][Hq][D]
  int q_f32;
  const int32_t* slots;    // [n]
  const uint8_t* first;    // [n]
  int n, L, Hq, D, M;
  double beta_s, beta_l;
  int* err;
};
cudaError_t launch_ema(const EmaArgs& a, cudaStream_t s);

// ---- A2: calibration + RoPE of the summaries ------------------------------
struct PrepArgs {
  const double* pool;      // [L][M][2][Hq][D]
  const void* q;           // [L][n][Hq][D] current query
  int q_f32;
  const DevReq* reqs;      // [n]
  int n, L, Hq, Hkv, D, M;
  const double* inv_freq;  // [D/2] theta^(-2i/D)
  float* qt;               // [n][L][Hkv][2G][D], scaled by log2(e)/sqrt(D)
  unsigned char* bq;       // optional tensor-core operand per unit (bq_bytes each)
  int* err;
  // counters the demand launches that follow need at zero (cleared here, so
  // the call needs no separate memset operations)
  unsigned* zero32;        // [n_zero32]
  size_t n_zero32;
  unsigned long long* zero64;  // [n_zero64]
  int n_zero64;
};
// Bytes of the tensor-core B operand of one unit: D/64 swizzle halves of NB
// rows x 128 B, NB = 3 x 2G rounded up to 16 (three bf16 parts per row).
__host__ __device__ inline size_t bq_bytes(int D, int G) { return (size_t)(D / 64) * ((6 * G + 15) / 16 * 16) * 128; }
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);

// ---- A3-A5: score scan, softmax, GQA mean, a-values, importance cache, D_p --
// The coverage level p of D_p (0 < p < 1) as a 64-bit binary fraction,
// floor(p 2^64): the select's target mass is ceil(T f / 2^64) in integers.
inline unsigned long long coverage_fraction(double p) { return (unsigned long long)std::ldexp(p, 64); }

struct DemandArgs {
  CUtensorMap kmap;        // K cache as [rows][D] bf16, box 64 x 128, 128-byte swizzle
  int variant;             // DEMAND_FFMA or DEMAND_TC
  const void* k_cache;     // [L][num_pages][Hkv][b][D]
  int kv_f32;
  int num_pages_total;
  int L, Hkv, D, G;
  int b, R;
  unsigned long long pfix; // coverage p as a binary fraction, floor(p 2^64)
  const float* qt;
  const unsigned char* bq; // tensor-core operand per unit (prep kernel output)
  const DevReq* reqs;
  const int32_t* bt;       // packed block tables
  const int32_t* work;     // request indices handled by this launch
  int n_work;
  int C;                   // CUDA-core scan: cluster size (CTAs per unit)
  int ppc;                 // CUDA-core scan: most pages one CTA scores
  // tensor-core scan: units split into parts (tc_parts), parts numbered in
  // work order; request work[i] owns parts [part_base[i], part_base[i+1])
  const int32_t* part_base;// [n_work + 1]
  int n_parts;
  float2* xstat;           // per unit and part: softmax statistics [n][units][TC_MAX_PARTS][16]
  unsigned* xcount;        // per unit: parts whose statistics are in, zero between calls
  float* scores;           // importance cache, log2 domain
  float* aval;             // a^S, a^L over C_t: per unit [2][(P-1) b]
  unsigned* tickets;       // [n][units] arrival counters, zero between calls
  int32_t* kout;           // D_p per unit: [n][units][2]
  unsigned long long* ksum;// sums over units: [n][2]
  int* err;
};
enum : int { DEMAND_FFMA = 0, DEMAND_TC = 1 };
cudaError_t launch_demand_ffma(const DemandArgs& a, cudaStream_t s);
cudaError_t launch_demand_tc(const DemandArgs& a, cudaStream_t s);
inline cudaError_t launch_demand(const DemandArgs& a, cudaStream_t s) {
  return a.variant == DEMAND_TC ? launch_demand_tc(a, s) : launch_demand_ffma(a, s);
}

// CTAs of the tensor-core demand kernel (head dim D, GQA group G) that the
// current device holds at once (one per SM); 0 if it cannot run.
int demand_tc_resident(int D, int G);

// How a request of P pages is scanned.
//
// Tensor-core variant (bf16 caches, P <= TC_MAX_PAGES, which covers every
// request the engine accepts, max_pages_per_req <= 256): a persistent
// cooperative grid of one CTA per SM.  Each unit (request, layer, KV head)
// is split into tc_parts(P) parts of balanced page ranges, at most
// TC_MAX_PPC pages each (a CTA keeps two parts of logits in TMEM beside its
// accumulator slots); CTA b takes parts b, b + grid, ... of the call's part
// list, which runs in unit order, so every CTA meets its units in
// increasing order and a unit's parts sit on different CTAs.  Within a unit
// the parts are listed from a rotating start, so the larger ranges of
// uneven splits spread over the CTAs.
//
// CUDA-core variant (fp32 caches, or when forced): a cluster of C CTAs per
// unit keeps its logits in shared memory, 8 pages per CTA up to 128 pages,
// 16 beyond (P <= 256).
constexpr int TC_MAX_PPC = 10;
constexpr int TC_MAX_PARTS = 26;  // ceil(256 / TC_MAX_PPC)
constexpr int TC_MAX_PAGES = TC_MAX_PARTS * TC_MAX_PPC;
__host__ __device__ inline int tc_parts(int P) { return P <= TC_MAX_PPC ? 1 : (P + TC_MAX_PPC - 1) / TC_MAX_PPC; }

struct DemandPlan {
  int variant, ppc, C;
};
inline DemandPlan demand_plan(int P, bool tc_ok) {
  DemandPlan pl;
  if (tc_ok && P <= TC_MAX_PAGES) {
    pl.variant = DEMAND_TC;
    pl.C = 1;
    pl.ppc = (P + tc_parts(P) - 1) / tc_parts(P);
  } else {
    pl.variant = DEMAND_FFMA;
    const int ppc = P <= 128 ? 8 : 16;
    pl.C = (P + ppc - 1) / ppc;
    if (pl.C < 1) pl.C = 1;
    pl.ppc = (P + pl.C - 1) / pl.C;
  }
  if (pl.ppc < 1) pl.ppc = 1;
  return pl;
}

// ---- entropy metric (Sec. 5.3 ablation): exp(H(a^x)) per unit ----------------
struct EntropyArgs {
  const DevReq* reqs;      // [n] (num_pages, aval_off)
  const float* aval;       // a^S, a^L over C_t of the demand call: per unit [2][(P-1) b]
  int n, units, b;
  double* out;             // [n][units][2]
};
cudaError_t launch_entropy(const EntropyArgs& a, cudaStream_t s);

// ---- A8-A10: window mask, Eq. 10 top-k, copy-on-write compaction -----------
struct CompressArgs {
  void* k_cache;
  void* v_cache;
  int num_pages_total;
  int L, Hkv, D, elt;      // elt = bytes per element
  int b, R, k_loc;
  int drop;                // pages' worth of history dropped: 1 Compress & Hold, 2 Shrink
  int fill;                // 1: hole-fill compaction (order-destroying), 0: stable
  int select_only;         // 1: write the keep masks (keep_out) and stop before the compaction
  const DevReq* reqs;
  const int32_t* old_bt;
  const int32_t* new_bt;
  const float* scores;     // importance cache (selection mode)
  const uint32_t* keep_in; // caller masks (given-mask mode) or null
  uint32_t* keep_out;      // keep masks written here (always)
  const int32_t* work;     // request indices
  int n_work;
  unsigned long long* moved;
  int* err;
  long long wait_limit;    // clock cycles a copy wait may take before the CTA gives up
                           // (ERR_TIMEOUT; 0: at once); drains of copies already issued
                           // always wait up to kDefaultWaitLimit
};
constexpr long long kDefaultWaitLimit = 1ll << 31;  // about one second of SM clock
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);

}  // namespace gp
