// Internal interface between the host engine (growpage.cpp) and the sm_103a
// kernels.  Plain structs of device pointers and sizes; no torch types.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gp {

// Per-request descriptor uploaded for one hot-path call.
struct DevReq {
  int32_t num_pages;   // P
  int32_t slot;        // summary-pool row
  int64_t pos;         // current decode position (RoPE)
  int64_t score_off;   // float offset of the request's importance cache
  int64_t dbg_off;     // float offset of its debug probabilities (or -1)
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
  double theta;
  float* qt;               // [n][L][Hkv][2G][D], scaled by log2(e)/sqrt(D)
  int* err;
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);

// ---- A3-A5: score scan, softmax, GQA mean, D_p, importance cache -----------
struct DemandArgs {
  const void* k_cache;     // [L][num_pages][Hkv][b][D]
  int kv_f32;
  int num_pages_total;
  int L, Hkv, D, G;
  int b, R;
  double p;
  const float* qt;
  const DevReq* reqs;
  const int32_t* bt;       // packed block tables
  const int32_t* work;     // request indices handled by this launch
  int n_work;
  int C;                   // cluster size (CTAs per unit)
  int ppc;                 // pages per CTA
  float* scores;           // importance cache, log2 domain
  int32_t* kout;           // [n][L*Hkv][2]
  unsigned long long* ksum;// [n][2]
  float* dbg;              // optional [..][2][(P-1) b] per unit
  int* err;
};
size_t demand_smem_bytes(int D, int G, int ppc);
cudaError_t launch_demand(const DemandArgs& a, cudaStream_t s);

// ---- A8-A10: window mask, Eq. 10 top-k, copy-on-write compaction -----------
struct CompressArgs {
  void* k_cache;
  void* v_cache;
  int num_pages_total;
  int L, Hkv, D, elt;      // elt = bytes per element
  int b, R, k_loc;
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
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);

}  // namespace gp
