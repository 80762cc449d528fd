// Internal interface between the host engine (growpage.cpp) and the decode
// attention kernels (k_attention.cu, k_attention_tc.cu).  Plain structs of
// device pointers and sizes; no torch types.
#pragma once

#include "gp_kernels.h"

namespace gp {

// ---- decode attention with the summary update fused in (one layer) -------
// One work item of the tensor-core kernel, built by the host: the split
// `split` (of nsp) of request r's attended pages, for KV head h, pages
// [p0, p0 + ceil(T / 2)) of its block table.
struct AttnItem {
  int32_t r, h, split, nsp;
  int32_t part_first;  // the first partial of (r, h); this item's is part_first + split
  int32_t p0;          // first page of the split
  int32_t T;           // tiles of 128 keys (0: no attended token)
  int32_t ntok;        // tokens the request attends to
  int32_t bt_off, slot;
  int64_t pos;
};
static_assert(sizeof(AttnItem) == 48, "three 16-byte loads per item");

struct AttnArgs {
  CUtensorMap kmap, vmap;  // K and V caches as [rows][D] bf16, box 64 x 128, 128-byte swizzle
  int tc;                  // 1: the tensor-core kernel (bf16 caches, D = 128, G = 2 or 4)
  const void* k_cache;     // [L][num_pages][Hkv][b][D], keys stored rotated
  const void* v_cache;
  int kv_f32;
  int num_pages_total;
  int layer, Hq, Hkv, D, G, M;
  const DevReq* reqs;      // [n] (num_pages, slot, pos, bt_off)
  const int32_t* bt;       // packed block tables
  const int32_t* ntok;     // [n] cached tokens attended to
  const void* q;           // [n][Hq][D] pre-RoPE query of this layer
  int q_f32;
  const uint8_t* first;    // [n] 1: the slot's first step (summaries initialised)
  double* pool;            // summary pool [L][M][2][Hq][D]
  double beta_s, beta_l;
  const double* inv_freq;  // [D/2]
  float* out;              // [n][Hq][D]
  float* part;             // split partials [n_ctas][G][D + 2], those of (r, h) together
  unsigned* tickets;       // [n][Hkv], zero before the launch
  const int32_t* split_base;  // [n + 1] first work item of each request, in `order`
  const int32_t* order;    // [n] requests, longest first; request order[i] has
                           // (split_base[i+1] - split_base[i]) / Hkv splits, work
                           // item split_base[i] + split * Hkv + h
  int n, n_ctas;           // n_ctas: work items (request, KV head, split); the
                           // CUDA-core kernel runs one CTA per item
  int grid;                // tensor-core kernel: persistent CTAs (<= n_ctas)
  const AttnItem* items;   // tensor-core kernel: [n_ctas] work items, those of CTA c at
  const int32_t* cta_begin;//   [cta_begin[c], cta_begin[c + 1]) ([grid + 1]); a pair's
                           //   items are consecutive, its partials part_first + split
  int* err;
};
cudaError_t launch_decode_attention(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_decode_attention_tc(const AttnArgs& a, cudaStream_t s);
// Whether the tensor-core attention kernel takes this shape.
inline bool attention_tc_shape(int D, int G) { return D == 128 && (G == 2 || G == 4); }

}  // namespace gp
