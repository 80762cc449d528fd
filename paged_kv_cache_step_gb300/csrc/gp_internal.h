// Read-only view of an engine context for translation units other than
// growpage.cpp (which owns the gp_ctx definition).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "growpage.h"

namespace gp {

struct CtxView {
  const gp_config* cfg;
  void* k_cache;
  void* v_cache;
  const double* pool;   // summary pool [L][M][2][Hq][D]
  cudaStream_t stream;
  int* err_dev;         // kernel error word
  bool host_only;
  const double* inv_freq;     // RoPE inverse frequencies [D/2]
  const CUtensorMap* kmap;    // K cache tensor map (valid when tc_ok)
  bool tc_ok;                 // the tensor-core scan may be used
  int scan_kernel;            // GP_SCAN_*
};

// Fills *out; false for a null context.
bool ctx_view(const gp_ctx* c, CtxView* out);
// True if `slot` is bound to a request.
bool ctx_slot_bound(const gp_ctx* c, int slot);
// Waits for a compaction still running on the side stream (see
// gp_set_compaction_stream) before the caller reads K/V or engine scratch.
gp_status ctx_join_compaction(gp_ctx* c);
// Waits for a speculative selection still running on the engine's selection
// stream (it writes the kernel error word and reads the upload buffer).
gp_status ctx_join_select(gp_ctx* c);
// Drops the demand record of `slot`, so that a following gp_compress_hold of
// that slot is refused with GP_ERR_STATE until a new gp_boundary_demand.
void ctx_forget_demand(gp_ctx* c, int slot);
// Status of a nonzero kernel error word: GP_ERR_TIMEOUT when only bounded
// waits gave up, GP_ERR_INVALID when a device-side check failed.
gp_status status_of_kernel_error(int bits);
// Records the text returned by gp_last_error and returns `st`.
gp_status ctx_fail(gp_ctx* c, gp_status st, const char* msg);

}  // namespace gp
