// The entropy metric of the dual-timescale ablation (GrowPage Sec. 5.3,
// Table 2), which puts attention entropy where the Top-p working set D_p
// stands.  The pages give no formula; the metric here is the effective
// support size E^x = exp(H(a^x)), H(a) = -sum_i a_i ln a_i over the demand
// candidates C_t, per (request, layer, KV head, summary).
//
// Input: the GQA-mean distributions a^S, a^L over C_t that the demand
// kernels keep for the D_p select (fp32, per unit [2][(P-1) b]).  One CTA
// per (request, unit, summary) streams its row with 16-byte loads; the four
// terms a ln a of a load are formed and added in fp32, and those partial
// sums are added in fp64 (GB300's fp64 rate is low, so one fp64 add per
// four candidates, not per candidate).  The row is 4 bytes per candidate,
// 1/64 of the K bytes the scan read at d = 128.
#include <cstdint>

#include "gp_kernels.h"

namespace gp {
namespace {

constexpr int NT = 256;

__device__ __forceinline__ float plogp(float v) { return v > 0.f ? v * logf(v) : 0.f; }

__global__ void __launch_bounds__(NT) k_entropy(EntropyArgs a) {
  __shared__ double part[NT / 32];
  const int x = blockIdx.x & 1;
  const int unit = (int)(blockIdx.x >> 1) % a.units;
  const int r = (int)(blockIdx.x >> 1) / a.units;
  const DevReq rq = a.reqs[r];
  const int ndem = (rq.num_pages - 1) * a.b;  // a multiple of 4: b = 256
  double acc = 0.0;
  if (ndem > 0) {
    const float4* row = reinterpret_cast<const float4*>(a.aval + rq.aval_off + ((size_t)unit * 2 + x) * ndem);
    for (int i = threadIdx.x; i < ndem / 4; i += NT) {
      const float4 v = __ldg(row + i);
      acc += (double)((plogp(v.x) + plogp(v.y)) + (plogp(v.z) + plogp(v.w)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double h = 0.0;
    for (int w = 0; w < NT / 32; ++w) h -= part[w];
    a.out[((size_t)r * a.units + unit) * 2 + x] = ndem > 0 ? exp(h) : 0.0;
  }
}

}  // namespace

cudaError_t launch_entropy(const EntropyArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  if (a.units < 1 || a.b % 4 != 0) return cudaErrorInvalidValue;
  k_entropy<<<dim3((unsigned)(a.n * a.units * 2)), NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gp
