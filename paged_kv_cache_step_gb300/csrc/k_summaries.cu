// Query-summary kernels for sm_103a.
//
//  k_ema_update  -- GrowPage Sec. 3.2 Eq. 6 with the App. E.1 first-step
//                   initialisation, in place on the fp64 summary pool
//                   [L][M][2][Hq][D] (App. E.1 Eq. 11).  Pure streaming: one
//                   thread per 4 elements, 16-byte loads/stores; 34 bytes of
//                   HBM traffic per element for bf16 queries.
//  k_prep_queries -- App. E.1 Eq. 12 calibration gamma = RMS(q_t)/RMS(qbar)
//                   and rotate-half RoPE at the current position, for the
//                   requests at a capacity boundary.  One warp per
//                   (request, layer, query head); fp64 arithmetic, rounded
//                   once to fp32 and pre-scaled by log2(e)/sqrt(D) so the
//                   score kernel works in base 2.
#include <cuda_bf16.h>

#include "gp_kernels.h"

namespace gp {
namespace {

__device__ __forceinline__ void load4(const void* q, int q_f32, size_t idx, double v[4]) {
  if (q_f32) {
    const float4 t = *reinterpret_cast<const float4*>(static_cast<const float*>(q) + idx);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(q) + idx);
    v[0] = __uint_as_float(t.x << 16);
    v[1] = __uint_as_float(t.x & 0xffff0000u);
    v[2] = __uint_as_float(t.y << 16);
    v[3] = __uint_as_float(t.y & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(256) k_ema_update(EmaArgs a) {
  const int dq = a.D / 4;
  const size_t total = (size_t)a.L * a.n * a.Hq * dq;
  const size_t hd = (size_t)a.Hq * a.D;
  const double ws = 1.0 - a.beta_s, wl = 1.0 - a.beta_l;
  for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (size_t)gridDim.x * blockDim.x) {
    const int d4 = (int)(it % dq);
    size_t rest = it / dq;
    const int g = (int)(rest % a.Hq);
    rest /= a.Hq;
    const int r = (int)(rest % a.n);
    const int l = (int)(rest / a.n);
    const int slot = a.slots[r];
    if (slot < 0 || slot >= a.M) {
      if (d4 == 0 && g == 0 && l == 0) atomicOr(a.err, ERR_BAD_SLOT);
      continue;
    }
    double q[4];
    load4(a.q, a.q_f32, (((size_t)l * a.n + r) * a.Hq + g) * a.D + d4 * 4, q);
    double2* row_s = reinterpret_cast<double2*>(
        a.pool + (((size_t)l * a.M + slot) * 2 + 0) * hd + (size_t)g * a.D + d4 * 4);
    double2* row_l = reinterpret_cast<double2*>(reinterpret_cast<double*>(row_s) + hd);
    double2 s0, s1, l0, l1;
    if (a.first[r]) {
      s0 = make_double2(q[0], q[1]);
      s1 = make_double2(q[2], q[3]);
      l0 = s0;
      l1 = s1;
    } else {
      const double2 os0 = row_s[0], os1 = row_s[1];
      const double2 ol0 = row_l[0], ol1 = row_l[1];
      s0 = make_double2(fma(a.beta_s, os0.x, ws * q[0]), fma(a.beta_s, os0.y, ws * q[1]));
      s1 = make_double2(fma(a.beta_s, os1.x, ws * q[2]), fma(a.beta_s, os1.y, ws * q[3]));
      l0 = make_double2(fma(a.beta_l, ol0.x, wl * q[0]), fma(a.beta_l, ol0.y, wl * q[1]));
      l1 = make_double2(fma(a.beta_l, ol1.x, wl * q[2]), fma(a.beta_l, ol1.y, wl * q[3]));
    }
    row_s[0] = s0;
    row_s[1] = s1;
    row_l[0] = l0;
    row_l[1] = l1;
  }
}

// One warp per (request, layer, query head).  Lane l owns elements
// l + 32 m, so each rotate-half pair (i, i + D/2) sits in one lane.
template <int D>
__global__ void __launch_bounds__(256) k_prep_queries(PrepArgs a) {
  constexpr int PER = D / 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = a.n * a.L * a.Hq;
  if (warp >= total) return;
  const int g = warp % a.Hq;
  const int l = (warp / a.Hq) % a.L;
  const int r = warp / (a.Hq * a.L);
  const DevReq rq = a.reqs[r];
  const int slot = rq.slot;
  const int G = a.Hq / a.Hkv;
  const int h = g / G, gi = g % G;
  if (slot < 0 || slot >= a.M) {
    if (lane == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }
  const size_t qoff = (((size_t)l * a.n + r) * a.Hq + g) * D;
  double q[PER];
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int i = lane + 32 * m;
    float v;
    if (a.q_f32) {
      v = static_cast<const float*>(a.q)[qoff + i];
    } else {
      v = __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qoff + i]);
    }
    q[m] = v;
  }
  double sq = 0.0;
#pragma unroll
  for (int m = 0; m < PER; ++m) sq += q[m] * q[m];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const double rms_q = sqrt(sq / D);
  const double scale = 1.4426950408889634 / sqrt((double)D);  // log2(e)/sqrt(D)
  const double pos = (double)rq.pos;
  const double ltheta = log2(a.theta);
  for (int x = 0; x < 2; ++x) {
    const double* row = a.pool + (((size_t)l * a.M + slot) * 2 + x) * ((size_t)a.Hq * D) + (size_t)g * D;
    double v[PER];
    double sv = 0.0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      v[m] = row[lane + 32 * m];
      sv += v[m] * v[m];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
    const double rms_v = sqrt(sv / D);
    const double gamma = rms_v > 0.0 ? rms_q / rms_v : 0.0;
    float* out = a.qt + ((((size_t)r * a.L + l) * a.Hkv + h) * (2 * G) + x * G + gi) * D;
#pragma unroll
    for (int m = 0; m < PER / 2; ++m) {
      const int i = lane + 32 * m;          // i < D/2; partner i + D/2 is v[m + PER/2]
      const double inv_freq = exp2(-(2.0 * i / D) * ltheta);
      double sn, cs;
      sincos(pos * inv_freq, &sn, &cs);
      const double x1 = gamma * v[m], x2 = gamma * v[m + PER / 2];
      out[i] = (float)((x1 * cs - x2 * sn) * scale);
      out[i + D / 2] = (float)((x2 * cs + x1 * sn) * scale);
    }
  }
}

}  // namespace

cudaError_t launch_ema(const EmaArgs& a, cudaStream_t s) {
  const size_t total = (size_t)a.L * a.n * a.Hq * (a.D / 4);
  if (total == 0) return cudaSuccess;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  k_ema_update<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  const int warps = a.n * a.L * a.Hq;
  if (warps == 0) return cudaSuccess;
  const int blocks = (warps * 32 + 255) / 256;
  if (a.D == 128) {
    k_prep_queries<128><<<blocks, 256, 0, s>>>(a);
  } else if (a.D == 64) {
    k_prep_queries<64><<<blocks, 256, 0, s>>>(a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gp
