// Query-summary kernels for sm_103a.
//
//  k_ema_update  -- GrowPage Sec. 3.2 Eq. 6 with the App. E.1 first-step
//                   initialisation, in place on the fp64 summary pool
//                   [L][M][2][Hq][D] (App. E.1 Eq. 11).  Pure streaming: one
//                   thread per 4 elements, 16-byte loads/stores; 34 bytes of
//                   HBM traffic per element for bf16 queries.
//  k_prep_queries -- App. E.1 Eq. 12 calibration gamma = RMS(q_t)/RMS(qbar)
//                   and rotate-half RoPE at the current position, for the
//                   requests at a capacity boundary, pre-scaled by
//                   log2(e)/sqrt(D) so the score kernels work in base 2.
//                   Writes the fp32 rows and their three-part bf16 split in
//                   the tensor-core operand layout.
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

// Block per (request, layer, 8 query heads); warp per query head.  The
// RoPE angles depend only on (position, pair index), so each block computes
// them once: the angle pos * theta^(-2i/d) and its reduction to [-pi, pi]
// in fp64 (exact enough for positions in the millions), cos/sin of the
// reduced angle in fp32.  Calibration and rotation run in fp32 on the fp64
// summaries rounded once; the result is rounded to fp32 (the qt rows) and
// split into three bf16 parts for the tensor-core scan.
template <int D>
__global__ void __launch_bounds__(256) k_prep_queries(PrepArgs a) {
  constexpr int PER = D / 32;
  __shared__ float cs_s[D / 2], sn_s[D / 2];
  const int hblocks = (a.Hq + 7) / 8;
  const int hb = blockIdx.x % hblocks;
  const int l = (blockIdx.x / hblocks) % a.L;
  const int r = blockIdx.x / (hblocks * a.L);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero32; i += (size_t)gridDim.x * blockDim.x)
    a.zero32[i] = 0u;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero64; i += gridDim.x * blockDim.x) a.zero64[i] = 0ull;
  const DevReq rq = a.reqs[r];
  if (threadIdx.x < D / 2) {
    const double ang = (double)rq.pos * a.inv_freq[threadIdx.x];
    const double k = rint(ang * 0.15915494309189535);                  // 1 / (2 pi)
    double red = fma(-k, 6.283185307179586, ang);                      // 2 pi, high part
    red = fma(-k, 2.4492935982947064e-16, red);                        // 2 pi, low part
    float sn, cs;
    sincosf((float)red, &sn, &cs);
    cs_s[threadIdx.x] = cs;
    sn_s[threadIdx.x] = sn;
  }
  __syncthreads();
  const int g = hb * 8 + warp;
  if (g >= a.Hq) return;
  const int slot = rq.slot;
  const int G = a.Hq / a.Hkv;
  const int h = g / G, gi = g % G;
  if (slot < 0 || slot >= a.M) {
    if (lane == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }
  const size_t qoff = (((size_t)l * a.n + r) * a.Hq + g) * D;
  float sq = 0.f;
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int i = lane + 32 * m;
    const float v = a.q_f32 ? static_cast<const float*>(a.q)[qoff + i]
                            : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qoff + i]);
    sq = fmaf(v, v, sq);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rms_q = sqrtf(sq / D);
  const float scale = 1.4426950408889634f / sqrtf((float)D);  // log2(e)/sqrt(D)
  const int ROWS = 2 * G;
  const int NB = (3 * ROWS + 15) / 16 * 16;
  unsigned char* bq = a.bq ? a.bq + (((size_t)r * a.L + l) * a.Hkv + h) * bq_bytes(D, G) : nullptr;
  for (int x = 0; x < 2; ++x) {
    const double* row = a.pool + (((size_t)l * a.M + slot) * 2 + x) * ((size_t)a.Hq * D) + (size_t)g * D;
    float v[PER];
    float sv = 0.f;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      v[m] = (float)row[lane + 32 * m];
      sv = fmaf(v[m], v[m], sv);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
    const float rms_v = sqrtf(sv / D);
    const float gs = rms_v > 0.f ? (rms_q / rms_v) * scale : 0.f;   // Eq. 12 gain, base-2 scale
    const int rr = x * G + gi;
    float* out = a.qt + ((((size_t)r * a.L + l) * a.Hkv + h) * ROWS + rr) * D;
#pragma unroll
    for (int m = 0; m < PER / 2; ++m) {
      const int i = lane + 32 * m;          // i < D/2; partner i + D/2 is v[m + PER/2]
      const float x1 = v[m], x2 = v[m + PER / 2];
      const float c = cs_s[i], sn = sn_s[i];
      const float o1 = gs * fmaf(x1, c, -x2 * sn);
      const float o2 = gs * fmaf(x2, c, x1 * sn);
      out[i] = o1;
      out[i + D / 2] = o2;
      if (bq) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = e ? i + D / 2 : i;
          const float q = e ? o2 : o1;
          const __nv_bfloat16 h1 = __float2bfloat16_rn(q);
          const float r1 = q - __bfloat162float(h1);
          const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
          const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
          const __nv_bfloat16 parts[3] = {h1, h2, h3};
#pragma unroll
          for (int sp = 0; sp < 3; ++sp) {
            const int n = sp * ROWS + rr;
            const size_t off = (size_t)(d >> 6) * NB * 128 + (size_t)n * 128 + ((((d & 63) >> 3) ^ (n & 7)) << 4) +
                               (size_t)(d & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(bq + off) = parts[sp];
          }
        }
      }
    }
  }
  // the padding rows of the unit's operand are zero
  if (bq && gi == 0) {
    const int pad_rows = NB - 3 * ROWS;
    for (int hf = 0; hf < D / 64; ++hf)
      for (int k = lane; k < pad_rows * 32; k += 32) {
        const int n = 3 * ROWS + k / 32;
        reinterpret_cast<uint32_t*>(bq + (size_t)hf * NB * 128 + (size_t)n * 128)[k % 32] = 0u;
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
  const int blocks = a.n * a.L * ((a.Hq + 7) / 8);
  if (blocks == 0) return cudaSuccess;
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
