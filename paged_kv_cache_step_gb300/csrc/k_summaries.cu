// Query-summary kernels for sm_103a.
//
//  k_ema_update  -- GrowPage Sec. 3.2 Eq. 6 with the App. E.1 first-step
//                   initialisation, in place on the fp64 summary pool
//                   [L][M][2][Hq][D] (App. E.1 Eq. 11).  Pure streaming: a
//                   block per (1024-element chunk, request, layer), whose
//                   queries and two summary rows are contiguous; one thread
//                   per 4 elements, 16-byte loads/stores; 34 bytes of HBM
//                   traffic per element for bf16 queries.
//  k_prep_queries -- App. E.1 Eq. 12 calibration gamma = RMS(q_t)/RMS(qbar)
//                   and rotate-half RoPE at the current position, for the
//                   requests at a capacity boundary, pre-scaled by
//                   log2(e)/sqrt(D) so the score kernels work in base 2.
//                   Writes the fp32 rows and their three-part bf16 split in
//                   the tensor-core operand layout.
#include <cuda_bf16.h>

#include <cstring>

#include "gp_kernels.h"

namespace gp {
namespace {

// Exact float -> double by integer operations (a normal or zero float: the
// exponent is rebased and the fraction moved up); other inputs take the
// ordinary conversion.  Keeps the widening of the queries off GB300's narrow
// fp64 pipe, which the two fused multiply-adds per summary element already use.
__device__ __forceinline__ double widen_exact(float f) {
  const unsigned u = __float_as_uint(f);
  const unsigned e = (u >> 23) & 0xffu;
  if ((u & 0x7fffffffu) == 0u) return __hiloint2double((int)(u & 0x80000000u), 0);
  if (e == 0u || e == 0xffu) return (double)f;
  const unsigned hi = (u & 0x80000000u) | ((e + 896u) << 20) | ((u & 0x7fffffu) >> 3);
  return __hiloint2double((int)hi, (int)((u & 7u) << 29));
}

// The fp64 product w q of a weight w = mw 2^(ew - 1075) (mw its 53-bit
// integer significand, 0 < w) and a bf16 query with bit pattern qb, by
// integer operations: the significands' product has 60 or 61 bits and is
// rounded to 53 (to nearest, ties to even), which is exactly what the fp64
// multiply returns.  False for a subnormal, infinite or NaN q, or a product
// outside the normal range.  k_ema_update uses it to build, per block, the
// products for the 128 bf16 significands, off GB300's narrow fp64 pipe.
__device__ __forceinline__ bool mul_w_bf16(unsigned long long mw, int ew, unsigned qb, double& out) {
  const unsigned eq = (qb >> 7) & 0xffu, sq = (qb >> 15) & 1u;
  if (eq == 0u) {
    if ((qb & 0x7fu) != 0u) return false;
    out = __hiloint2double((int)(sq << 31), 0);  // +-0 (w > 0)
    return true;
  }
  if (eq == 0xffu) return false;
  const unsigned long long p = mw * (unsigned long long)(0x80u | (qb & 0x7fu));  // [2^59, 2^61)
  int sh = (p >> 60) != 0ull ? 8 : 7;
  unsigned long long m = p >> sh;
  const unsigned long long rem = p & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
  if (rem > half || (rem == half && (m & 1ull))) {
    ++m;
    if (m == (1ull << 53)) {
      m >>= 1;
      ++sh;
    }
  }
  // value = m 2^(ew - 1075 + eq - 134 + sh); biased exponent of m 2^k with m in [2^52, 2^53)
  const int be = ew + (int)eq - 134 + sh;
  if (be < 1 || be > 2046) return false;
  const unsigned long long bits = ((unsigned long long)sq << 63) | ((unsigned long long)be << 52) |
                                  (m & ((1ull << 52) - 1ull));
  out = __longlong_as_double((long long)bits);
  return true;
}

// The fp64 multiply for the queries the table does not cover (zero,
// subnormal, infinite or NaN bf16, or fp32 queries).  A function of its own
// so that the compiler keeps it behind a branch: if-converted into the main
// path it would issue two fp64 multiplies for every element.
__device__ __noinline__ double mul_fp64(double w, double q) { return w * q; }

// grid (ceil(Hq D / 1024), n, L), 256 threads: thread t of block (c, r, l)
// owns elements [4 (256 c + t), +4) of the (layer l, request r) row.
// (mws, ews), (mwl, ewl): 1 - beta_s and 1 - beta_l as significand and
// biased exponent.  tab: both are at least 2^-896, so that every product
// with a normal bf16 query is a normal double.
//
// (1 - beta) q for a normal bf16 query q = (-1)^s (1 + f/128) 2^(e - 127)
// is RN((1 - beta)(1 + f/128)) with e - 127 added to its exponent and s put
// in its sign bit: scaling by a power of two is exact while the result
// stays normal.  The block first forms the 128 rounded products of each
// weight with 1 + f/128, with integer operations, in shared memory; each
// element then takes one 16-byte shared load and two integer adds, and
// only the two fused multiply-adds run on the fp64 pipe.
__global__ void __launch_bounds__(256) k_ema_update(EmaArgs a, unsigned long long mws, int ews,
                                                    unsigned long long mwl, int ewl, int tab) {
  // {low word, high word - (127 << 20)} of both products, per fraction f
  __shared__ uint4 wq[128];
  const int r = blockIdx.y, l = blockIdx.z;
  const int row = a.Hq * a.D;
  const int e0 = (blockIdx.x * 256 + threadIdx.x) * 4;
  const int slot = a.slots[r];
  const bool first = a.first[r] != 0;  // loaded beside the slot, not after it
  if (threadIdx.x < 128) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (tab) {
      double ps, pl;
      mul_w_bf16(mws, ews, 0x3f80u | threadIdx.x, ps);  // q = 1 + f/128
      mul_w_bf16(mwl, ewl, 0x3f80u | threadIdx.x, pl);
      const unsigned long long bs = (unsigned long long)__double_as_longlong(ps);
      const unsigned long long bl = (unsigned long long)__double_as_longlong(pl);
      v = make_uint4((unsigned)bs, (unsigned)(bs >> 32) - (127u << 20), (unsigned)bl,
                     (unsigned)(bl >> 32) - (127u << 20));
    }
    wq[threadIdx.x] = v;
  }
  __syncthreads();
  if (slot < 0 || slot >= a.M) {
    if (blockIdx.x == 0 && l == 0 && threadIdx.x == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }
  if (e0 >= row) return;
  const size_t qi = ((size_t)l * a.n + r) * row + e0;
  float qf[4];
  unsigned qb[4] = {0u, 0u, 0u, 0u};  // bf16 bit patterns
  if (a.q_f32) {
    const float4 t = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qi);
    qf[0] = t.x; qf[1] = t.y; qf[2] = t.z; qf[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.q) + qi);
    qb[0] = t.x & 0xffffu;
    qb[1] = t.x >> 16;
    qb[2] = t.y & 0xffffu;
    qb[3] = t.y >> 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) qf[i] = __uint_as_float(qb[i] << 16);
  }
  double2* row_s = reinterpret_cast<double2*>(a.pool + ((size_t)l * a.M + slot) * 2 * row + e0);
  double2* row_l = reinterpret_cast<double2*>(reinterpret_cast<double*>(row_s) + row);
  // the old summaries are loaded whatever `first` says, so that their loads
  // leave with the query's instead of waiting for the flag
  const double2 os0 = __ldcs(row_s), os1 = __ldcs(row_s + 1);
  const double2 ol0 = __ldcs(row_l), ol1 = __ldcs(row_l + 1);
  const double os[4] = {os0.x, os0.y, os1.x, os1.y}, ol[4] = {ol0.x, ol0.y, ol1.x, ol1.y};
  double ns[4], nl[4];
  bool other = a.q_f32 || !tab;  // a query the table does not cover
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned e7 = qb[i] & 0x7f80u;
    other |= e7 == 0u || e7 == 0x7f80u;
  }
  if (first) {
#pragma unroll
    for (int i = 0; i < 4; ++i) ns[i] = nl[i] = widen_exact(qf[i]);
  } else if (!other) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = wq[qb[i] & 0x7fu];
      const unsigned adj = ((qb[i] & 0x7f80u) << 13) | ((qb[i] & 0x8000u) << 16);  // (e << 20) | (s << 31)
      ns[i] = fma(a.beta_s, os[i], __hiloint2double((int)(t.y + adj), (int)t.x));
      nl[i] = fma(a.beta_l, ol[i], __hiloint2double((int)(t.w + adj), (int)t.z));
    }
  } else {
    const double ws = 1.0 - a.beta_s, wl = 1.0 - a.beta_l;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const double q = widen_exact(qf[i]);
      ns[i] = fma(a.beta_s, os[i], mul_fp64(ws, q));
      nl[i] = fma(a.beta_l, ol[i], mul_fp64(wl, q));
    }
  }
  const double2 s0 = make_double2(ns[0], ns[1]), s1 = make_double2(ns[2], ns[3]);
  const double2 l0 = make_double2(nl[0], nl[1]), l1 = make_double2(nl[2], nl[3]);
  __stcs(row_s, s0);
  __stcs(row_s + 1, s1);
  __stcs(row_l, l0);
  __stcs(row_l + 1, l1);
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
  const int g = hb * 8 + warp;
  const int slot = rq.slot;
  const bool live = g < a.Hq && slot >= 0 && slot < a.M;
  // The warp's loads -- the query row and both summary rows -- leave
  // together, before the angles are computed, so the block waits on memory
  // once.
  float qv[PER], vs[2][PER];
  if (live) {
    const size_t qoff = (((size_t)l * a.n + r) * a.Hq + g) * D;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int i = lane + 32 * m;
      qv[m] = a.q_f32 ? static_cast<const float*>(a.q)[qoff + i]
                      : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qoff + i]);
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const double* row = a.pool + (((size_t)l * a.M + slot) * 2 + x) * ((size_t)a.Hq * D) + (size_t)g * D;
#pragma unroll
      for (int m = 0; m < PER; ++m) vs[x][m] = (float)row[lane + 32 * m];
    }
  }
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
  if (g >= a.Hq) return;
  const int G = a.Hq / a.Hkv;
  const int h = g / G, gi = g % G;
  if (!live) {
    if (lane == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }
  float sq = 0.f;
#pragma unroll
  for (int m = 0; m < PER; ++m) sq = fmaf(qv[m], qv[m], sq);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rms_q = sqrtf(sq / D);
  const float scale = 1.4426950408889634f / sqrtf((float)D);  // log2(e)/sqrt(D)
  const int ROWS = 2 * G;
  const int NB = (3 * ROWS + 15) / 16 * 16;
  unsigned char* bq = a.bq ? a.bq + (((size_t)r * a.L + l) * a.Hkv + h) * bq_bytes(D, G) : nullptr;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const float* v = vs[x];
    float sv = 0.f;
#pragma unroll
    for (int m = 0; m < PER; ++m) sv = fmaf(v[m], v[m], sv);
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
  if (a.n == 0 || a.L == 0) return cudaSuccess;
  if (a.D % 4 != 0 || a.n > 65535 || a.L > 65535) return cudaErrorInvalidValue;
  const int row = a.Hq * a.D;
  // 1 - beta as significand and biased exponent (0 < 1 - beta <= 1: normal)
  auto split = [](double w, unsigned long long& m, int& e) {
    unsigned long long b;
    std::memcpy(&b, &w, sizeof(b));
    e = (int)((b >> 52) & 0x7ffull);
    m = (b & ((1ull << 52) - 1ull)) | (1ull << 52);
  };
  unsigned long long mws, mwl;
  int ews, ewl;
  split(1.0 - a.beta_s, mws, ews);
  split(1.0 - a.beta_l, mwl, ewl);
  if (ews == 0 || ewl == 0) return cudaErrorInvalidValue;
  const int tab = ews >= 127 && ewl >= 127;  // both weights at least 2^-896
  k_ema_update<<<dim3((row + 1023) / 1024, a.n, a.L), 256, 0, s>>>(a, mws, ews, mwl, ewl, tab);
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
