// Decode attention over the paged cache with the summary update fused in:
// the integration point of GrowPage Sec. 4.1 ("the decode attention kernel
// updates the query summaries in passing") for one layer of a decode step.
//
// Per request r and query head g (KV head h = g / G):
//   summaries (Eq. 6, App. E.1): on the slot's first step both are q;
//     else qbar^x <- beta_x qbar^x + (1 - beta_x) q, with q the pre-RoPE query;
//   attention: z_i = RoPE_pos(q) . k_i / sqrt(d) over the request's first
//     num_tokens cached tokens (keys are stored rotated), a = softmax(z),
//     out = sum_i a_i v_i (fp32).
//
// Work: one CTA per (request, KV head, split of the request's pages), 256
// threads.  The split-0 CTA also updates the G heads' summaries, from the
// query it has loaded anyway.  Per page of 256 keys:
//   logits -- a lane pair per key, each lane half of the row's 16-byte
//             chunks, a shuffle to finish the G dot products;
//   softmax -- online, base 2, per query row (a warp per row);
//   values  -- thread t owns 8 dimensions (16 bytes) of keys t/16, t/16+16,
//              ...: coalesced rows, G x 8 fp32 accumulators.
// Split partials (max, sum, G x d) go to scratch; the last CTA of a
// (request, KV head) merges them.  Bounded by HBM: K and V are read once.
#include <cuda_bf16.h>

#include "gp_kernels.h"

namespace gp {
namespace {

constexpr int NT = 256;
constexpr int PAGE = 256;
constexpr float NEGF = -1.0e30f;

__device__ __forceinline__ uint4 ld_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float bf_lo(unsigned u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(unsigned u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int G, bool F32>
__global__ void __launch_bounds__(NT) k_decode_attn(AttnArgs a) {
  constexpr int HALFC = D / 16;  // 16-byte chunks per half key row (bf16)
  __shared__ float qs[G][D];     // rotated query rows, scaled by log2(e)/sqrt(d)
  __shared__ float lg[G][PAGE];  // logits, then weights of the current page
  __shared__ float rs[G][3];     // running max, running sum, rescale of this page
  __shared__ int s_last;
  extern __shared__ float accs[];  // [KG][G][D] partial sums of the key groups (dynamic)
  constexpr int NCH = D / 8;       // 8-dimension chunks of a row
  constexpr int KG = NT / NCH;     // key groups of the value pass

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x % a.nsplit;
  const int h = (blockIdx.x / a.nsplit) % a.Hkv;
  const int r = blockIdx.x / (a.nsplit * a.Hkv);
  const DevReq rq = a.reqs[r];
  const int ntok = a.ntok[r];
  const int P = rq.num_pages;
  const int p0 = (split * P) / a.nsplit, p1 = ((split + 1) * P) / a.nsplit;
  const int slot = rq.slot;
  if (slot < 0 || slot >= a.M) {
    if (tid == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }

  // ---- query rows: summary update (split 0) and RoPE ----------------------
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    const int g = h * G + gi;
    const size_t qi = ((size_t)r * a.Hq + g) * D + d;
    const double qv = a.q_f32 ? (double)static_cast<const float*>(a.q)[qi]
                              : (double)__bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qi]);
    if (split == 0) {
      double* row = a.pool + (((size_t)a.layer * a.M + slot) * 2) * ((size_t)a.Hq * D) + (size_t)g * D + d;
      double* row_l = row + (size_t)a.Hq * D;
      if (a.first[r]) {
        *row = qv;
        *row_l = qv;
      } else {
        *row = fma(a.beta_s, *row, (1.0 - a.beta_s) * qv);
        *row_l = fma(a.beta_l, *row_l, (1.0 - a.beta_l) * qv);
      }
    }
    qs[gi][d] = (float)qv;
  }
  __syncthreads();
  {
    // rotate-half RoPE at the request's position: pairs (i, i + D/2)
    for (int e = tid; e < G * (D / 2); e += NT) {
      const int gi = e / (D / 2), i = e % (D / 2);
      const double ang = (double)rq.pos * a.inv_freq[i];
      const double k = rint(ang * 0.15915494309189535);
      double red2 = fma(-k, 6.283185307179586, ang);
      red2 = fma(-k, 2.4492935982947064e-16, red2);
      float sn, cs;
      sincosf((float)red2, &sn, &cs);
      const float x1 = qs[gi][i], x2 = qs[gi][i + D / 2];
      const float sc = 1.4426950408889634f / sqrtf((float)D);
      const float o1 = sc * fmaf(x1, cs, -x2 * sn), o2 = sc * fmaf(x2, cs, x1 * sn);
      qs[gi][i] = o1;
      qs[gi][i + D / 2] = o2;
    }
  }
  if (tid < G) {
    rs[tid][0] = NEGF;
    rs[tid][1] = 0.f;
    rs[tid][2] = 1.f;
  }
  __syncthreads();

  // value accumulators: dims [8 c, 8 c + 8) of keys kg, kg + KG, ...
  const int c = tid % NCH, kg = tid / NCH;
  float acc[G][8];
#pragma unroll
  for (int gi = 0; gi < G; ++gi)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[gi][j] = 0.f;

  const unsigned char* kc = static_cast<const unsigned char*>(a.k_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(a.v_cache);
  constexpr int RB = F32 ? D * 4 : D * 2;
  const size_t head_stride = (size_t)PAGE * RB;
  for (int j = p0; j < p1; ++j) {
    int pg = a.bt[rq.bt_off + j];
    if (pg < 0 || pg >= a.num_pages_total) {
      if (tid == 0) atomicOr(a.err, ERR_BAD_PAGE);
      pg = 0;
    }
    const size_t base = (((size_t)a.layer * a.num_pages_total + pg) * a.Hkv + h) * head_stride;
    const int nvalid = min(PAGE, max(0, ntok - j * PAGE));
    // ---- logits: lane pair per key ----
    for (int k0 = warp * 32; k0 < warp * 32 + 32; k0 += 16) {
      const int key = k0 + (lane >> 1), half = lane & 1;
      float dot[G];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) dot[gi] = 0.f;
      if (key < nvalid) {
        if constexpr (F32) {
          const unsigned char* row = kc + base + (size_t)key * RB + half * (RB / 2);
#pragma unroll
          for (int ch = 0; ch < RB / 32; ++ch) {
            const uint4 v = ld_nc(row + ch * 16);
            const int d0 = half * (D / 2) + ch * 4;
            const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
              for (int t = 0; t < 4; ++t) dot[gi] = fmaf(qs[gi][d0 + t], f[t], dot[gi]);
          }
        } else {
          const unsigned char* row = kc + base + (size_t)key * RB + half * (RB / 2);
          uint4 v[HALFC];
#pragma unroll
          for (int ch = 0; ch < HALFC; ++ch) v[ch] = ld_nc(row + ch * 16);
#pragma unroll
          for (int ch = 0; ch < HALFC; ++ch) {
            const int d0 = half * (D / 2) + ch * 8;
            const float f[8] = {bf_lo(v[ch].x), bf_hi(v[ch].x), bf_lo(v[ch].y), bf_hi(v[ch].y),
                                bf_lo(v[ch].z), bf_hi(v[ch].z), bf_lo(v[ch].w), bf_hi(v[ch].w)};
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
              for (int t = 0; t < 8; ++t) dot[gi] = fmaf(qs[gi][d0 + t], f[t], dot[gi]);
          }
        }
      }
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const float tot = dot[gi] + __shfl_xor_sync(0xffffffffu, dot[gi], 1);
        if (half == 0) lg[gi][key] = key < nvalid ? tot : NEGF;
      }
    }
    __syncthreads();
    // ---- online softmax: warp gi takes row gi ----
    if (warp < G) {
      float m = NEGF;
      for (int i = lane; i < PAGE; i += 32) m = fmaxf(m, lg[warp][i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float mold = rs[warp][0];
      const float mnew = fmaxf(mold, m);
      float s = 0.f;
      for (int i = lane; i < PAGE; i += 32) {
        const float w = lg[warp][i] > 0.5f * NEGF ? ex2f(lg[warp][i] - mnew) : 0.f;
        lg[warp][i] = w;
        s += w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) {
        const float scale = mold > 0.5f * NEGF ? ex2f(mold - mnew) : 0.f;
        rs[warp][0] = mnew;
        rs[warp][1] = rs[warp][1] * scale + s;
        rs[warp][2] = scale;
      }
    }
    __syncthreads();
    // ---- values ----
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const float sc = rs[gi][2];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[gi][t] *= sc;
    }
    for (int key = kg; key < nvalid; key += KG) {
      float f[8];
      if constexpr (F32) {
        const unsigned char* row = vc + base + (size_t)key * RB + c * 32;
        const uint4 v0 = ld_nc(row), v1 = ld_nc(row + 16);
        f[0] = __uint_as_float(v0.x); f[1] = __uint_as_float(v0.y); f[2] = __uint_as_float(v0.z); f[3] = __uint_as_float(v0.w);
        f[4] = __uint_as_float(v1.x); f[5] = __uint_as_float(v1.y); f[6] = __uint_as_float(v1.z); f[7] = __uint_as_float(v1.w);
      } else {
        const uint4 v = ld_nc(vc + base + (size_t)key * RB + c * 16);
        f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
        f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
      }
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const float w = lg[gi][key];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[gi][t] = fmaf(w, f[t], acc[gi][t]);
      }
    }
    __syncthreads();  // lg is overwritten by the next page
  }

  // ---- the split's partial: sum the KG key groups ----
  float* part = accs;  // [KG][G][D]
#pragma unroll
  for (int gi = 0; gi < G; ++gi)
#pragma unroll
    for (int t = 0; t < 8; ++t) part[((size_t)kg * G + gi) * D + 8 * c + t] = acc[gi][t];
  __syncthreads();
  float* po = a.part + (((size_t)r * a.Hkv + h) * a.nsplit + split) * (size_t)G * (D + 2);
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    float s = 0.f;
    for (int q = 0; q < KG; ++q) s += part[((size_t)q * G + gi) * D + d];
    po[gi * (D + 2) + d] = s;
  }
  if (tid < G) {
    po[tid * (D + 2) + D] = rs[tid][0];
    po[tid * (D + 2) + D + 1] = rs[tid][1];
  }
  // ---- the last split of (request, KV head) merges ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(a.tickets + (size_t)r * a.Hkv + h, 1u);
    s_last = old == (unsigned)(a.nsplit - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  const float* pb = a.part + ((size_t)r * a.Hkv + h) * a.nsplit * (size_t)G * (D + 2);
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    float M = NEGF;
    for (int sp = 0; sp < a.nsplit; ++sp) M = fmaxf(M, __ldcg(pb + ((size_t)sp * G + gi) * (D + 2) + D));
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) {
      const float* q = pb + ((size_t)sp * G + gi) * (D + 2);
      const float m = __ldcg(q + D);
      const float w = m > 0.5f * NEGF ? ex2f(m - M) : 0.f;
      num = fmaf(w, __ldcg(q + d), num);
      den = fmaf(w, __ldcg(q + D + 1), den);
    }
    a.out[((size_t)r * a.Hq + h * G + gi) * D + d] = den > 0.f ? num / den : 0.f;
  }
}

template <int D, int G, bool F32>
cudaError_t launch_t(const AttnArgs& a, cudaStream_t s) {
  const int smem = (NT / (D / 8)) * G * D * (int)sizeof(float);
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(k_decode_attn<D, G, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_decode_attn<D, G, F32><<<dim3(a.n * a.Hkv * a.nsplit), NT, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention(const AttnArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  if (a.nsplit < 1) return cudaErrorInvalidValue;
  const bool f32 = a.kv_f32 != 0;
  if (a.D == 128 && a.G == 4) return f32 ? launch_t<128, 4, true>(a, s) : launch_t<128, 4, false>(a, s);
  if (a.D == 128 && a.G == 2) return f32 ? launch_t<128, 2, true>(a, s) : launch_t<128, 2, false>(a, s);
  if (a.D == 64 && a.G == 4) return f32 ? launch_t<64, 4, true>(a, s) : launch_t<64, 4, false>(a, s);
  if (a.D == 64 && a.G == 2) return f32 ? launch_t<64, 2, true>(a, s) : launch_t<64, 2, false>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
