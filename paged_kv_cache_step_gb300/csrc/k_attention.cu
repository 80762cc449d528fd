// Decode attention over the paged cache with the summary update fused in:
// the integration point of GrowPage Sec. 4.1, where the decode attention
// kernel updates the query summaries as a side effect, for one layer of a
// decode step.
//
// Per request r and query head g (KV head h = g / G):
//   summaries (Eq. 6, App. E.1): on the slot's first step both are q;
//     else qbar^x <- beta_x qbar^x + (1 - beta_x) q, with q the pre-RoPE query;
//   attention: z_i = RoPE_pos(q) . k_i / sqrt(d) over the request's first
//     num_tokens cached tokens (keys are stored rotated), a = softmax(z),
//     out = sum_i a_i v_i (fp32).
//
// Work: one CTA per (request, KV head, split of the request's attended
// pages), 256 threads, two CTAs per SM.  The host sizes the splits by pages
// and orders the requests longest first.  The split-0 CTA also updates the
// G heads' summaries from the query it loads anyway.
//   copies  -- one thread streams stages of 16 KB of K rows and the same V
//              rows into a ring of three shared-memory stages with bulk async
//              copies (a page's rows of one head are contiguous);
//   compute -- a key row is read by D/8 lanes, each owning 8 dimensions, so
//              the lanes of a quarter warp read 128 contiguous bytes.  Each
//              group of D/8 lanes keeps its own online softmax (base 2) over
//              its rows: logits by a shuffle reduction over the group, one
//              rescale per stage, then the weighted V rows.
// The key groups merge in shared memory; the splits write (max, sum, G x d)
// partials to scratch and the last CTA of a (request, KV head) merges them.
// Bounded by HBM: K and V are read once.
#include <cuda_bf16.h>

#include <cstdint>

#include "attn_kernels.h"
#include "gp_kernels.h"

namespace gp {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int PAGE = 256;
constexpr int NSTAGE = 3;                    // stages in flight per CTA
constexpr int TBYTES = 16 * 1024;            // K (and V) bytes of one stage
constexpr int STAGE = 2 * TBYTES;
constexpr float NEGF = -1.0e30f;
constexpr long long kWaitLimit = 1ll << 31;  // clock cycles (about one second)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase of an mbarrier; false when the limit passed.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  if (bar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!bar_try(bar, parity))
    if (clock64() - t0 > kWaitLimit) return false;
  return true;
}
__device__ __forceinline__ float bf_lo(unsigned u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(unsigned u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Dimension t (0..7) of the 8 that lane c of a key group owns: one 16-byte
// piece of a bf16 row, or two 16-byte pieces of an fp32 row (one in each
// half), so that the lanes of a quarter warp always read contiguous bytes.
template <int D, bool F32>
__device__ __forceinline__ int lane_dim(int c, int t) {
  if constexpr (F32) return t < 4 ? 4 * c + t : D / 2 + 4 * c + (t - 4);
  else return 8 * c + t;
}
template <int D, bool F32>
__device__ __forceinline__ void load_row(const unsigned char* row, int c, float f[8]) {
  if constexpr (F32) {
    const float4 x0 = *reinterpret_cast<const float4*>(row + c * 16);
    const float4 x1 = *reinterpret_cast<const float4*>(row + (c + D / 8) * 16);
    f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w;
    f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(row + c * 16);
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
  }
}

template <int D, int G, bool F32>
__global__ void __launch_bounds__(NT, 2) k_decode_attn(AttnArgs a) {
  constexpr int RB = F32 ? 4 * D : 2 * D;  // bytes of a cached row
  constexpr int SR = TBYTES / RB;          // rows of a stage
  constexpr int NCH = D / 8;               // lanes of a key group
  constexpr int KG = NWARP * (32 / NCH);   // key groups of the CTA
  constexpr int UK = SR / KG;              // rows of a stage per key group
  static_assert(PAGE % SR == 0 && SR % KG == 0 && UK >= 1, "stage shape");
  static_assert(KG * G * (D + 2) * 4 <= NSTAGE * STAGE, "the group merge fits in the ring");
  __shared__ float qs[G][D];  // rotated query rows, scaled by log2(e)/sqrt(d)
  __shared__ __align__(8) uint64_t full_bar[NSTAGE];
  __shared__ int s_last;
  extern __shared__ __align__(128) unsigned char ring[];  // NSTAGE x (K rows, V rows)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- this CTA's (request, KV head, split); requests in the host's order ----
  int lo = 0, hi = a.n;  // split_base[lo] <= blockIdx.x < split_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.split_base[mid] <= (int)blockIdx.x) lo = mid;
    else hi = mid;
  }
  const int r = a.order[lo];
  const int nsp = (a.split_base[lo + 1] - a.split_base[lo]) / a.Hkv;
  const int local = (int)blockIdx.x - a.split_base[lo];
  const int h = local % a.Hkv, split = local / a.Hkv;
  const int part_first = a.split_base[lo] + h * nsp;  // partials of (r, h): nsp from here
  const DevReq rq = a.reqs[r];
  const int ntok = a.ntok[r];
  const int npg = (ntok + PAGE - 1) / PAGE;  // pages attended
  const int p0 = (split * npg) / nsp, p1 = ((split + 1) * npg) / nsp;
  const int span = min(ntok - p0 * PAGE, (p1 - p0) * PAGE);
  const int T = span > 0 ? (span + SR - 1) / SR : 0;  // stages of this split
  const int slot = rq.slot;
  if (slot < 0 || slot >= a.M) {
    if (tid == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }

  const unsigned char* kc = static_cast<const unsigned char*>(a.k_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(a.v_cache);
  const size_t head_stride = (size_t)PAGE * RB;
  int issued = 0;  // stages handed to the copy engine (thread 0)
  // thread 0 streams stage k (rows [k SR, k SR + SR) of the split) into buffer k % NSTAGE
  auto issue = [&](int k) {
    const uint32_t bar = smem_addr(&full_bar[k % NSTAGE]);
    const int j = p0 + (k * SR) / PAGE;
    const int pg = a.bt[rq.bt_off + j];
    bool ok = pg >= 0 && pg < a.num_pages_total;
    size_t off = 0;
    if (ok) {
      off = (((size_t)a.layer * a.num_pages_total + pg) * a.Hkv + h) * head_stride + (size_t)((k * SR) % PAGE) * RB;
      ok = ((reinterpret_cast<uintptr_t>(kc + off) | reinterpret_cast<uintptr_t>(vc + off)) & 15) == 0;
    }
    ++issued;
    if (!ok) {
      // a bad page: record it and complete the phase without data
      atomicOr(a.err, ERR_BAD_PAGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      return;
    }
    const uint32_t dst = smem_addr(ring + (size_t)(k % NSTAGE) * STAGE);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)STAGE) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(kc + off), "r"((uint32_t)TBYTES), "r"(bar)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst + (uint32_t)TBYTES),
                 "l"(vc + off), "r"((uint32_t)TBYTES), "r"(bar)
                 : "memory");
  };
  if (tid == 0) {
    for (int st = 0; st < NSTAGE; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full_bar[st])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // the stage barriers exist before any copy or wait uses them
  if (tid == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int k = 0; k < NSTAGE && k < T; ++k) issue(k);
  }

  // ---- query rows: summary update (split 0) and RoPE, while the copies fly ----
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
  // rotate-half RoPE at the request's position: pairs (i, i + D/2)
  for (int e = tid; e < G * (D / 2); e += NT) {
    const int gi = e / (D / 2), i = e % (D / 2);
    const double ang = (double)rq.pos * a.inv_freq[i];
    const double kk = rint(ang * 0.15915494309189535);
    double red2 = fma(-kk, 6.283185307179586, ang);
    red2 = fma(-kk, 2.4492935982947064e-16, red2);
    float sn, cs;
    sincosf((float)red2, &sn, &cs);
    const float x1 = qs[gi][i], x2 = qs[gi][i + D / 2];
    const float sc = 1.4426950408889634f / sqrtf((float)D);
    qs[gi][i] = sc * fmaf(x1, cs, -x2 * sn);
    qs[gi][i + D / 2] = sc * fmaf(x2, cs, x1 * sn);
  }
  __syncthreads();

  const int c = lane % NCH;                        // lane within the key group
  const int grp = warp * (32 / NCH) + lane / NCH;  // key group: rows grp, grp + KG, ... of a stage
  float qr[G][8], acc[G][8], m[G], s[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = NEGF;
    s[g] = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      qr[g][t] = qs[g][lane_dim<D, F32>(c, t)];
      acc[g][t] = 0.f;
    }
  }

  // ---- the stages: logits, online softmax per key group, weighted values ----
  int k = 0;
  bool aborted = false;
  for (; k < T; ++k) {
    const int st = k % NSTAGE;
    const bool ok = bar_wait(smem_addr(&full_bar[st]), (uint32_t)((k / NSTAGE) & 1));
    if (__syncthreads_or(!ok)) {  // every thread leaves together
      aborted = true;
      break;
    }
    // every thread is done with stage k - 1: its buffer takes stage k - 1 + NSTAGE
    if (tid == 0 && k >= 1 && k - 1 + NSTAGE < T) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(k - 1 + NSTAGE);
    }
    const unsigned char* sk = ring + (size_t)st * STAGE;
    const unsigned char* sv = sk + TBYTES;
    const int nval = min(SR, ntok - (p0 * PAGE + k * SR));  // rows of the stage that hold tokens
    float z[UK][G];
#pragma unroll
    for (int u = 0; u < UK; ++u) {
      float f[8];
      load_row<D, F32>(sk + (size_t)(grp + KG * u) * RB, c, f);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float dot = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) dot = fmaf(qr[g][t], f[t], dot);
        z[u][g] = dot;
      }
    }
    // the group's lanes are aligned on NCH, so xor partners stay inside it
#pragma unroll
    for (int o = NCH / 2; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < UK; ++u)
#pragma unroll
        for (int g = 0; g < G; ++g) z[u][g] += __shfl_xor_sync(0xffffffffu, z[u][g], o);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = NEGF;
#pragma unroll
      for (int u = 0; u < UK; ++u)
        if (grp + KG * u < nval) mx = fmaxf(mx, z[u][g]);
      const float mn = fmaxf(m[g], mx);
      const float sc = ex2f(m[g] - mn);
      m[g] = mn;
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < UK; ++u) {
        const float w = grp + KG * u < nval ? ex2f(z[u][g] - mn) : 0.f;
        z[u][g] = w;
        sum += w;
      }
      s[g] = fmaf(s[g], sc, sum);
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[g][t] *= sc;
    }
#pragma unroll
    for (int u = 0; u < UK; ++u) {
      if (grp + KG * u < nval) {
        float f[8];
        load_row<D, F32>(sv + (size_t)(grp + KG * u) * RB, c, f);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int t = 0; t < 8; ++t) acc[g][t] = fmaf(z[u][g], f[t], acc[g][t]);
      }
    }
  }
  if (aborted) {
    // copies still in flight land before the CTA's shared memory goes away (bounded)
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      for (int q = k; q < issued; ++q) bar_wait(smem_addr(&full_bar[q % NSTAGE]), (uint32_t)((q / NSTAGE) & 1));
    }
    return;
  }

  // ---- merge the key groups (the ring is free: every copy has landed) ----
  __syncthreads();
  float* red = reinterpret_cast<float*>(ring);  // [KG][G][D] partial outputs
  float* rms = red + KG * G * D;                 // [KG][G] (max, sum)
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int t = 0; t < 8; ++t) red[((size_t)grp * G + g) * D + lane_dim<D, F32>(c, t)] = acc[g][t];
    if (c == 0) {
      rms[(grp * G + g) * 2] = m[g];
      rms[(grp * G + g) * 2 + 1] = s[g];
    }
  }
  __syncthreads();
  float* po = a.part + (size_t)(part_first + split) * G * (D + 2);
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    float M = NEGF;
    for (int q = 0; q < KG; ++q) M = fmaxf(M, rms[(q * G + gi) * 2]);
    float num = 0.f, den = 0.f;
    for (int q = 0; q < KG; ++q) {
      const float mq = rms[(q * G + gi) * 2];
      const float w = mq > 0.5f * NEGF ? ex2f(mq - M) : 0.f;
      num = fmaf(w, red[((size_t)q * G + gi) * D + d], num);
      den = fmaf(w, rms[(q * G + gi) * 2 + 1], den);
    }
    po[gi * (D + 2) + d] = num;
    if (d == 0) {
      po[gi * (D + 2) + D] = M;
      po[gi * (D + 2) + D + 1] = den;
    }
  }
  // ---- the last split of (request, KV head) merges ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(a.tickets + (size_t)r * a.Hkv + h, 1u);
    s_last = old == (unsigned)(nsp - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  const float* pb = a.part + (size_t)part_first * G * (D + 2);
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    float M = NEGF;
    for (int sp = 0; sp < nsp; ++sp) M = fmaxf(M, __ldcg(pb + ((size_t)sp * G + gi) * (D + 2) + D));
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
      const float* q = pb + ((size_t)sp * G + gi) * (D + 2);
      const float mq = __ldcg(q + D);
      const float w = mq > 0.5f * NEGF ? ex2f(mq - M) : 0.f;
      num = fmaf(w, __ldcg(q + d), num);
      den = fmaf(w, __ldcg(q + D + 1), den);
    }
    a.out[((size_t)r * a.Hq + h * G + gi) * D + d] = den > 0.f ? num / den : 0.f;
  }
}

template <int D, int G, bool F32>
cudaError_t launch_t(const AttnArgs& a, cudaStream_t s) {
  constexpr int smem = NSTAGE * STAGE;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(k_decode_attn<D, G, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_decode_attn<D, G, F32><<<dim3(a.n_ctas), NT, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention(const AttnArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  if (a.tc) return launch_decode_attention_tc(a, s);
  if (a.n_ctas < a.n * a.Hkv) return cudaErrorInvalidValue;
  const bool f32 = a.kv_f32 != 0;
  if (a.D == 128 && a.G == 4) return f32 ? launch_t<128, 4, true>(a, s) : launch_t<128, 4, false>(a, s);
  if (a.D == 128 && a.G == 2) return f32 ? launch_t<128, 2, true>(a, s) : launch_t<128, 2, false>(a, s);
  if (a.D == 64 && a.G == 4) return f32 ? launch_t<64, 4, true>(a, s) : launch_t<64, 4, false>(a, s);
  if (a.D == 64 && a.G == 2) return f32 ? launch_t<64, 2, true>(a, s) : launch_t<64, 2, false>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
