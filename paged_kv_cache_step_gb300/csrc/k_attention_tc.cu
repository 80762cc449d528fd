// Decode attention over the paged cache with the summary update fused in,
// tensor-core variant (tcgen05, sm_103a), for bf16 caches with d = 128 and
// G = 2 or 4 query heads per KV head: the integration point of GrowPage
// Sec. 4.1, where the decode attention kernel updates the query summaries
// as a side effect, for one layer of a decode step.
//
// The work split and the outputs are those of the CUDA-core kernel
// (k_attention.cu): one CTA per (request, KV head, split of the request's
// attended pages); the split-0 CTA updates the G heads' summaries (Eq. 6,
// App. E.1); each split writes (max, sum, G x d) partials and the last CTA
// of a (request, KV head) merges them.  Within a CTA the split's keys are
// taken in tiles of 128:
//   S   = K q~^T   M = 128 keys, N = 16, K = d: the G rotated, scaled query
//                  rows, each split into three bf16 parts h1 + h2 + h3 that
//                  carry its fp32 value (so K . q~ is computed to fp32
//                  precision from bf16 operands), rows part * G + g;
//   P   = 2^(S - m) online softmax per head in base 2 (CUDA cores), the
//                  fp32 weights split into three bf16 parts the same way;
//   O_t = V^T P^T  M = d = 128, N = 16, K = 128 keys, V^T read MN-major
//                  straight from the TMA tile;
//   out = out * 2^(m_prev - m) + O_t  (CUDA cores, fp32).
// Roles (12 warps; one CTA per SM, its shared memory holds three tiles of K
// and V in flight):
//   warp 0      producer: K and V tiles (box 64 x 128, 128-byte swizzle)
//               through an NSTAGE ring;
//   warp 1      MMA issuer: S of tile t, then O of tile t - 1 once its P is
//               in shared memory, so the score MMA of the next tile runs
//               while the softmax of this one is computed;
//   warps 2-3   query: summary update, RoPE, the operand q~; then idle;
//   warps 4-7   softmax: thread = key (TMEM lane), P into the slot's operand;
//   warps 8-11  correction: thread = dimension d (TMEM lane), running output.
// TMEM holds NS slots of 32 columns: S (16) and O_t (16) of one tile.
// Every wait is bounded: on expiry the CTA records ERR_TIMEOUT, raises an
// abort flag that ends every role's loop, waits (bounded) for its copies and
// MMAs in flight, frees its TMEM and returns without writing a partial.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "gp_kernels.h"
#include "tc_ptx.cuh"

namespace gp {
namespace {

using namespace tc;

constexpr int NT = 384;
constexpr int W_Q0 = 2;     // query warps 2..3
constexpr int NQ_THR = 64;
constexpr int W_SM0 = 4;    // softmax warps 4..7 (TMEM lane quadrants 0..3)
constexpr int W_CR0 = 8;    // correction warps 8..11
constexpr int BAR_Q = 1;    // named barriers
constexpr int BAR_SM = 2;
constexpr int PAGE = 256;
constexpr int D = 128;
constexpr int TK = 128;              // keys per tile
constexpr int NSTAGE = 3;            // K and V tiles in flight
constexpr int NS = 4;                // TMEM slots
constexpr int TMEM_COLS = 128;       // NS x 32, a power of two
constexpr int NB = 16;               // MMA N: three bf16 parts x G heads, padded
constexpr int HALF = TK * 128;       // one 64-element span of a tile: 128 rows x 128 bytes
constexpr int KBYTES = 2 * HALF;     // a K (or V) tile
constexpr int STAGE = 2 * KBYTES;    // K tile, then V tile
constexpr int OPB = 2 * NB * 128;    // a B operand: two 64-element spans of NB rows
constexpr float NEG = -1.0e30f;
constexpr long long kWaitLimit = 1ll << 31;  // clock cycles (about one second)
static_assert(NS * 32 <= TMEM_COLS, "TMEM slots");

// f32 accumulator, bf16 A and B, N = 16, M = 128; A K-major (S) or MN-major (O).
constexpr uint32_t IDESC_QK = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NB >> 3) << 17) |
                              ((uint32_t)(128 >> 4) << 24);
constexpr uint32_t IDESC_PV = IDESC_QK | (1u << 15);

// Shared memory after aligning the dynamic base to 1 KiB.
template <int G>
struct Sm {
  static constexpr size_t ST = 0;                                 // [NSTAGE] K tile, V tile
  static constexpr size_t QB = ST + (size_t)NSTAGE * STAGE;       // operand q~
  static constexpr size_t PB = QB + OPB;                          // [NS] operands P
  static constexpr size_t QS = PB + (size_t)NS * OPB;             // float [G][D] queries
  static constexpr size_t RED = QS + sizeof(float) * G * D;       // float [2][4][G] tile maxima
  static constexpr size_t SCL = RED + sizeof(float) * 8 * G;      // float [NS][G] rescale factors
  static constexpr size_t FIN = SCL + sizeof(float) * NS * G;     // float [4][G] sums, [G] maxima
  static constexpr size_t BARS = (FIN + sizeof(float) * 5 * G + 7) & ~size_t(7);
  // full[NSTAGE], empty[NSTAGE], qready, mmadone, sready[NS], pready[NS], oready[NS], sfree[NS]
  static constexpr int NBARS = 2 * NSTAGE + 2 + 4 * NS;
  static constexpr size_t MISC = BARS + 8 * (size_t)NBARS;        // ints: TMEM base, flags
  static constexpr size_t BYTES = MISC + 64 + 1024;               // + alignment slack
};

// Byte offset of element (k, n) of a K-major B operand with NB rows of 128-key
// (or 128-dimension) extent: two 64-element spans, 128 bytes per row,
// 16-byte chunks swizzled by the row within each group of 8.
__device__ __forceinline__ uint32_t op_off(int k, int n) {
  return (uint32_t)((k >> 6) * (NB * 128) + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ void st_bf16(unsigned char* base, uint32_t off, __nv_bfloat16 v) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = v;
}

// Three bf16 parts of x whose sum carries x to fp32 precision.
__device__ __forceinline__ void split3(float x, __nv_bfloat16& h1, __nv_bfloat16& h2, __nv_bfloat16& h3) {
  h1 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h1);
  h2 = __float2bfloat16_rn(r1);
  h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
}

// Bounded wait; gives up when the limit passes or *abort is set.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitLimit) return false;
  }
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int G>
__global__ void __launch_bounds__(NT, 1) k_decode_attn_tc(const __grid_constant__ AttnArgs a) {
  using L = Sm<G>;
  static_assert(3 * G <= NB, "three parts per head fit the MMA N");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
  float* qs = reinterpret_cast<float*>(sm + L::QS);
  float* red = reinterpret_cast<float*>(sm + L::RED);
  float* scl = reinterpret_cast<float*>(sm + L::SCL);
  float* fin = reinterpret_cast<float*>(sm + L::FIN);
  int* misc = reinterpret_cast<int*>(sm + L::MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = misc + 1;
  volatile int* sm_fail = misc + 2;  // [2] a softmax warp's wait gave up, by tile parity
  int* s_last = misc + 4;
  const uint32_t bar0 = sb + (uint32_t)L::BARS;
  const uint32_t qready = bar0 + 8u * (2 * NSTAGE), mmadone = qready + 8u;
  auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(NSTAGE + s); };
  auto sready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + j); };
  auto pready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + NS + j); };
  auto oready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + 2 * NS + j); };
  auto sfree = [&](int j) { return mmadone + 8u * (uint32_t)(1 + 3 * NS + j); };

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
  const int T = span > 0 ? (span + TK - 1) / TK : 0;  // tiles of this split
  const int slot = rq.slot;
  if (slot < 0 || slot >= a.M) {
    if (tid == 0) atomicOr(a.err, ERR_BAD_SLOT);
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < L::NBARS; ++i) {
      uint32_t cnt = 1;                                                      // one arrival (copy or commit)
      if (i >= 2 * NSTAGE + 2 + NS && i < 2 * NSTAGE + 2 + 2 * NS) cnt = 4;  // pready: the softmax warps
      if (i >= 2 * NSTAGE + 2 + 3 * NS) cnt = 8;                             // sfree: softmax and correction
      mbar_init(bar0 + 8u * (uint32_t)i, cnt);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort = 0;
    sm_fail[0] = 0;
    sm_fail[1] = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(tmem_holder))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  float acc[G];  // correction warps: the running output of dimension d
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = 0.f;

  if (warp == 0) {
    // ---- producer ------------------------------------------------------------
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      const size_t layer_rows = (size_t)a.layer * a.num_pages_total;
      for (int t = 0; t < T; ++t) {
        const int s = t % NSTAGE;
        if (t >= NSTAGE && !(ok = wait_bar(empty(s), (uint32_t)(((t / NSTAGE) - 1) & 1), abort))) break;
        int pg = a.bt[rq.bt_off + p0 + (t >> 1)];
        if (pg < 0 || pg >= a.num_pages_total) {
          atomicOr(a.err, ERR_BAD_PAGE);
          pg = 0;
        }
        const int y = (int)(((layer_rows + (size_t)pg) * a.Hkv + h) * PAGE + (t & 1) * TK);
        const uint32_t dst = sb + (uint32_t)(L::ST + (size_t)s * STAGE);
        mbar_expect_tx(full(s), STAGE);
        tma_load_2d(dst, &a.kmap, 0, y, full(s));
        tma_load_2d(dst + HALF, &a.kmap, 64, y, full(s));
        tma_load_2d(dst + KBYTES, &a.vmap, 0, y, full(s));
        tma_load_2d(dst + KBYTES + HALF, &a.vmap, 64, y, full(s));
        issued = t + 1;
      }
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
      }
      // every copy issued has landed before the CTA moves on (bounded)
      const int zero = 0;
      for (int t = issued > NSTAGE ? issued - NSTAGE : 0; t < issued; ++t)
        wait_bar(full(t % NSTAGE), (uint32_t)((t / NSTAGE) & 1), &zero);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------
    if (lane == 0) {
      const uint32_t qb = sb + (uint32_t)L::QB;
      // O of tile u: V^T (MN-major, the second d span 16 KiB on) times P^T
      auto pv = [&](int u) -> bool {
        const int j = u % NS, s = u % NSTAGE;
        if (!wait_bar(pready(j), (uint32_t)((u / NS) & 1), abort)) return false;
        tc_fence_after();
        const uint32_t v0 = sb + (uint32_t)(L::ST + (size_t)s * STAGE + KBYTES);
        const uint32_t pb = sb + (uint32_t)(L::PB + (size_t)j * OPB);
#pragma unroll
        for (int k = 0; k < TK / 16; ++k)
          mma_f16(tmem + (uint32_t)(j * 32 + 16), sw128_mn_desc(v0 + (uint32_t)k * 2048u, HALF),
                  sw128_desc(pb + (uint32_t)((k >> 2) * (NB * 128) + (k & 3) * 32)), IDESC_PV, k > 0 ? 1u : 0u);
        mma_commit(oready(j));
        mma_commit(empty(s));  // the stage's K and V are read
        return true;
      };
      bool ok = wait_bar(qready, 0u, abort);
      for (int t = 0; ok && t < T; ++t) {
        const int j = t % NS, s = t % NSTAGE;
        if (t >= NS && !(ok = wait_bar(sfree(j), (uint32_t)(((t / NS) - 1) & 1), abort))) break;
        if (!(ok = wait_bar(full(s), (uint32_t)((t / NSTAGE) & 1), abort))) break;
        tc_fence_after();
        const uint32_t k0 = sb + (uint32_t)(L::ST + (size_t)s * STAGE);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_f16(tmem + (uint32_t)(j * 32), sw128_desc(k0 + (uint32_t)((k >> 2) * HALF + (k & 3) * 32)),
                  sw128_desc(qb + (uint32_t)((k >> 2) * (NB * 128) + (k & 3) * 32)), IDESC_QK, k > 0 ? 1u : 0u);
        mma_commit(sready(j));
        if (t >= 1) ok = pv(t - 1);
      }
      if (ok && T > 0) ok = pv(T - 1);
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
      }
      // every MMA issued has completed before TMEM is released (bounded)
      mma_commit(mmadone);
      const int zero = 0;
      wait_bar(mmadone, 0u, &zero);
    }
    __syncwarp();
  } else if (warp < W_SM0) {
    // ---- query: summary update (split 0), RoPE, the operand q~ ---------------
    const int qt = tid - 32 * W_Q0;
    unsigned char* qb = sm + L::QB;
    unsigned char* pbuf = sm + L::PB;
    for (int e = qt; e < G * D; e += NQ_THR) {
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
      qs[gi * D + d] = (float)qv;
    }
    // the padding rows of the operands (q~ and every slot's P) are zero
    for (int e = qt; e < (NB - 3 * G) * D; e += NQ_THR) {
      const int n = 3 * G + e / D, k = e % D;
      st_bf16(qb, op_off(k, n), __float2bfloat16_rn(0.f));
#pragma unroll
      for (int j = 0; j < NS; ++j) st_bf16(pbuf + (size_t)j * OPB, op_off(k, n), __float2bfloat16_rn(0.f));
    }
    asm volatile("bar.sync %0, %1;" ::"n"(BAR_Q), "n"(NQ_THR) : "memory");
    // rotate-half RoPE at the request's position (pairs (i, i + D/2)) and the
    // log2(e)/sqrt(d) scale, then the three bf16 parts: rows gi, G + gi, 2G + gi
    const float sc = 1.4426950408889634f / sqrtf((float)D);
    for (int e = qt; e < G * (D / 2); e += NQ_THR) {
      const int gi = e / (D / 2), i = e % (D / 2);
      const double ang = (double)rq.pos * a.inv_freq[i];
      const double kk = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
      double red2 = fma(-kk, 6.283185307179586, ang);     // 2 pi, high part
      red2 = fma(-kk, 2.4492935982947064e-16, red2);      // 2 pi, low part
      float sn, cs;
      sincosf((float)red2, &sn, &cs);
      const float x1 = qs[gi * D + i], x2 = qs[gi * D + i + D / 2];
      const float o[2] = {sc * fmaf(x1, cs, -x2 * sn), sc * fmaf(x2, cs, x1 * sn)};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int d = i + hf * (D / 2);
        __nv_bfloat16 h1, h2, h3;
        split3(o[hf], h1, h2, h3);
        st_bf16(qb, op_off(d, gi), h1);
        st_bf16(qb, op_off(d, G + gi), h2);
        st_bf16(qb, op_off(d, 2 * G + gi), h3);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
    asm volatile("bar.sync %0, %1;" ::"n"(BAR_Q), "n"(NQ_THR) : "memory");
    if (qt == 0) mbar_arrive(qready);
  } else if (warp < W_CR0) {
    // ---- softmax: thread = key of the tile -------------------------------------
    const int quad = warp & 3, key = 32 * quad + lane;
    const uint32_t lanes = (uint32_t)(32 * quad) << 16;
    unsigned char* pbuf = sm + L::PB;
    float m[G], ssum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = NEG;
      ssum[g] = 0.f;
    }
    for (int t = 0; t < T; ++t) {
      const int j = t % NS;
      const bool ok = __all_sync(0xffffffffu, wait_bar(sready(j), (uint32_t)((t / NS) & 1), abort));
      float v[16];
      if (ok) {
        tc_fence_after();
        tmem_ld<16>(tmem + lanes + (uint32_t)(j * 32), v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree(j));  // S is read
      } else if (lane == 0) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
        sm_fail[t & 1] = 1;
      }
      const bool in_range = p0 * PAGE + t * TK + key < ntok;
      const bool valid = ok && in_range;
      if (ok && !in_range) {
        // a slot past the attended tokens (ragged last tile): its weight is 0,
        // but the cache may hold any bits there, and 0 x inf or NaN would
        // reach the output through the MMA; its V row is zeroed instead.  The
        // tile has landed (the score MMA read it), and the stage cannot be
        // reloaded before this tile's P is released.
        const int s = t % NSTAGE;
        wait_bar(full(s), (uint32_t)((t / NSTAGE) & 1), abort);
        unsigned char* vrow = sm + L::ST + (size_t)s * STAGE + KBYTES + (size_t)key * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          reinterpret_cast<uint4*>(vrow)[c] = make_uint4(0u, 0u, 0u, 0u);
          reinterpret_cast<uint4*>(vrow + HALF)[c] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float z[G], wm[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        z[g] = valid ? v[g] + (v[G + g] + v[2 * G + g]) : NEG;
        wm[g] = z[g];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) wm[g] = fmaxf(wm[g], __shfl_xor_sync(0xffffffffu, wm[g], o));
      if (lane == 0)
#pragma unroll
        for (int g = 0; g < G; ++g) red[((t & 1) * 4 + quad) * G + g] = wm[g];
      asm volatile("bar.sync %0, %1;" ::"n"(BAR_SM), "n"(128) : "memory");
      if (sm_fail[t & 1]) break;  // written only before the barrier: every softmax thread agrees
      unsigned char* pb = pbuf + (size_t)j * OPB;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float tm = red[((t & 1) * 4) * G + g];
#pragma unroll
        for (int q = 1; q < 4; ++q) tm = fmaxf(tm, red[((t & 1) * 4 + q) * G + g]);
        const float mn = fmaxf(m[g], tm);
        const float rs = ex2f(m[g] - mn);
        m[g] = mn;
        const float p = valid ? ex2f(z[g] - mn) : 0.f;
        ssum[g] = fmaf(ssum[g], rs, p);
        if (warp == W_SM0 && lane == 0) scl[j * G + g] = rs;
        __nv_bfloat16 h1, h2, h3;
        split3(p, h1, h2, h3);
        st_bf16(pb, op_off(key, g), h1);
        st_bf16(pb, op_off(key, G + g), h2);
        st_bf16(pb, op_off(key, 2 * G + g), h3);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P (and zeroed V rows) visible to the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(pready(j));
    }
    // the sums of this warp's keys, and the final maxima
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float s = ssum[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) fin[quad * G + g] = s;
      if (warp == W_SM0 && lane == 0) fin[4 * G + g] = m[g];
    }
  } else {
    // ---- correction: thread = dimension d --------------------------------------
    const int quad = warp & 3;
    const uint32_t lanes = (uint32_t)(32 * quad) << 16;
    for (int t = 0; t < T; ++t) {
      const int j = t % NS;
      bool ok = __all_sync(0xffffffffu, wait_bar(pready(j), (uint32_t)((t / NS) & 1), abort));
      float rs[G];
      if (ok) {
#pragma unroll
        for (int g = 0; g < G; ++g) rs[g] = scl[j * G + g];
        ok = __all_sync(0xffffffffu, wait_bar(oready(j), (uint32_t)((t / NS) & 1), abort));
      }
      if (!ok) {
        if (lane == 0) {
          atomicOr(a.err, ERR_TIMEOUT);
          *abort = 1;
        }
        break;
      }
      tc_fence_after();
      float o[16];
      tmem_ld<16>(tmem + lanes + (uint32_t)(j * 32 + 16), o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree(j));  // O_t is read
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = fmaf(acc[g], rs[g], o[g] + (o[G + g] + o[2 * G + g]));
    }
  }

  // ---- every role is done: TMEM back, the split's partial out ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
  if (*abort) return;  // set only before the barrier above: the whole CTA agrees
  float* po = a.part + (size_t)(part_first + split) * G * (D + 2);
  if (warp >= W_CR0) {
    const int d = 32 * (warp & 3) + lane;
#pragma unroll
    for (int g = 0; g < G; ++g) po[g * (D + 2) + d] = acc[g];
  }
  if (tid < G) {
    const float den = fin[tid] + fin[G + tid] + fin[2 * G + tid] + fin[3 * G + tid];
    po[tid * (D + 2) + D] = fin[4 * G + tid];
    po[tid * (D + 2) + D + 1] = den;
  }
  // ---- the last split of (request, KV head) merges ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(a.tickets + (size_t)r * a.Hkv + h, 1u);
    *s_last = old == (unsigned)(nsp - 1);
    if (*s_last) __threadfence();
  }
  __syncthreads();
  if (!*s_last) return;
  const float* pbs = a.part + (size_t)part_first * G * (D + 2);
  for (int e = tid; e < G * D; e += NT) {
    const int gi = e / D, d = e % D;
    float M = NEG;
    for (int sp = 0; sp < nsp; ++sp) M = fmaxf(M, __ldcg(pbs + ((size_t)sp * G + gi) * (D + 2) + D));
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
      const float* q = pbs + ((size_t)sp * G + gi) * (D + 2);
      const float mq = __ldcg(q + D);
      const float w = mq > 0.5f * NEG ? ex2f(mq - M) : 0.f;
      num = fmaf(w, __ldcg(q + d), num);
      den = fmaf(w, __ldcg(q + D + 1), den);
    }
    a.out[((size_t)r * a.Hq + h * G + gi) * D + d] = den > 0.f ? num / den : 0.f;
  }
}

template <int G>
cudaError_t launch_tc(const AttnArgs& a, cudaStream_t s) {
  constexpr size_t smem = Sm<G>::BYTES;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_decode_attn_tc<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_decode_attn_tc<G><<<dim3((unsigned)a.n_ctas), NT, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention_tc(const AttnArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  if (a.n_ctas < a.n * a.Hkv || !a.tc || a.kv_f32 || !attention_tc_shape(a.D, a.G)) return cudaErrorInvalidValue;
  return a.G == 4 ? launch_tc<4>(a, s) : launch_tc<2>(a, s);
}

}  // namespace gp
