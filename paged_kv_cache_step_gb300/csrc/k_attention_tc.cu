// Decode attention over the paged cache with the summary update fused in,
// tensor-core variant (tcgen05, sm_103a), for bf16 caches with d = 128 and
// G = 2 or 4 query heads per KV head: the integration point of GrowPage
// Sec. 4.1, where the decode attention kernel updates the query summaries
// as a side effect, for one layer of a decode step.
//
// The outputs are those of the CUDA-core kernel (k_attention.cu); the work
// is split differently.  The grid is persistent, one CTA per SM: the host
// lays every (request, KV head) pair's attended pages end to end, cuts them
// into one even range per SM, and gives each CTA the items of its range --
// whole pairs, and at most two pieces of pairs it shares with its
// neighbours.  The first piece of a pair updates the G heads' summaries
// (Eq. 6, App. E.1); a pair in one piece writes its output directly, the
// pieces of a shared pair write (max, sum, G x d) partials and the last of
// them to finish merges them.  Every role runs on into the next item, so the
// copies of the next piece stream while this one finishes.  Within an item
// the keys are taken in tiles of 128:
//   S   = K q~^T   M = 128 keys, N = 16, K = d: the G rotated, scaled query
//                  rows, each split into three bf16 parts h1 + h2 + h3 that
//                  carry its fp32 value (so K . q~ is computed to fp32
//                  precision from bf16 operands), rows part * G + g;
//   P   = 2^(S - m) online softmax per head in base 2 (CUDA cores), the
//                  fp32 weights split into three bf16 parts the same way;
//   O_t = V^T P^T  M = d = 128, N = 16, K = 128 keys, V^T read MN-major
//                  straight from the TMA tile;
//   out = out * 2^(m_prev - m) + O_t  (CUDA cores, fp32), and the sum alike.
// Roles (12 warps; one CTA per SM, its shared memory holds three tiles of K
// and V in flight):
//   warp 0      producer: K and V tiles (box 64 x 128, 128-byte swizzle)
//               through an NSTAGE ring, across items;
//   warp 1      MMA issuer: S of tile t, then O of tile t - 1 once its P is
//               in shared memory, so the score MMA of the next tile runs
//               while the softmax of this one is computed;
//   warps 2-3   query: summary update, RoPE and the operand q~ of the next
//               item, into one of two buffers;
//   warps 4-7   softmax: thread = key (TMEM lane); P into the slot's
//               operand, the tile's rescale factor, maximum and sums beside it;
//   warps 8-11  correction: thread = dimension d (TMEM lane); the running
//               output and sum, the item's partial, and (warp 8) the merge.
// TMEM holds NS slots of 32 columns: S (16) and O_t (16) of one tile.
// Every wait is bounded: on expiry the CTA records ERR_TIMEOUT, raises an
// abort flag that ends every role's loop, waits (bounded) for its copies and
// MMAs in flight, frees its TMEM and returns; the items it had not finished
// write no partial.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "attn_kernels.h"
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
constexpr int NEND = 8;              // item-end barriers (the correction warps run at most NS items apart)
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
  static constexpr size_t QB = ST + (size_t)NSTAGE * STAGE;       // [2] operands q~
  static constexpr size_t PB = QB + 2 * (size_t)OPB;              // [NS] operands P
  static constexpr size_t QS = PB + (size_t)NS * OPB;             // float [G][D] queries
  static constexpr size_t RED = QS + sizeof(float) * G * D;       // float [2][4][G] tile maxima
  static constexpr size_t SCL = RED + sizeof(float) * 8 * G;      // float [NS][G] rescale factors
  static constexpr size_t TSUM = SCL + sizeof(float) * NS * G;    // float [NS][4][G] per-warp tile sums
  static constexpr size_t TMAX = TSUM + sizeof(float) * NS * 4 * G;  // float [NS][G] maxima after the tile
  static constexpr size_t MW = TMAX + sizeof(float) * NS * G;    // float [64][G] merge weights (warp 8)
  static constexpr size_t BARS = (MW + sizeof(float) * 64 * G + 7) & ~size_t(7);
  // full[NSTAGE], empty[NSTAGE], qready[2], qfree[2], mmadone, sready[NS],
  // pready[NS], oready[NS], sfree[NS], endbar[NEND]
  static constexpr int NBARS = 2 * NSTAGE + 5 + 4 * NS + NEND;
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

// Work item i (the host's table), and whether its slot is in range.
struct Item {
  AttnItem w;
  bool ok;
};
__device__ __forceinline__ Item load_item(const AttnArgs& a, int i) {
  Item it;
  const int4* src = reinterpret_cast<const int4*>(a.items + i);
  const int4 x = __ldg(src), y = __ldg(src + 1), z = __ldg(src + 2);
  it.w.r = x.x;
  it.w.h = x.y;
  it.w.split = x.z;
  it.w.nsp = x.w;
  it.w.part_first = y.x;
  it.w.p0 = y.y;
  it.w.T = y.z;
  it.w.ntok = y.w;
  it.w.bt_off = z.x;
  it.w.slot = z.y;
  it.w.pos = (int64_t)(((uint64_t)(uint32_t)z.w << 32) | (uint32_t)z.z);
  it.ok = it.w.slot >= 0 && it.w.slot < a.M;
  return it;
}

// A partial of the tensor-core kernel: [G][D] outputs, then [G] maxima and
// [G] sums (the same G (D + 2) floats as the CUDA-core kernel's, laid out so
// that the outputs of every partial start on a 16-byte boundary).
template <int G>
constexpr int kPartFloats = G * (D + 2);

// The merged output of (request, KV head), by one warp: the last of its
// items to finish combines the nsp (<= 64) partials.  The per-head weights
// 2^(m_split - m) are computed once (into mw, [nsp][G] in shared memory);
// then each lane owns float4 pieces of the G x D outputs and keeps one load
// per split in flight for each.
template <int G>
__device__ __forceinline__ void merge_splits(const AttnArgs& a, const AttnItem& it, float* mw, int lane) {
  const float* base = a.part + (size_t)it.part_first * kPartFloats<G>;
  float M[G], den[G];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    M[gg] = NEG;
    den[gg] = 0.f;
  }
  for (int sp = lane; sp < it.nsp; sp += 32)
#pragma unroll
    for (int gg = 0; gg < G; ++gg) M[gg] = fmaxf(M[gg], __ldcg(base + (size_t)sp * kPartFloats<G> + G * D + gg));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int gg = 0; gg < G; ++gg) M[gg] = fmaxf(M[gg], __shfl_xor_sync(0xffffffffu, M[gg], o));
  for (int sp = lane; sp < it.nsp; sp += 32) {
    const float* ps = base + (size_t)sp * kPartFloats<G> + G * D;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const float mq = __ldcg(ps + gg);
      const float w = mq > 0.5f * NEG ? ex2f(mq - M[gg]) : 0.f;
      mw[sp * G + gg] = w;
      den[gg] = fmaf(w, __ldcg(ps + G + gg), den[gg]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int gg = 0; gg < G; ++gg) den[gg] += __shfl_xor_sync(0xffffffffu, den[gg], o);
  __syncwarp();
  constexpr int PIECES = G * D / 4 / 32;  // float4 pieces of the outputs per lane
  float4 acc[PIECES];
#pragma unroll
  for (int c = 0; c < PIECES; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  // two splits' loads in flight per step (the second is a repeat of the
  // first, with weight 0, when nsp is odd)
  for (int sp = 0; sp < it.nsp; sp += 2) {
    const int sq = sp + 1 < it.nsp ? sp + 1 : sp;
    const float4* s0 = reinterpret_cast<const float4*>(base + (size_t)sp * kPartFloats<G>);
    const float4* s1 = reinterpret_cast<const float4*>(base + (size_t)sq * kPartFloats<G>);
    float4 v0[PIECES], v1[PIECES];
#pragma unroll
    for (int c = 0; c < PIECES; ++c) {
      v0[c] = __ldcg(s0 + lane + 32 * c);
      v1[c] = __ldcg(s1 + lane + 32 * c);
    }
#pragma unroll
    for (int c = 0; c < PIECES; ++c) {
      const int gg = (4 * (lane + 32 * c)) / D;
      const float w0 = mw[sp * G + gg], w1 = sq != sp ? mw[sq * G + gg] : 0.f;
      acc[c].x = fmaf(w1, v1[c].x, fmaf(w0, v0[c].x, acc[c].x));
      acc[c].y = fmaf(w1, v1[c].y, fmaf(w0, v0[c].y, acc[c].y));
      acc[c].z = fmaf(w1, v1[c].z, fmaf(w0, v0[c].z, acc[c].z));
      acc[c].w = fmaf(w1, v1[c].w, fmaf(w0, v0[c].w, acc[c].w));
    }
  }
  const bool vec = (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0;  // the caller's buffer may be offset
#pragma unroll
  for (int c = 0; c < PIECES; ++c) {
    const int e = 4 * (lane + 32 * c), gg = e / D, d = e % D;
    float dn = den[0];
#pragma unroll
    for (int k = 1; k < G; ++k) dn = gg == k ? den[k] : dn;
    const float inv = dn > 0.f ? 1.f / dn : 0.f;
    float* dst = a.out + ((size_t)it.r * a.Hq + it.h * G + gg) * D + d;
    const float4 o = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
    if (vec) {
      *reinterpret_cast<float4*>(dst) = o;
    } else {
      dst[0] = o.x;
      dst[1] = o.y;
      dst[2] = o.z;
      dst[3] = o.w;
    }
  }
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
  float* tsum = reinterpret_cast<float*>(sm + L::TSUM);
  float* tmax = reinterpret_cast<float*>(sm + L::TMAX);
  int* misc = reinterpret_cast<int*>(sm + L::MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = misc + 1;
  volatile int* sm_fail = misc + 2;  // [2] a softmax warp's wait gave up, by tile parity
  volatile int* q_fail = misc + 4;   // the query warps' wait gave up
  const uint32_t bar0 = sb + (uint32_t)L::BARS;
  auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(NSTAGE + s); };
  auto qready = [&](int b) { return bar0 + 8u * (uint32_t)(2 * NSTAGE + b); };
  auto qfree = [&](int b) { return bar0 + 8u * (uint32_t)(2 * NSTAGE + 2 + b); };
  const uint32_t mmadone = bar0 + 8u * (uint32_t)(2 * NSTAGE + 4);
  auto sready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + j); };
  auto pready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + NS + j); };
  auto oready = [&](int j) { return mmadone + 8u * (uint32_t)(1 + 2 * NS + j); };
  auto sfree = [&](int j) { return mmadone + 8u * (uint32_t)(1 + 3 * NS + j); };
  auto endbar = [&](int e) { return mmadone + 8u * (uint32_t)(1 + 4 * NS + e); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = (int)blockIdx.x;
  // Every role walks the same items, this CTA's list from the host; the
  // next item's record is loaded while f runs on this one.  Items whose slot
  // is out of range are skipped (the first query thread records the error).
  // f returns false to stop.
  const int i_begin = a.cta_begin[cta], i_end = a.cta_begin[cta + 1];
  auto for_items = [&](auto&& f) {
    if (i_begin >= i_end) return;
    Item cur = load_item(a, i_begin);
    for (int i = i_begin; i < i_end; ++i) {
      const bool more = i + 1 < i_end;
      Item nxt;
      if (more) nxt = load_item(a, i + 1);
      if (!cur.ok) {
        if (tid == 32 * W_Q0) atomicOr(a.err, ERR_BAD_SLOT);
      } else if (!f(cur.w)) {
        break;
      }
      if (more) cur = nxt;
    }
  };

  if (tid == 0) {
    for (int i = 0; i < L::NBARS; ++i) {
      uint32_t cnt = 1;                                                      // one arrival (copy, commit, thread)
      if (i >= 2 * NSTAGE + 5 + NS && i < 2 * NSTAGE + 5 + 2 * NS) cnt = 4;  // pready: the softmax warps
      if (i >= 2 * NSTAGE + 5 + 3 * NS && i < 2 * NSTAGE + 5 + 4 * NS) cnt = 8;  // sfree: softmax + correction
      if (i >= 2 * NSTAGE + 5 + 4 * NS) cnt = 4;                             // endbar: the correction warps
      mbar_init(bar0 + 8u * (uint32_t)i, cnt);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort = 0;
    sm_fail[0] = 0;
    sm_fail[1] = 0;
    *q_fail = 0;
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

  if (warp == 0) {
    // ---- producer: every item's tiles, in order ----------------------------
    if (lane == 0) {
      int g = 0;  // tiles issued
      bool ok = true;
      const size_t layer_rows = (size_t)a.layer * a.num_pages_total;
      for_items([&](const AttnItem& it) {
        for (int t = 0; t < it.T; ++t, ++g) {
          const int s = g % NSTAGE;
          if (g >= NSTAGE && !(ok = wait_bar(empty(s), (uint32_t)(((g / NSTAGE) - 1) & 1), abort))) return false;
          int pg = a.bt[it.bt_off + it.p0 + (t >> 1)];
          if (pg < 0 || pg >= a.num_pages_total) {
            atomicOr(a.err, ERR_BAD_PAGE);
            pg = 0;
          }
          const int y = (int)(((layer_rows + (size_t)pg) * a.Hkv + it.h) * PAGE + (t & 1) * TK);
          const uint32_t dst = sb + (uint32_t)(L::ST + (size_t)s * STAGE);
          mbar_expect_tx(full(s), STAGE);
          tma_load_2d(dst, &a.kmap, 0, y, full(s));
          tma_load_2d(dst + HALF, &a.kmap, 64, y, full(s));
          tma_load_2d(dst + KBYTES, &a.vmap, 0, y, full(s));
          tma_load_2d(dst + KBYTES + HALF, &a.vmap, 64, y, full(s));
        }
        return true;
      });
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
      }
      // every copy issued has landed before the CTA moves on (bounded)
      const int zero = 0;
      for (int x = g > NSTAGE ? g - NSTAGE : 0; x < g; ++x)
        wait_bar(full(x % NSTAGE), (uint32_t)((x / NSTAGE) & 1), &zero);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer ----------------------------------------------------------
    if (lane == 0) {
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
      int g = 0, kq = 0;
      bool ok = true;
      for_items([&](const AttnItem& it) {
        const int b = kq & 1;
        if (!(ok = wait_bar(qready(b), (uint32_t)((kq >> 1) & 1), abort))) return false;
        const uint32_t qb = sb + (uint32_t)(L::QB + (size_t)b * OPB);
        for (int t = 0; t < it.T; ++t, ++g) {
          const int j = g % NS, s = g % NSTAGE;
          if (g >= NS && !(ok = wait_bar(sfree(j), (uint32_t)(((g / NS) - 1) & 1), abort))) return false;
          if (!(ok = wait_bar(full(s), (uint32_t)((g / NSTAGE) & 1), abort))) return false;
          tc_fence_after();
          const uint32_t k0 = sb + (uint32_t)(L::ST + (size_t)s * STAGE);
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_f16(tmem + (uint32_t)(j * 32), sw128_desc(k0 + (uint32_t)((k >> 2) * HALF + (k & 3) * 32)),
                    sw128_desc(qb + (uint32_t)((k >> 2) * (NB * 128) + (k & 3) * 32)), IDESC_QK, k > 0 ? 1u : 0u);
          mma_commit(sready(j));
          if (g >= 1 && !(ok = pv(g - 1))) return false;
        }
        mma_commit(qfree(b));  // the item's score MMAs read its q~
        ++kq;
        return true;
      });
      if (ok && g > 0) ok = pv(g - 1);
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
    unsigned char* pbuf = sm + L::PB;
    // the padding rows of the operands (both q~ and every slot's P) are zero
    for (int e = qt; e < (NB - 3 * G) * D; e += NQ_THR) {
      const int n = 3 * G + e / D, k = e % D;
#pragma unroll
      for (int b = 0; b < 2; ++b) st_bf16(sm + L::QB + (size_t)b * OPB, op_off(k, n), __float2bfloat16_rn(0.f));
#pragma unroll
      for (int j = 0; j < NS; ++j) st_bf16(pbuf + (size_t)j * OPB, op_off(k, n), __float2bfloat16_rn(0.f));
    }
    const float sc = 1.4426950408889634f / sqrtf((float)D);
    int kq = 0;
    for_items([&](const AttnItem& it) {
      const int b = kq & 1;
      unsigned char* qb = sm + L::QB + (size_t)b * OPB;
      if (qt == 0) {  // buffer b is free once the MMAs of item kq - 2 have read it
        const bool okw = kq < 2 || wait_bar(qfree(b), (uint32_t)(((kq >> 1) - 1) & 1), abort);
        if (!okw) {
          atomicOr(a.err, ERR_TIMEOUT);
          *abort = 1;
        }
        *q_fail = okw ? 0 : 1;
      }
      asm volatile("bar.sync %0, %1;" ::"n"(BAR_Q), "n"(NQ_THR) : "memory");
      if (*q_fail) return false;  // written only before the barrier: both query warps agree
      for (int e = qt; e < G * D; e += NQ_THR) {
        const int gi = e / D, d = e % D;
        const int g = it.h * G + gi;
        const size_t qi = ((size_t)it.r * a.Hq + g) * D + d;
        const double qv = a.q_f32 ? (double)static_cast<const float*>(a.q)[qi]
                                  : (double)__bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qi]);
        if (it.split == 0) {
          double* row =
              a.pool + (((size_t)a.layer * a.M + it.slot) * 2) * ((size_t)a.Hq * D) + (size_t)g * D + d;
          double* row_l = row + (size_t)a.Hq * D;
          if (a.first[it.r]) {
            *row = qv;
            *row_l = qv;
          } else {
            *row = fma(a.beta_s, *row, (1.0 - a.beta_s) * qv);
            *row_l = fma(a.beta_l, *row_l, (1.0 - a.beta_l) * qv);
          }
        }
        qs[gi * D + d] = (float)qv;
      }
      asm volatile("bar.sync %0, %1;" ::"n"(BAR_Q), "n"(NQ_THR) : "memory");
      // rotate-half RoPE at the request's position (pairs (i, i + D/2)) and the
      // log2(e)/sqrt(d) scale, then the three bf16 parts: rows gi, G + gi, 2G + gi
      for (int e = qt; e < G * (D / 2); e += NQ_THR) {
        const int gi = e / (D / 2), i = e % (D / 2);
        const double ang = (double)it.pos * a.inv_freq[i];
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
      if (qt == 0) mbar_arrive(qready(b));
      ++kq;
      return true;
    });
  } else if (warp < W_CR0) {
    // ---- softmax: thread = key of the tile -------------------------------------
    const int quad = warp & 3, key = 32 * quad + lane;
    const uint32_t lanes = (uint32_t)(32 * quad) << 16;
    unsigned char* pbuf = sm + L::PB;
    int g = 0;  // tiles, over the items
    for_items([&](const AttnItem& it) {
      float m[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) m[gg] = NEG;
      for (int t = 0; t < it.T; ++t, ++g) {
        const int j = g % NS;
        const bool ok = __all_sync(0xffffffffu, wait_bar(sready(j), (uint32_t)((g / NS) & 1), abort));
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
          sm_fail[g & 1] = 1;
        }
        const bool in_range = it.p0 * PAGE + t * TK + key < it.ntok;
        const bool valid = ok && in_range;
        if (ok && !in_range) {
          // a slot past the attended tokens (ragged last tile): its weight is 0,
          // but the cache may hold any bits there, and 0 x inf or NaN would
          // reach the output through the MMA; its V row is zeroed instead.  The
          // tile has landed (the score MMA read it), and the stage cannot be
          // reloaded before this tile's P is released.
          const int s = g % NSTAGE;
          wait_bar(full(s), (uint32_t)((g / NSTAGE) & 1), abort);
          unsigned char* vrow = sm + L::ST + (size_t)s * STAGE + KBYTES + (size_t)key * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            reinterpret_cast<uint4*>(vrow)[c] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(vrow + HALF)[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        float z[G], wm[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          z[gg] = valid ? v[gg] + (v[G + gg] + v[2 * G + gg]) : NEG;
          wm[gg] = z[gg];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) wm[gg] = fmaxf(wm[gg], __shfl_xor_sync(0xffffffffu, wm[gg], o));
        if (lane == 0)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) red[((g & 1) * 4 + quad) * G + gg] = wm[gg];
        asm volatile("bar.sync %0, %1;" ::"n"(BAR_SM), "n"(128) : "memory");
        if (sm_fail[g & 1]) return false;  // written only before the barrier: every softmax thread agrees
        unsigned char* pb = pbuf + (size_t)j * OPB;
        float ps[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float tm = red[((g & 1) * 4) * G + gg];
#pragma unroll
          for (int q = 1; q < 4; ++q) tm = fmaxf(tm, red[((g & 1) * 4 + q) * G + gg]);
          const float mn = fmaxf(m[gg], tm);
          const float rs = ex2f(m[gg] - mn);
          m[gg] = mn;
          const float p = valid ? ex2f(z[gg] - mn) : 0.f;
          ps[gg] = p;
          if (warp == W_SM0 && lane == 0) {
            scl[j * G + gg] = rs;
            tmax[j * G + gg] = mn;
          }
          __nv_bfloat16 h1, h2, h3;
          split3(p, h1, h2, h3);
          st_bf16(pb, op_off(key, gg), h1);
          st_bf16(pb, op_off(key, G + gg), h2);
          st_bf16(pb, op_off(key, 2 * G + gg), h3);
        }
        // the tile's weight sums of this warp's keys, for the correction warps
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) ps[gg] += __shfl_xor_sync(0xffffffffu, ps[gg], o);
        if (lane == 0)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) tsum[(j * 4 + quad) * G + gg] = ps[gg];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P (and zeroed V rows) visible to the MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(pready(j));
      }
      return true;
    });
  } else {
    // ---- correction: thread = dimension d --------------------------------------
    const int quad = warp & 3, d = 32 * quad + lane;
    const uint32_t lanes = (uint32_t)(32 * quad) << 16;
    int g = 0, ke = 0;  // tiles and non-empty items, over the items
    for_items([&](const AttnItem& it) {
      // empty items (no attended token in the split) are warp 8's alone
      if (it.T == 0 && warp != W_CR0) return true;
      float acc[G], den[G], mx[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        acc[gg] = 0.f;
        den[gg] = 0.f;
        mx[gg] = NEG;
      }
      for (int t = 0; t < it.T; ++t, ++g) {
        const int j = g % NS;
        bool ok = __all_sync(0xffffffffu, wait_bar(pready(j), (uint32_t)((g / NS) & 1), abort));
        float rs[G], ts[G], tm[G];
        if (ok) {
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            rs[gg] = scl[j * G + gg];
            tm[gg] = tmax[j * G + gg];
            ts[gg] = tsum[(j * 4) * G + gg] + tsum[(j * 4 + 1) * G + gg] + tsum[(j * 4 + 2) * G + gg] +
                     tsum[(j * 4 + 3) * G + gg];
          }
          ok = __all_sync(0xffffffffu, wait_bar(oready(j), (uint32_t)((g / NS) & 1), abort));
        }
        if (!ok) {
          if (lane == 0) {
            atomicOr(a.err, ERR_TIMEOUT);
            *abort = 1;
          }
          return false;
        }
        tc_fence_after();
        float o[16];
        tmem_ld<16>(tmem + lanes + (uint32_t)(j * 32 + 16), o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree(j));  // O_t and the tile's factors are read
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          acc[gg] = fmaf(acc[gg], rs[gg], o[gg] + (o[G + gg] + o[2 * G + gg]));
          den[gg] = fmaf(den[gg], rs[gg], ts[gg]);
          mx[gg] = tm[gg];
        }
      }
      if (it.nsp == 1) {
        // the pair's only split: its output directly, no partial, ticket or merge
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
          a.out[((size_t)it.r * a.Hq + it.h * G + gg) * D + d] = den[gg] > 0.f ? acc[gg] / den[gg] : 0.f;
        if (it.T == 0)  // warp 8 alone (the other warps skipped the item): every d of the pair
          for (int e = lane; e < G * D; e += 32) a.out[((size_t)it.r * a.Hq + it.h * G) * D + e] = 0.f;
        return true;
      }
      // the item's partial: output of dimension d, and (warp 8) maxima and sums
      float* po = a.part + (size_t)(it.part_first + it.split) * kPartFloats<G>;
      if (it.T > 0) {
#pragma unroll
        for (int gg = 0; gg < G; ++gg) po[gg * D + d] = acc[gg];
      } else {  // warp 8 alone: a zero output for every d
        for (int e = lane; e < G * D; e += 32) po[e] = 0.f;
      }
      if (warp == W_CR0)
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
          if (lane == gg) {
            po[G * D + gg] = mx[gg];
            po[G * D + G + gg] = den[gg];
          }
      // ordered before the ticket by the item-end barrier (release / acquire
      // within the CTA) and the ticket thread's fence at GPU scope, which is
      // cumulative over what that barrier made visible to it
      __syncwarp();
      if (it.T > 0 && lane == 0) mbar_arrive(endbar(ke % NEND));
      if (warp == W_CR0) {
        // every correction warp's part of the partial is out: ticket, and the
        // last item of (request, KV head) merges
        if (it.T > 0 &&
            !__all_sync(0xffffffffu, wait_bar(endbar(ke % NEND), (uint32_t)((ke / NEND) & 1), abort))) {
          if (lane == 0) {
            atomicOr(a.err, ERR_TIMEOUT);
            *abort = 1;
          }
          return false;
        }
        unsigned last = 0u;
        if (lane == 0) {
          __threadfence();
          const unsigned old = atomicAdd(a.tickets + (size_t)it.r * a.Hkv + it.h, 1u);
          last = old == (unsigned)(it.nsp - 1) ? 1u : 0u;
          if (last) __threadfence();
        }
        if (__shfl_sync(0xffffffffu, last, 0)) merge_splits<G>(a, it, reinterpret_cast<float*>(sm + L::MW), lane);
      }
      if (it.T > 0) ++ke;
      return true;
    });
  }

  // ---- every role is done: TMEM back ------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
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
  k_decode_attn_tc<G><<<dim3((unsigned)a.grid), NT, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention_tc(const AttnArgs& a, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  if (a.n_ctas < a.n * a.Hkv || a.grid < 1 || a.grid > a.n_ctas || !a.tc || a.kv_f32 || !attention_tc_shape(a.D, a.G))
    return cudaErrorInvalidValue;
  return a.G == 4 ? launch_tc<4>(a, s) : launch_tc<2>(a, s);
}

}  // namespace gp
