// Device code shared by the two boundary-demand kernels (CUDA-core FMA and
// tcgen05 variants): work-unit decoding, base-2 softmax statistics and their
// merge, the a-value / importance epilogue, and the p-coverage demand D_p.
//
// GrowPage Sec. 3.2 Eqs. 2, 7 and App. E.1 define what is computed:
//   a^x_i  = (1/G) sum_g softmax_{C_t}(q~^x_g . k_i / sqrt(d))_i   (i in C_t)
//   D_p    = min { |S| : S subset of C_t, sum_{i in S} a^x_i >= p }   (Eq. 2)
//   I_i    = max_x (1/G) sum_g softmax_{C_cmp}(...)_i                  (Eq. 9)
// Logits arrive in base 2 (the summaries are pre-scaled by log2(e)/sqrt(d)),
// so every exponential is a single ex2.
#pragma once

#include <cooperative_groups.h>

#include <cfloat>
#include <cstdint>

#include "gp_kernels.h"

namespace gp {
namespace dem {

namespace cg = cooperative_groups;

constexpr int NT = 256;    // threads per CTA
constexpr int NW = 8;      // warps per CTA
constexpr int PAGE = 256;  // tokens per page (b)
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One (request, layer, KV head) handled by a cluster of C CTAs.
struct Unit {
  int r, unit, layer, h;
  int P, ndem, ncmp;
  int crank, j0, npg;   // CTA's rank, first logical page, pages it scores
  DevReq rq;
};

__device__ __forceinline__ Unit make_unit(const DemandArgs& a) {
  Unit u;
  const int units = a.L * a.Hkv;
  const int wi = blockIdx.x / a.C;
  u.crank = blockIdx.x % a.C;
  u.r = a.work[wi / units];
  u.unit = wi % units;
  u.layer = u.unit / a.Hkv;
  u.h = u.unit % a.Hkv;
  u.rq = a.reqs[u.r];
  u.P = u.rq.num_pages;
  u.ndem = (u.P - 1) * PAGE;
  u.ncmp = u.P * PAGE - a.R;
  u.j0 = (u.crank * u.P) / a.C;  // balanced range: at most ceil(P / C) <= ppc pages
  u.npg = ((u.crank + 1) * u.P) / a.C - u.j0;
  return u;
}

// Physical page of logical page j of the unit's request, checked.
__device__ __forceinline__ int checked_page(const DemandArgs& a, const Unit& u, int j) {
  int pg = a.bt[u.rq.bt_off + j];
  if (pg < 0 || pg >= a.num_pages_total) {
    atomicOr(a.err, ERR_BAD_PAGE);
    pg = 0;
  }
  return pg;
}

// ---- softmax statistics --------------------------------------------------
// (m, s) with s = sum 2^(z - m).  An empty set is (NEG, 0): a finite
// sentinel keeps every update branch-free (2^(NEG - z) flushes to 0 and
// NEG - NEG = 0 multiplies a zero sum).
constexpr float NEG = -1.0e30f;

__device__ __forceinline__ void online(float& m, float& s, float z) {
  const float mn = fmaxf(m, z);
  s = s * ex2(m - mn) + ex2(z - mn);
  m = mn;
}

__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  s = s * ex2(m - mn) + s2 * ex2(m2 - mn);
  m = mn;
}

__device__ __forceinline__ void warp_combine(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(FULL, m, o);
    const float s2 = __shfl_xor_sync(FULL, s, o);
    combine(m, s, m2, s2);
  }
}

// Reduce N statistics (a power of two <= 16) over the warp with a
// reduce-scatter butterfly: at each of the first log2(N) levels a lane keeps
// half of its statistics and trades the other half with its partner, so the
// warp moves 2 (N - 1) + 2 (5 - log2 N) values per lane instead of 10 N.
// On return the lane holds statistic `idx` (lanes idx * 32/N ... +32/N-1).
template <int N>
__device__ __forceinline__ void warp_reduce_stats(float (&m)[N], float (&s)[N], int lane, float& om, float& os,
                                                  int& idx) {
  static_assert(N == 1 || N == 2 || N == 4 || N == 8 || N == 16, "power of two");
  idx = 0;
  int cnt = N;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const bool up = (lane & off) != 0;
    if (cnt > 1) {
      const int h = cnt / 2;
#pragma unroll
      for (int j = 0; j < N / 2; ++j) {
        if (j < h) {
          const float sm_ = up ? m[j] : m[j + h], ss_ = up ? s[j] : s[j + h];
          float km = up ? m[j + h] : m[j], ks = up ? s[j + h] : s[j];
          const float rm = __shfl_xor_sync(FULL, sm_, off), rs = __shfl_xor_sync(FULL, ss_, off);
          combine(km, ks, rm, rs);
          m[j] = km;
          s[j] = ks;
        }
      }
      idx = idx * 2 + (up ? 1 : 0);
      cnt = h;
    } else {
      const float rm = __shfl_xor_sync(FULL, m[0], off), rs = __shfl_xor_sync(FULL, s[0], off);
      combine(m[0], s[0], rm, rs);
    }
  }
  om = m[0];
  os = s[0];
}

// Compensated fp32 accumulation (Knuth's TwoSum).
struct Comp {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    const float bp = t - s;
    c += (s - (t - bp)) + (x - bp);
    s = t;
  }
  __device__ __forceinline__ float value() const { return s + c; }
};

// Exchange buffer written by every rank of the cluster into every rank:
// slot [rank][set][row] with set 0 = C_t keys, set 1 = the rest of C_cmp
// (the last page's keys below the recent window).
struct StatXchg {
  float m[16][2][8];
  float s[16][2][8];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, int rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Every CTA of a cluster must have started before any of them touches
// another's shared memory: each kernel opens with an arrive and waits on it
// before its first remote store.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Push this CTA's statistics into every rank of the cluster, then
// synchronise the cluster.  Thread t < 2 * ROWS holds statistic t (set
// t / ROWS, row t % ROWS) in (m, s).  All threads of the CTA must call it,
// after the cluster barrier phase opened by cluster_arrive_relaxed().
template <int ROWS>
__device__ __forceinline__ void push_stats(StatXchg* xg, int crank, int csize, float m, float s) {
  const int tid = threadIdx.x;
  cluster_wait();  // every rank has started
  if (tid < 2 * ROWS) {
    const int set = tid / ROWS, row = tid % ROWS;
    const uint32_t am = smem_u32(&xg->m[crank][set][row]);
    const uint32_t as = smem_u32(&xg->s[crank][set][row]);
    for (int c = 0; c < csize; ++c) {
      st_cluster_f32(am, c, m);
      st_cluster_f32(as, c, s);
    }
  }
  cluster_sync_all();
}

// Merge C ranks' statistics (m[c], s[c], stride `st` between ranks) into a
// base-2 log-sum-exp; *mx and *sx receive the merged (m, s).
__device__ __forceinline__ void merge_ranks(const float* m, const float* s, int C, int st, float* mx, float* sx) {
  float M = NEG;
  for (int c = 0; c < C; ++c) M = fmaxf(M, m[c * st]);
  Comp acc;
  for (int c = 0; c < C; ++c) acc.add(s[c * st] * ex2(m[c * st] - M));
  *mx = M;
  *sx = acc.value();
}

__device__ __forceinline__ void lse_pair(float md, float sd, float mt, float stl, float* lse_dem, float* lse_cmp) {
  *lse_dem = sd > 0.f ? md + lg2(sd) : 0.f;
  const float mc = fmaxf(md, mt);
  const float sc = sd * ex2(md - mc) + stl * ex2(mt - mc);
  *lse_cmp = sc > 0.f ? mc + lg2(sc) : 0.f;
}

// Merge the cluster's statistics into base-2 log-sum-exps:
// lse_dem[row] over C_t and lse_cmp[row] over C_cmp (C_t plus the tail).
template <int ROWS>
__device__ __forceinline__ void merge_stats(const StatXchg* xg, int csize, float* lse_dem, float* lse_cmp) {
  const int tid = threadIdx.x;
  if (tid < ROWS) {
    float md, sd, mt, stl;
    merge_ranks(&xg->m[0][0][tid], &xg->s[0][0][tid], csize, 16, &md, &sd);
    merge_ranks(&xg->m[0][1][tid], &xg->s[0][1][tid], csize, 16, &mt, &stl);
    lse_pair(md, sd, mt, stl, lse_dem + tid, lse_cmp + tid);
  }
}

// ---- per-key epilogue ----------------------------------------------------
// z[ROWS] base-2 logits of key i (rows x * G + g).  Writes a^S, a^L for
// i < ndem and the base-2 log importance for i < ncmp.
// a_out (optional) receives a^S, a^L when i < ndem.
template <int ROWS>
__device__ __forceinline__ void key_values(const float* z, int i, int ndem, int ncmp, const float* lse_dem,
                                           const float* lse_cmp, float* av, float* sc, float* a_out = nullptr) {
  constexpr int G = ROWS / 2;
  if (i < ndem) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      float s = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) s += ex2(z[x * G + g] - lse_dem[x * G + g]);
      s *= 1.0f / G;
      __stcg(av + (size_t)x * ndem + i, s);
      if (a_out) a_out[x] = s;
    }
  }
  if (i < ncmp) {
    float best = -FLT_MAX;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      float t[G];
      float m = -FLT_MAX;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        t[g] = z[x * G + g] - lse_cmp[x * G + g];
        m = fmaxf(m, t[g]);
      }
      float s = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) s += ex2(t[g] - m);
      best = fmaxf(best, m + lg2(s) - (G == 4 ? 2.f : 1.f));
    }
    sc[i] = best;
  }
}

// ---- p-coverage demand D_p (Eq. 2) ----------------------------------------
// Exact on the fp32 a-values of one summary: a value's mass is its product
// with 2^40 rounded to the nearest integer (ties to even), so every sum is an
// integer sum and the threshold test is exact.  With T the total mass and
// target = ceil(p T) (p a 64-bit binary fraction), D_p is the number of the
// largest values whose mass first reaches the target:
//   D_p = #(a > t) + ceil((target - mass(a > t)) / mass(t))
// for the threshold value t.  The values are non-negative, so their fp32 bit
// patterns order like the values and t is found by digits of the pattern.
//
//   1. One pass over the values: the exact total T, and a histogram over the
//      first digit (bits [29:20]: exponent and 3 mantissa bits) of each
//      value's mass >> 9, one 32-bit shared atomic per value of non-zero
//      approximate mass.  A block scan from the top picks the bin b where
//      that approximate mass reaches the target.
//   2. A second pass sums exactly the mass and count of the values above b
//      and the mass of b, and compacts b's members.  If the exact sums place
//      the target inside b, b is the threshold bin; if not (the truncated
//      masses can move the crossing across a bin edge), the first digit is
//      redone with exact histograms.
//   3. Within the bin, a few hundred members at most: every member counts
//      the members above it and their mass, and the member where the
//      cumulative mass reaches the target is t.  More members than that: two
//      more 10-bit digits ([19:10], [9:0]) with exact histograms of count and
//      mass (mass split in two 32-bit sums, mass >> 16 and mass & 0xffff).
// All of it in 32-bit integer and fp32 arithmetic: GB300 runs 64-bit
// conversions and divisions on its slow FP64 path.

// The bits of a value that take part: values >= 2 (not probabilities, or
// negative, inf, NaN) count as zero.
__device__ __forceinline__ unsigned sel_bits(unsigned u) { return u >= 0x40000000u ? 0u : u; }

// The mass of a value (bits u, 0 <= a < 2) as hi 2^23 + lo, 0 <= lo <= 2^23:
// hi = floor(a 2^17) and lo = the rest of a 2^40 rounded to nearest even.
// a 2^40 is exact, so is the remainder r = a 2^40 - hi 2^23 < 2^23 (a
// multiple of ulp(a 2^40) below 2^23), and adding 2^23 (ulp 1 on [2^23,
// 2^24)) rounds r to an integer with ties to even; floor(a 2^17) < 2^18 is
// taken the same way with round-toward-zero.
__device__ __forceinline__ void mass40(unsigned u, unsigned& hi, unsigned& lo) {
  const float a = __uint_as_float(u);
  const float t = __fadd_rz(__fmul_rn(a, 131072.0f), 8388608.0f);  // 2^23 + floor(a 2^17)
  hi = __float_as_uint(t) - 0x4B000000u;
  const float r = __fmaf_rn(-(t - 8388608.0f), 8388608.0f, __fmul_rn(a, 1099511627776.0f));
  lo = __float_as_uint(__fadd_rn(r, 8388608.0f)) - 0x4B000000u;
}
__device__ __forceinline__ unsigned long long mass40(unsigned u) {
  unsigned hi, lo;
  mass40(u, hi, lo);
  return ((unsigned long long)hi << 23) + lo;
}

// ceil(t * f / 2^64), at least 1: the target mass for the fraction f.
__device__ __forceinline__ unsigned long long coverage_target(unsigned long long t, unsigned long long f) {
  const unsigned long long hi = __umul64hi(t, f), lo = t * f;
  const unsigned long long g = hi + (lo != 0ull ? 1ull : 0ull);
  return g < 1ull ? 1ull : g;
}

// min(cap, ceil(need / f)) for f >= 1, need >= 1, without a 64-bit division:
// a float estimate, good to well under one unit when the result is at most
// cap + 2 < 2^20, then exact integer steps.
__device__ __forceinline__ unsigned ceil_div_capped(unsigned long long need, unsigned long long f, unsigned cap) {
  const float q = __fdiv_rn((float)need, (float)f);
  if (!(q <= (float)cap + 2.0f)) return cap;
  unsigned j = (unsigned)q;
  while (j > 0u && (unsigned long long)(j - 1u) * f >= need) --j;
  while ((unsigned long long)j * f < need) ++j;
  return j < cap ? j : cap;
}

constexpr int SEL_BINS = 1024;  // every digit
constexpr int APPROX_SHIFT = 9;  // first-digit histogram: mass >> 9 (sums stay below 2^32)

struct DpState {
  unsigned prefix, cnt_above, cnt_eq;
  unsigned long long mass_above, target;
  int bad;
};

struct DpSmem {
  unsigned am[SEL_BINS];   // first digit: approximate mass
  unsigned cnt[SEL_BINS];  // exact digits: count,
  unsigned mhi[SEL_BINS];  //   mass >> 16,
  unsigned mlo[SEL_BINS];  //   mass & 0xffff
  unsigned long long wm[32], we[32];  // per-warp partial sums
  unsigned wc[32];
  DpState st;
  unsigned ncomp;          // members of the threshold bin appended so far
  unsigned res;            // D_p once found (~0u before)
};

__device__ __forceinline__ void hist_add(DpSmem* sm, int bin, unsigned u) {
  unsigned hi, lo;
  mass40(u, hi, lo);
  atomicAdd(&sm->cnt[bin], 1u);
  atomicAdd(&sm->mhi[bin], (hi << 7) + (lo >> 16));
  atomicAdd(&sm->mlo[bin], lo & 0xFFFFu);
}
__device__ __forceinline__ unsigned long long bin_mass(const DpSmem* sm, int bin) {
  return ((unsigned long long)sm->mhi[bin] << 16) + sm->mlo[bin];
}

template <int NTH>
__device__ __forceinline__ void clear_exact_hist(DpSmem* sm, int tid) {
  for (int k = tid; k < SEL_BINS; k += NTH) {
    sm->cnt[k] = 0u;
    sm->mhi[k] = 0u;
    sm->mlo[k] = 0u;
  }
}

// Barrier over the NTH threads that run a select (id 0 with the whole CTA).
template <int NTH, int BAR>
__device__ __forceinline__ void sel_sync() {
  if constexpr (BAR == 0) {
    __syncthreads();
  } else {
    asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NTH) : "memory");
  }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ unsigned warp_sum_u32(unsigned v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// One exact digit: scan the bins from the top (a block-wide prefix sum over
// thread-owned runs of bins) and record the bin where the cumulative mass
// reaches the target.  need = target - mass above the bins, read by every
// thread before the barrier inside, so the crossing thread may update st.
template <int NTH, int BAR>
__device__ __forceinline__ void pick_digit(DpSmem* sm, int shift, unsigned long long need, int tid) {
  constexpr int NWS = NTH / 32;
  constexpr int PER = (SEL_BINS + NTH - 1) / NTH;
  const int lane = tid & 31, wid = tid >> 5;
  const int q0 = tid * PER, q1 = min(SEL_BINS, q0 + PER);  // positions from the top
  unsigned long long lm = 0ull;
  unsigned lc = 0u;
  for (int q = q0; q < q1; ++q) {
    lm += bin_mass(sm, SEL_BINS - 1 - q);
    lc += sm->cnt[SEL_BINS - 1 - q];
  }
  unsigned long long im = lm;
  unsigned ic = lc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long om = __shfl_up_sync(FULL, im, o);
    const unsigned oc = __shfl_up_sync(FULL, ic, o);
    if (lane >= o) {
      im += om;
      ic += oc;
    }
  }
  if (lane == 31) {
    sm->wm[wid] = im;
    sm->wc[wid] = ic;
  }
  sel_sync<NTH, BAR>();
  unsigned long long base_m = 0ull;
  unsigned base_c = 0u;
#pragma unroll
  for (int w = 0; w < NWS; ++w) {
    if (w < wid) {
      base_m += sm->wm[w];
      base_c += sm->wc[w];
    }
  }
  const unsigned long long incl = base_m + im, excl = incl - lm;
  if ((excl < need && need <= incl) || (tid == NTH - 1 && incl < need)) {
    DpState& st = sm->st;
    unsigned long long cum = excl;
    unsigned cnt = base_c + ic - lc;
    int chosen = -1;
    for (int q = q0; q < q1; ++q) {
      const unsigned long long mb = bin_mass(sm, SEL_BINS - 1 - q);
      if (cum + mb >= need) {
        chosen = SEL_BINS - 1 - q;
        break;
      }
      cum += mb;
      cnt += sm->cnt[SEL_BINS - 1 - q];
    }
    if (chosen < 0) {  // the target lies beyond all mass: inconsistent input
      st.bad = 1;
      chosen = 0;
    }
    st.prefix |= (unsigned)chosen << shift;
    st.mass_above += cum;
    st.cnt_above += cnt;
    st.cnt_eq = sm->cnt[chosen];
  }
}

// Mbarrier helpers for the staging copy of the select.
__device__ __forceinline__ bool sel_bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Append the kept values among v[0..3] of every lane of the warp to
// dst[*count ...] with one shared atomic per warp (order is irrelevant).
// Positions at or beyond `room` are counted but not written.
__device__ __forceinline__ void warp_append4(const unsigned (&v)[4], const bool (&keep)[4], unsigned* dst,
                                             unsigned* count, unsigned room, int lane) {
  const unsigned c = (unsigned)keep[0] + keep[1] + keep[2] + keep[3];
  if (!__any_sync(FULL, c != 0u)) return;
  unsigned incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned tot = __shfl_sync(FULL, incl, 31);
  unsigned base = 0u;
  if (lane == 31) base = atomicAdd(count, tot);
  base = __shfl_sync(FULL, base, 31);
  unsigned pos = base + incl - c;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (keep[k]) {
      if (pos < room) dst[pos] = v[k];
      ++pos;
    }
}

// Whether coverage_demand stages the n values in its scratch of cap words
// (and so uses its staging barrier, whose phase the caller then flips).
__host__ __device__ __forceinline__ bool sel_resident(int n, int cap) { return n <= cap; }

// D_p of one summary from its n a-values av[n] (global, written by the
// unit's CTAs, 16-byte aligned, n a multiple of 256), for the target
// fraction pfix / 2^64.  Called by NTH threads (tid in [0, NTH), whole warps)
// that synchronise on named barrier BAR.  sm: shared DpSmem; buf: shared
// scratch of `cap` words, 16-byte aligned.
//   * n <= cap: the values are staged in buf -- by one bulk async copy
//     completing on the initialised mbarrier `bar` (phase `parity`) when
//     bar != 0, else by 16-byte loads -- and every pass reads them there;
//   * otherwise the passes read global memory.
// The threshold bin's members are compacted behind the staged values (or at
// the start of buf) when they fit.  Every thread returns D_p.
template <int NTH, int BAR>
__device__ __forceinline__ unsigned coverage_demand(const float* av, int n, unsigned long long pfix, unsigned* buf,
                                                    int cap, DpSmem* sm, int* err, int tid, uint32_t bar,
                                                    uint32_t parity) {
  static_assert(NTH % 32 == 0 && NTH <= 1024, "whole warps");
  constexpr int NWS = NTH / 32;
  const int lane = tid & 31, wid = tid >> 5;
  const bool resident = sel_resident(n, cap);
  if (tid == 0) {
    DpState& s = sm->st;
    s.prefix = 0u;
    s.cnt_above = 0u;
    s.cnt_eq = 0u;
    s.mass_above = 0ull;
    s.target = 0ull;
    s.bad = 0;
    sm->ncomp = 0u;
    sm->res = ~0u;
  }
  const uint4* src4 = reinterpret_cast<const uint4*>(av);
  const int n4 = n / 4;  // 16-byte groups
  if (resident && bar != 0u && tid == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // buf was last read by ordinary loads
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)(4 * n))
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(buf)),
                 "l"(av), "r"((uint32_t)(4 * n)), "r"(bar)
                 : "memory");
  }
  for (int k = tid; k < SEL_BINS; k += NTH) sm->am[k] = 0u;
  if (resident) {
    if (bar != 0u) {
      bool ok = sel_bar_try(bar, parity);
      if (!ok) {
        const long long t0 = clock64();
        while (!(ok = sel_bar_try(bar, parity)) && clock64() - t0 < (1ll << 31)) {
        }
      }
      if (!ok) atomicOr(err, ERR_TIMEOUT);
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(buf);
      int i = tid;
      for (; i + 3 * NTH < n4; i += 4 * NTH) {
        const uint4 v0 = __ldcg(src4 + i), v1 = __ldcg(src4 + i + NTH), v2 = __ldcg(src4 + i + 2 * NTH),
                    v3 = __ldcg(src4 + i + 3 * NTH);
        d4[i] = v0;
        d4[i + NTH] = v1;
        d4[i + 2 * NTH] = v2;
        d4[i + 3 * NTH] = v3;
      }
      for (; i < n4; i += NTH) d4[i] = __ldcg(src4 + i);
    }
  }
  sel_sync<NTH, BAR>();
  // Visit every value as f(bits[4], in range), four 16-byte groups in flight
  // per thread; bits already through sel_bits, zero out of range.
  auto each_value = [&](auto&& f) {
    for (int i0 = 0; i0 < n4; i0 += 4 * NTH) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * NTH + tid;
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < n4) v[j] = resident ? reinterpret_cast<const uint4*>(buf)[i] : __ldcg(src4 + i);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned w[4] = {sel_bits(v[j].x), sel_bits(v[j].y), sel_bits(v[j].z), sel_bits(v[j].w)};
        f(w);
      }
    }
  };

  // 1. exact total, approximate first-digit histogram
  {
    unsigned thi = 0u, tlo = 0u;  // sums of hi (< 2^18 each) and lo (<= 2^23 each)
    each_value([&](const unsigned (&w)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        unsigned hi, lo;
        mass40(w[k], hi, lo);
        thi += hi;
        tlo += lo;
        const unsigned h = (hi << (23 - APPROX_SHIFT)) + (lo >> APPROX_SHIFT);
        if (h != 0u) atomicAdd(&sm->am[w[k] >> 20], h);
      }
    });
    const unsigned long long tot = warp_sum_u64(((unsigned long long)thi << 23) + tlo);
    if (lane == 0) sm->wm[wid] = tot;
  }
  sel_sync<NTH, BAR>();
  unsigned long long tot = 0ull;
#pragma unroll
  for (int w = 0; w < NWS; ++w) tot += sm->wm[w];
  if (tot == 0ull) return 0u;  // no mass at all: nothing to cover
  const unsigned long long target = coverage_target(tot, pfix);
  {
    constexpr int PER = (SEL_BINS + NTH - 1) / NTH;
    const int q0 = tid * PER, q1 = min(SEL_BINS, q0 + PER);
    unsigned ls = 0u;
    for (int q = q0; q < q1; ++q) ls += sm->am[SEL_BINS - 1 - q];
    unsigned is = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL, is, o);
      if (lane >= o) is += t;
    }
    if (lane == 31) sm->wc[wid] = is;
    sel_sync<NTH, BAR>();
    unsigned base = 0u;
#pragma unroll
    for (int w = 0; w < NWS; ++w)
      if (w < wid) base += sm->wc[w];
    const unsigned long long incl = (unsigned long long)(base + is) << APPROX_SHIFT;
    const unsigned long long excl = (unsigned long long)(base + is - ls) << APPROX_SHIFT;
    if ((excl < target && target <= incl) || (tid == NTH - 1 && incl < target)) {
      unsigned long long cum = excl;
      int chosen = 0;
      for (int q = q0; q < q1; ++q) {
        const unsigned long long mb = (unsigned long long)sm->am[SEL_BINS - 1 - q] << APPROX_SHIFT;
        if (cum + mb >= target) {
          chosen = SEL_BINS - 1 - q;
          break;
        }
        cum += mb;
      }
      sm->st.prefix = (unsigned)chosen;  // the candidate bin, checked below
    }
    sel_sync<NTH, BAR>();
  }

  // 2. exact mass and count above the candidate bin, its mass and members
  const unsigned bsel = sm->st.prefix;
  const unsigned cbase = resident ? (unsigned)n : 0u;
  const unsigned space = (unsigned)cap > cbase ? (unsigned)cap - cbase : 0u;
  unsigned* memb = buf + cbase;
  {
    unsigned ahi = 0u, alo = 0u, ehi = 0u, elo = 0u, ca = 0u;
    each_value([&](const unsigned (&w)[4]) {
      bool keep[4], above[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const unsigned b = w[k] >> 20;
        keep[k] = w[k] != 0u && b == bsel;
        above[k] = b > bsel;
      }
      const bool any_above = above[0] || above[1] || above[2] || above[3];
      const bool any_keep = keep[0] || keep[1] || keep[2] || keep[3];
      if (__any_sync(FULL, any_above || any_keep)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          unsigned hi, lo;
          mass40(w[k], hi, lo);
          if (above[k]) {
            ahi += hi;
            alo += lo;
            ++ca;
          }
          if (keep[k]) {
            ehi += hi;
            elo += lo;
          }
        }
        warp_append4(w, keep, memb, &sm->ncomp, space, lane);
      }
    });
    const unsigned long long ma = warp_sum_u64(((unsigned long long)ahi << 23) + alo);
    const unsigned long long me = warp_sum_u64(((unsigned long long)ehi << 23) + elo);
    ca = warp_sum_u32(ca);
    if (lane == 0) {
      sm->wm[wid] = ma;
      sm->we[wid] = me;
      sm->wc[wid] = ca;
    }
  }
  sel_sync<NTH, BAR>();
  unsigned long long above = 0ull, in_bin = 0ull;
  unsigned cnt_above = 0u;
#pragma unroll
  for (int w = 0; w < NWS; ++w) {
    above += sm->wm[w];
    in_bin += sm->we[w];
    cnt_above += sm->wc[w];
  }
  const unsigned m = sm->ncomp;
  const bool first_ok = above < target && target <= above + in_bin;
  // 3a layout: members padded with zeros (mass 0, never above or equal to a
  // member of positive mass) to tpc chunks of a multiple of 4, then their
  // masses; tpc threads share a member.
  unsigned tpc = 1u;
  while (tpc < 32u && m * tpc * 2u <= (unsigned)NTH) tpc <<= 1;
  const unsigned chunk = ((m + tpc - 1u) / tpc + 3u) & ~3u, mpad = chunk * tpc;
  bool compacted = first_ok && m <= space;

  if (first_ok && 3u * mpad <= space && m * m <= 128u * NTH) {
    // 3a. rank every member among the members
    unsigned long long* fm = reinterpret_cast<unsigned long long*>(memb + mpad);  // 16-byte aligned
    for (unsigned i = tid; i < mpad; i += NTH) {
      const unsigned u = i < m ? memb[i] : 0u;
      if (i >= m) memb[i] = 0u;
      fm[i] = mass40(u);
    }
    sel_sync<NTH, BAR>();
    const unsigned long long need = target - above;
    const unsigned per_pass = NTH / tpc, part = (unsigned)tid % tpc;
    for (unsigned i0 = 0; i0 < m; i0 += per_pass) {
      const unsigned i = i0 + (unsigned)tid / tpc;
      const unsigned v = i < m ? memb[i] : 0u;
      unsigned long long g_mass = 0ull;
      unsigned g_cnt = 0u, e_cnt = 0u;
      if (i < m) {
        const uint4* c4 = reinterpret_cast<const uint4*>(memb + part * chunk);
        const ulonglong2* f2 = reinterpret_cast<const ulonglong2*>(fm + part * chunk);
        for (int q = 0; q < (int)(chunk / 4u); ++q) {
          const uint4 c = c4[q];
          const ulonglong2 fa = f2[2 * q], fb = f2[2 * q + 1];
          g_mass += (c.x > v ? fa.x : 0ull) + (c.y > v ? fa.y : 0ull) + (c.z > v ? fb.x : 0ull) +
                    (c.w > v ? fb.y : 0ull);
          g_cnt += (unsigned)(c.x > v) + (unsigned)(c.y > v) + (unsigned)(c.z > v) + (unsigned)(c.w > v);
          e_cnt += (unsigned)(c.x == v) + (unsigned)(c.y == v) + (unsigned)(c.z == v) + (unsigned)(c.w == v);
        }
      }
      for (unsigned o = 1; o < tpc; o <<= 1) {
        g_mass += __shfl_xor_sync(FULL, g_mass, o);
        g_cnt += __shfl_xor_sync(FULL, g_cnt, o);
        e_cnt += __shfl_xor_sync(FULL, e_cnt, o);
      }
      if (i < m && part == 0u) {
        const unsigned long long fv = fm[i];
        if (g_mass < need && fv > 0ull && need - g_mass <= fv * e_cnt)  // the same for every member equal to t
          sm->res = cnt_above + g_cnt + ceil_div_capped(need - g_mass, fv, e_cnt);
      }
    }
    sel_sync<NTH, BAR>();
    const unsigned r = sm->res;
    sel_sync<NTH, BAR>();  // the scratch may be reused once every thread is done
    if (r != ~0u) return r;
    if (tid == 0) atomicOr(err, ERR_BAD_COUNT);  // unreachable for consistent sums
    return 0u;
  }

  // 3b. exact digits
  if (tid == 0) {
    DpState& s = sm->st;
    s.target = target;
    if (first_ok) {
      s.prefix = bsel << 20;
      s.mass_above = above;
      s.cnt_above = cnt_above;
      s.cnt_eq = m;
    } else {
      s.prefix = 0u;
      s.mass_above = 0ull;
      s.cnt_above = 0u;
    }
  }
  clear_exact_hist<NTH>(sm, tid);
  sel_sync<NTH, BAR>();
  if (!first_ok) {
    compacted = false;
    each_value([&](const unsigned (&w)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (w[k] != 0u) hist_add(sm, (int)(w[k] >> 20), w[k]);
    });
    sel_sync<NTH, BAR>();
    pick_digit<NTH, BAR>(sm, 20, target, tid);
  }
#pragma unroll
  for (int ro = 0; ro < 2; ++ro) {
    const int sh = ro == 0 ? 10 : 0;
    const unsigned hi_mask = ro == 0 ? 0x3FF00000u : 0x3FFFFC00u;  // bits already fixed
    sel_sync<NTH, BAR>();
    const unsigned pf = sm->st.prefix;
    const unsigned long long need = target - sm->st.mass_above;
    if (ro == 1 || !first_ok) {  // the histograms of the previous digit are done with
      clear_exact_hist<NTH>(sm, tid);
      sel_sync<NTH, BAR>();
    }
    if (compacted) {
      for (unsigned i = tid; i < m; i += NTH) {
        const unsigned u = memb[i];
        if ((u & hi_mask) == pf) hist_add(sm, (int)((u >> sh) & (SEL_BINS - 1)), u);
      }
    } else {
      each_value([&](const unsigned (&w)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (w[k] != 0u && (w[k] & hi_mask) == pf) hist_add(sm, (int)((w[k] >> sh) & (SEL_BINS - 1)), w[k]);
      });
    }
    sel_sync<NTH, BAR>();
    pick_digit<NTH, BAR>(sm, sh, need, tid);
  }
  sel_sync<NTH, BAR>();
  const DpState& s = sm->st;
  const unsigned long long tf = mass40(s.prefix);
  const unsigned long long need = s.target - s.mass_above;
  const unsigned j = tf > 0ull ? ceil_div_capped(need, tf, s.cnt_eq) : s.cnt_eq;
  const unsigned res = s.cnt_above + (j < 1u ? 1u : j);
  if (s.bad && tid == 0) atomicOr(err, ERR_BAD_COUNT);
  sel_sync<NTH, BAR>();  // the scratch may be reused once every thread is done
  return res;
}

// After a CTA has written its a-values: the last of the unit's C CTAs to get
// here (global ticket) computes D_p for the unit.  Returns true in that CTA.
__device__ __forceinline__ bool last_of_unit(const DemandArgs& a, const Unit& u, int* flag_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // the CTA's a-values (ordered by the barrier) before the ticket
    unsigned* t = a.tickets + (size_t)u.r * (a.L * a.Hkv) + u.unit;
    const unsigned old = atomicAdd(t, 1u);
    const bool last = old == (unsigned)(a.C - 1);
    if (last) __threadfence();
    *flag_smem = last ? 1 : 0;
  }
  __syncthreads();
  return *flag_smem != 0;
}

// Stores D_p of summary x of a unit and adds it to the request's sum (one thread).
__device__ __forceinline__ void write_demand(const DemandArgs& a, int r, int unit, int x, unsigned k) {
  const int units = a.L * a.Hkv;
  a.kout[((size_t)r * units + unit) * 2 + x] = (int32_t)k;
  atomicAdd(a.ksum + (size_t)r * 2 + x, (unsigned long long)k);
}

// Launch with a cluster of a.C CTAs along x.
template <typename K>
cudaError_t launch_cluster(K kern, const DemandArgs& a, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.C * a.n_work * a.L * a.Hkv, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace dem
}  // namespace gp
