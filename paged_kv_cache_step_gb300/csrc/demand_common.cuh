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
  u.j0 = u.crank * a.ppc;
  u.npg = max(0, min(u.P, u.j0 + a.ppc) - u.j0);
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
// Exact on the fp32 a-values: masses are fixed point with 40 fractional bits,
// so every sum is an integer sum and the threshold test is exact.  A radix
// select on the fp32 bit pattern (a >= 0, so the bits order like the values)
// walks three 10-bit digits from the top -- bits [29:20] (exponent and 3
// mantissa bits), [19:10], [9:0] -- keeping the bin where the cumulative
// mass, counted from the largest values down, reaches ceil(p * total).  Then
// D_p = #(a > t) + ceil((target - mass(a > t)) / mass(t)).
// A bin holds its count and its mass split in two 32-bit sums (mass >> 16,
// mass & 0xffff), each fed by a native 32-bit shared atomic; the first digit
// reaches into the mantissa, so even a flat distribution spreads over many
// bins and the atomics rarely collide.

__device__ __forceinline__ unsigned long long fixed40(unsigned u) {
  const int e = (int)(u >> 23) & 255;
  if (e == 0 || e > 128) return 0ull;  // zero, or not a probability (inf / NaN)
  const unsigned long long m = (u & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 110;  // value * 2^40 = m * 2^(e - 110)
  if (sh >= 0) return m << sh;
  const int s = -sh;
  if (s >= 25) return 0ull;  // below one half
  const unsigned long long q = m >> s, r = m & ((1ull << s) - 1), half = 1ull << (s - 1);
  return q + ((r > half || (r == half && (q & 1ull))) ? 1ull : 0ull);
}

constexpr int SEL_BINS = 1024;  // every digit

struct DpState {
  unsigned prefix, cnt_above, cnt_eq;
  unsigned long long mass_above, target;
  int bad, done;
};

struct DpSmem {
  unsigned cnt[2][SEL_BINS];
  unsigned mhi[2][SEL_BINS];             // sum of mass >> 16
  unsigned mlo[2][SEL_BINS];             // sum of mass & 0xffff
  unsigned long long wm[2][32];          // per-warp scan totals: mass
  unsigned wc[2][32];                    //                       count
  DpState st[2];
  unsigned ncomp[2];
  int compact;
};

__device__ __forceinline__ void hist_add(DpSmem* sm, int x, int bin, unsigned long long w) {
  atomicAdd(&sm->cnt[x][bin], 1u);
  atomicAdd(&sm->mhi[x][bin], (unsigned)(w >> 16));
  atomicAdd(&sm->mlo[x][bin], (unsigned)(w & 0xFFFFull));
}
__device__ __forceinline__ unsigned long long bin_mass(const DpSmem* sm, int x, int bin) {
  return ((unsigned long long)sm->mhi[x][bin] << 16) + sm->mlo[x][bin];
}

// The bits of a value that take part: values >= 2 (not probabilities) count
// as zero.
__device__ __forceinline__ unsigned sel_bits(unsigned u) { return u >= 0x40000000u ? 0u : u; }

// Values below 2^-41 (biased exponent <= 85) have exactly zero fixed-point
// mass.  They lie in first-digit bins strictly below any bin holding a value
// of positive mass, and the threshold bin always holds one, so they never
// reach the count or mass above the threshold: the histograms skip them.
constexpr unsigned MIN_MASS_BITS = 86u << 23;

template <int NTH>
__device__ __forceinline__ void clear_hist(DpSmem* sm, int tid) {
  for (int k = tid; k < 2 * SEL_BINS; k += NTH) {
    (&sm->cnt[0][0])[k] = 0u;
    (&sm->mhi[0][0])[k] = 0u;
    (&sm->mlo[0][0])[k] = 0u;
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

// One digit for both summaries: scan the bins from the top (a block-wide
// prefix sum over thread-owned runs of bins), fix the target on the first
// digit, and record the bin where the mass reaches it.
template <int NTH, int BAR>
__device__ __forceinline__ void pick_digit(DpSmem* sm, int shift, bool first, double p, int tid) {
  constexpr int nbins = SEL_BINS;
  constexpr int NWS = NTH / 32;
  const int lane = tid & 31, wid = tid >> 5;
  const int per = (nbins + NTH - 1) / NTH;
  const int q0 = tid * per, q1 = min(nbins, q0 + per);  // positions from the top
  unsigned long long lm[2] = {0ull, 0ull};
  unsigned lc[2] = {0u, 0u};
  for (int q = q0; q < q1; ++q) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      lm[x] += bin_mass(sm, x, nbins - 1 - q);
      lc[x] += sm->cnt[x][nbins - 1 - q];
    }
  }
  unsigned long long im[2] = {lm[0], lm[1]};
  unsigned ic[2] = {lc[0], lc[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const unsigned long long om = __shfl_up_sync(FULL, im[x], o);
      const unsigned oc = __shfl_up_sync(FULL, ic[x], o);
      if (lane >= o) {
        im[x] += om;
        ic[x] += oc;
      }
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      sm->wm[x][wid] = im[x];
      sm->wc[x][wid] = ic[x];
    }
  }
  sel_sync<NTH, BAR>();
  unsigned long long base_m[2] = {0ull, 0ull}, tot[2] = {0ull, 0ull};
  unsigned base_c[2] = {0u, 0u};
#pragma unroll
  for (int x = 0; x < 2; ++x)
    for (int w = 0; w < NWS; ++w) {
      if (w < wid) {
        base_m[x] += sm->wm[x][w];
        base_c[x] += sm->wc[x][w];
      }
      tot[x] += sm->wm[x][w];
    }
  if (first && tid < 2) {
    DpState& st = sm->st[tid];
    if (tot[tid] == 0ull) {
      st.done = 1;
    } else {
      unsigned long long tg = (unsigned long long)ceil(p * (double)tot[tid]);
      if (tg < 1ull) tg = 1ull;
      if (tg > tot[tid]) tg = tot[tid];
      st.target = tg;
    }
  }
  if (first) sel_sync<NTH, BAR>();
  // Every thread reads the state before the crossing thread updates it.
  unsigned long long needs[2];
  bool dones[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    dones[x] = sm->st[x].done != 0;
    needs[x] = sm->st[x].target - sm->st[x].mass_above;
  }
  sel_sync<NTH, BAR>();
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    DpState& st = sm->st[x];
    if (dones[x]) continue;
    const unsigned long long need = needs[x];
    const unsigned long long incl = base_m[x] + im[x], excl = incl - lm[x];
    const bool last = tid == NTH - 1;
    if ((excl < need && need <= incl) || (last && incl < need)) {
      unsigned long long cum = excl;
      unsigned cnt = base_c[x] + ic[x] - lc[x];
      int chosen = -1;
      for (int q = q0; q < q1; ++q) {
        const unsigned long long mb = bin_mass(sm, x, nbins - 1 - q);
        if (cum + mb >= need) {
          chosen = nbins - 1 - q;
          break;
        }
        cum += mb;
        cnt += sm->cnt[x][nbins - 1 - q];
      }
      if (chosen < 0) {  // the target lies beyond all mass: inconsistent input
        st.bad = 1;
        chosen = 0;
      }
      st.prefix |= (unsigned)chosen << shift;
      st.mass_above += cum;
      st.cnt_above += cnt;
      st.cnt_eq = sm->cnt[x][chosen];
    }
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
__device__ __forceinline__ void warp_append4(const unsigned (&v)[4], const bool (&keep)[4], unsigned* dst,
                                             unsigned* count, int lane) {
  const unsigned c = (unsigned)keep[0] + keep[1] + keep[2] + keep[3];
  if (!__any_sync(FULL, c != 0u)) return;
  unsigned incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned tot = __shfl_sync(FULL, incl, 31);
  if (tot == 0u) return;
  unsigned base = 0u;
  if (lane == 31) base = atomicAdd(count, tot);
  base = __shfl_sync(FULL, base, 31);
  unsigned pos = base + incl - c;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (keep[k]) dst[pos++] = v[k];
}

// D_p of both summaries of one unit from its a-values av[2][ndem] (global,
// written by the unit's CTAs, 16-byte aligned, ndem a multiple of 256).
// Called by NTH threads (tid in [0, NTH), whole warps) that synchronise on
// named barrier BAR.  sm: shared DpSmem; buf: shared scratch of `cap` words.
//   * 2 ndem <= cap: the a-values are staged in buf -- by one bulk async
//     copy completing on the initialised mbarrier `bar` (phase `parity`) when
//     bar != 0, else by 16-byte loads -- and the first digit reads them there;
//   * otherwise the first digit reads global memory (four 16-byte loads in
//     flight per thread).
// Then the members of the first digit's bin are compacted behind the staged
// values (or at the start of buf) when they fit, and the other two digits
// run over them; if they do not fit, those digits re-scan every value.
// Thread x < 2 returns D_p for summary x.
template <int NTH, int BAR>
__device__ __forceinline__ unsigned coverage_demand(const float* av, int ndem, double p, unsigned* buf, int cap,
                                                    DpSmem* sm, int* err, int tid, uint32_t bar, uint32_t parity) {
  static_assert(NTH % 32 == 0 && NTH <= 1024, "whole warps");
  const int lane = tid & 31;
  const bool resident = 2 * ndem <= cap;
  if (tid < 2) {
    DpState& s = sm->st[tid];
    s.prefix = 0u;
    s.cnt_above = 0u;
    s.cnt_eq = 0u;
    s.mass_above = 0ull;
    s.target = 0ull;
    s.bad = 0;
    s.done = 0;
    sm->ncomp[tid] = 0u;
  }
  const uint4* src4 = reinterpret_cast<const uint4*>(av);
  const int n4 = ndem / 4;  // 16-byte groups per summary
  if (resident && bar != 0u && tid == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // buf was last read by ordinary loads
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)(8 * ndem))
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(buf)),
                 "l"(av), "r"((uint32_t)(8 * ndem)), "r"(bar)
                 : "memory");
  }
  clear_hist<NTH>(sm, tid);
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
      for (; i + 3 * NTH < 2 * n4; i += 4 * NTH) {
        const uint4 v0 = __ldcg(src4 + i), v1 = __ldcg(src4 + i + NTH), v2 = __ldcg(src4 + i + 2 * NTH),
                    v3 = __ldcg(src4 + i + 3 * NTH);
        d4[i] = v0;
        d4[i + NTH] = v1;
        d4[i + 2 * NTH] = v2;
        d4[i + 3 * NTH] = v3;
      }
      for (; i < 2 * n4; i += NTH) d4[i] = __ldcg(src4 + i);
    }
  }
  sel_sync<NTH, BAR>();
  // The a-values of summary x, 16 bytes at a time, from buf or global memory.
  auto group = [&](int x, int i) -> uint4 {
    return resident ? reinterpret_cast<const uint4*>(buf)[(size_t)x * n4 + i] : __ldcg(src4 + (size_t)x * n4 + i);
  };
  // digit 1: bits [29:20]
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    for (int i0 = 0; i0 < n4; i0 += 4 * NTH) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * NTH + tid;
        v[j] = i < n4 ? group(x, i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned w[4] = {sel_bits(v[j].x), sel_bits(v[j].y), sel_bits(v[j].z), sel_bits(v[j].w)};
        if (i0 + j * NTH + tid < n4) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (w[k] >= MIN_MASS_BITS) hist_add(sm, x, (int)(w[k] >> 20), fixed40(w[k]));
        }
      }
    }
  }
  sel_sync<NTH, BAR>();
  pick_digit<NTH, BAR>(sm, 20, true, p, tid);
  sel_sync<NTH, BAR>();
  // stream compaction of the first digit's bin
  const unsigned cbase = resident ? (unsigned)(2 * ndem) : 0u;
  const bool compact = cbase + sm->st[0].cnt_eq + sm->st[1].cnt_eq <= (unsigned)cap;
  const unsigned off1 = cbase + sm->st[0].cnt_eq;
  if (compact) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (sm->st[x].done) continue;
      const unsigned want = sm->st[x].prefix >> 20;
      unsigned* dst = buf + (x ? off1 : cbase);
      for (int i0 = 0; i0 < n4; i0 += 4 * NTH) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * NTH + tid;
          v[j] = i < n4 ? group(x, i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool in = i0 + j * NTH + tid < n4;
          const unsigned w[4] = {sel_bits(v[j].x), sel_bits(v[j].y), sel_bits(v[j].z), sel_bits(v[j].w)};
          const bool keep[4] = {in && (w[0] >> 20) == want, in && (w[1] >> 20) == want,
                                in && (w[2] >> 20) == want, in && (w[3] >> 20) == want};
          warp_append4(w, keep, dst, &sm->ncomp[x], lane);
        }
      }
    }
  }
  // digits 2 and 3: bits [19:10] and [9:0] of the values matching the prefix
#pragma unroll
  for (int ro = 0; ro < 2; ++ro) {
    const int sh = ro == 0 ? 10 : 0;
    const unsigned hi_mask = ro == 0 ? 0x3FF00000u : 0x3FFFFC00u;  // bits already fixed
    sel_sync<NTH, BAR>();
    clear_hist<NTH>(sm, tid);
    sel_sync<NTH, BAR>();
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (sm->st[x].done) continue;
      const unsigned pf = sm->st[x].prefix;
      if (compact) {
        const unsigned n = sm->ncomp[x];
        const unsigned* bb = buf + (x ? off1 : cbase);
        for (unsigned i = tid; i < n; i += NTH) {
          const unsigned u = bb[i];
          if ((u & hi_mask) == pf) hist_add(sm, x, (int)((u >> sh) & (SEL_BINS - 1)), fixed40(u));
        }
      } else {
        for (int i0 = 0; i0 < n4; i0 += 4 * NTH) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * NTH + tid;
            v[j] = i < n4 ? group(x, i) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (i0 + j * NTH + tid >= n4) continue;
            const unsigned w[4] = {sel_bits(v[j].x), sel_bits(v[j].y), sel_bits(v[j].z), sel_bits(v[j].w)};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if ((w[k] & hi_mask) == pf) hist_add(sm, x, (int)((w[k] >> sh) & (SEL_BINS - 1)), fixed40(w[k]));
          }
        }
      }
    }
    sel_sync<NTH, BAR>();
    pick_digit<NTH, BAR>(sm, sh, false, p, tid);
  }
  sel_sync<NTH, BAR>();
  unsigned res = 0;
  if (tid < 2) {
    const DpState& s = sm->st[tid];
    if (!s.done) {
      const unsigned long long tf = fixed40(s.prefix);
      const unsigned long long need = s.target - s.mass_above;
      unsigned j = s.cnt_eq;
      if (tf > 0) {
        const unsigned long long q = (need + tf - 1) / tf;
        if (q < j) j = (unsigned)q;
      }
      if (j < 1) j = 1;
      res = s.cnt_above + j;
      if (s.bad) atomicOr(err, ERR_BAD_COUNT);
    }
  }
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

// Thread x < 2 of the select stores D_p of summary x and adds it to the sums.
__device__ __forceinline__ void write_demand(const DemandArgs& a, int r, int unit, int x, unsigned k) {
  if (x < 2) {
    const int units = a.L * a.Hkv;
    a.kout[((size_t)r * units + unit) * 2 + x] = (int32_t)k;
    atomicAdd(a.ksum + (size_t)r * 2 + x, (unsigned long long)k);
  }
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
