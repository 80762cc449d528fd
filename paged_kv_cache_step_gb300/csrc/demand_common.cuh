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

// log2 of a positive double: exponent exactly, mantissa through lg2.approx.
__device__ __forceinline__ float log2_pos(double s) {
  int e;
  const double m = frexp(s, &e);  // s = m 2^e, m in [0.5, 1)
  return (float)e + lg2((float)m);
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
// (m, s) with s = sum 2^(z - m); an empty set is (-inf, 0).
__device__ __forceinline__ void online(float& m, float& s, float z) {
  const float mn = fmaxf(m, z);
  s = s * ex2(m - mn) + ex2(z - mn);
  m = mn;
}

__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  if (s2 <= 0.f) return;
  if (s <= 0.f) {
    m = m2;
    s = s2;
    return;
  }
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

// Merge the cluster's statistics into base-2 log-sum-exps:
// lse_dem[row] over C_t and lse_cmp[row] over C_cmp (C_t plus the tail).
template <int ROWS>
__device__ __forceinline__ void merge_stats(const StatXchg* xg, int csize, float* lse_dem, float* lse_cmp) {
  const int tid = threadIdx.x;
  if (tid < ROWS) {
    float md = -INFINITY, mt = -INFINITY;
    for (int c = 0; c < csize; ++c) {
      if (xg->s[c][0][tid] > 0.f) md = fmaxf(md, xg->m[c][0][tid]);
      if (xg->s[c][1][tid] > 0.f) mt = fmaxf(mt, xg->m[c][1][tid]);
    }
    double sd = 0.0, stl = 0.0;
    for (int c = 0; c < csize; ++c) {
      const float s0 = xg->s[c][0][tid], s1 = xg->s[c][1][tid];
      if (s0 > 0.f) sd += (double)s0 * (double)ex2(xg->m[c][0][tid] - md);
      if (s1 > 0.f) stl += (double)s1 * (double)ex2(xg->m[c][1][tid] - mt);
    }
    lse_dem[tid] = sd > 0.0 ? md + log2_pos(sd) : 0.f;
    // C_cmp = C_t plus the tail
    const float mc = fmaxf(sd > 0.0 ? md : -INFINITY, stl > 0.0 ? mt : -INFINITY);
    double sc = 0.0;
    if (sd > 0.0) sc += sd * (double)ex2(md - mc);
    if (stl > 0.0) sc += stl * (double)ex2(mt - mc);
    lse_cmp[tid] = sc > 0.0 ? mc + log2_pos(sc) : 0.f;
  }
}

// ---- per-key epilogue ----------------------------------------------------
// z[ROWS] base-2 logits of key i (rows x * G + g).  Writes a^S, a^L for
// i < ndem and the base-2 log importance for i < ncmp.
template <int ROWS>
__device__ __forceinline__ void key_values(const float* z, int i, int ndem, int ncmp, const float* lse_dem,
                                           const float* lse_cmp, float* av, float* sc) {
  constexpr int G = ROWS / 2;
  if (i < ndem) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      float s = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) s += ex2(z[x * G + g] - lse_dem[x * G + g]);
      __stcg(av + (size_t)x * ndem + i, s * (1.0f / G));
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
// walks the digits {exponent, 8, 8, 7 mantissa bits} from the top, keeping
// the bin where the cumulative mass reaches ceil(p * total).  Then
// D_p = #(a > t) + ceil((target - mass(a > t)) / mass(t)).

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

struct DpState {
  unsigned prefix, mask, cnt_above, cnt_eq;
  unsigned long long mass_above, target;
  int bad, done;
};

struct DpSmem {
  unsigned cnt[2][256];
  unsigned mhi[2][256];  // sum of (mass >> 16)
  unsigned mlo[2][256];  // sum of (mass & 0xffff)
  DpState st[2];
  unsigned ncomp[2];
  int compact;
};

// Warp-cooperative histogram update: lanes sharing a bin are summed with one
// reduction and one set of atomics (up to two groups), the rest add directly.
__device__ __forceinline__ void hist_add(DpSmem* sm, int x, int bin, bool valid, unsigned long long w) {
  const int lane = threadIdx.x & 31;
  const unsigned whi = (unsigned)(w >> 16), wlo = (unsigned)(w & 0xFFFFull);
  unsigned act = __ballot_sync(FULL, valid);
#pragma unroll 1
  for (int it = 0; it < 2 && act; ++it) {
    const int leader = __ffs(act) - 1;
    const int lb = __shfl_sync(FULL, bin, leader);
    const unsigned peers = __ballot_sync(FULL, ((act >> lane) & 1u) && bin == lb);
    const unsigned np = __popc(peers);
    if (np < 3) break;
    const bool in = (peers >> lane) & 1u;
    const unsigned shi = __reduce_add_sync(FULL, in ? whi : 0u);
    const unsigned slo = __reduce_add_sync(FULL, in ? wlo : 0u);
    if (lane == leader) {
      atomicAdd(&sm->cnt[x][lb], np);
      atomicAdd(&sm->mhi[x][lb], shi);
      atomicAdd(&sm->mlo[x][lb], slo);
    }
    act &= ~peers;
  }
  if ((act >> lane) & 1u) {
    atomicAdd(&sm->cnt[x][bin], 1u);
    atomicAdd(&sm->mhi[x][bin], whi);
    atomicAdd(&sm->mlo[x][bin], wlo);
  }
}

// Warp x picks the bin of this round (digit at `shift`, `bits` wide).
__device__ __forceinline__ void pick_bin(DpSmem* sm, int x, int shift, int bits, bool first, double p) {
  const int lane = threadIdx.x & 31;
  DpState& st = sm->st[x];
  const int top = 255 - 8 * lane;
  unsigned lc = 0;
  unsigned long long lm = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int b = top - k;
    lc += sm->cnt[x][b];
    lm += ((unsigned long long)sm->mhi[x][b] << 16) + sm->mlo[x][b];
  }
  if (first) {
    unsigned long long tot = lm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
    if (lane == 0) {
      if (tot == 0) {
        st.done = 1;
      } else {
        unsigned long long tg = (unsigned long long)ceil(p * (double)tot);
        if (tg < 1) tg = 1;
        if (tg > tot) tg = tot;
        st.target = tg;
      }
    }
    __syncwarp();
  }
  if (st.done) return;
  const unsigned long long need = st.target - st.mass_above;
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
  const unsigned hit = __ballot_sync(FULL, im >= need);
  const int src = hit ? __ffs(hit) - 1 : 31;
  if (lane == src) {
    unsigned long long cum = im - lm;
    unsigned cnt = ic - lc;
    int chosen = top - 7;
    bool found = false;
    for (int k = 0; k < 8; ++k) {
      const int b = top - k;
      const unsigned long long mb = ((unsigned long long)sm->mhi[x][b] << 16) + sm->mlo[x][b];
      if (cum + mb >= need) {
        chosen = b;
        found = true;
        break;
      }
      cum += mb;
      cnt += sm->cnt[x][b];
    }
    if (!found || !hit) st.bad = 1;
    st.prefix |= (unsigned)chosen << shift;
    st.mask |= ((1u << bits) - 1u) << shift;
    st.mass_above += cum;
    st.cnt_above += cnt;
    st.cnt_eq = sm->cnt[x][chosen];
  }
  __syncwarp();
}

__device__ __forceinline__ void clear_hist(DpSmem* sm) {
  for (int k = threadIdx.x; k < 2 * 256; k += NT) {
    (&sm->cnt[0][0])[k] = 0u;
    (&sm->mhi[0][0])[k] = 0u;
    (&sm->mlo[0][0])[k] = 0u;
  }
}

// D_p of both summaries of one unit from its a-values av[2][ndem] (global,
// written by the unit's CTAs).  buf: shared scratch of `cap` words for the
// candidates that survive the exponent round.  All threads call it; thread
// x < 2 returns D_p for summary x.
__device__ __noinline__ static unsigned coverage_demand(const float* av, int ndem, double p, unsigned* buf, int cap, DpSmem* sm,
                                    int* err) {
  const int tid = threadIdx.x;
  if (tid < 2) {
    DpState& s = sm->st[tid];
    s.prefix = 0u;
    s.mask = 0u;
    s.cnt_above = 0u;
    s.cnt_eq = 0u;
    s.mass_above = 0ull;
    s.target = 0ull;
    s.bad = 0;
    s.done = 0;
    sm->ncomp[tid] = 0u;
  }
  clear_hist(sm);
  __syncthreads();
  const unsigned* src = reinterpret_cast<const unsigned*>(av);
  // round 0: exponent digit, straight from global memory (L2)
  for (int base = 0; base < ndem; base += NT) {
    const int i = base + tid;
    const bool v = i < ndem;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const unsigned u = v ? __ldcg(src + (size_t)x * ndem + i) : 0u;
      hist_add(sm, x, (int)(u >> 23), v, fixed40(u));
    }
  }
  __syncthreads();
  if ((tid >> 5) < 2) pick_bin(sm, tid >> 5, 23, 8, true, p);
  __syncthreads();
  // stream compaction of the exponent bin's members (ballot + warp prefix)
  const bool compact = sm->st[0].cnt_eq + sm->st[1].cnt_eq <= (unsigned)cap;
  const unsigned off1 = sm->st[0].cnt_eq;
  if (compact) {
    const int lane = tid & 31;
    for (int base = 0; base < ndem; base += NT) {
      const int i = base + tid;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const unsigned u = i < ndem ? __ldcg(src + (size_t)x * ndem + i) : 0u;
        const bool keep = i < ndem && !sm->st[x].done && (u >> 23) == (sm->st[x].prefix >> 23);
        const unsigned bal = __ballot_sync(FULL, keep);
        unsigned pos = 0;
        if (lane == 0 && bal) pos = atomicAdd(&sm->ncomp[x], (unsigned)__popc(bal));
        pos = __shfl_sync(FULL, pos, 0);
        if (keep) buf[(x ? off1 : 0u) + pos + __popc(bal & ((1u << lane) - 1u))] = u;
      }
    }
  }
#pragma unroll
  for (int ro = 0; ro < 3; ++ro) {
    __syncthreads();
    clear_hist(sm);
    __syncthreads();
    const int sh = ro == 0 ? 15 : (ro == 1 ? 7 : 0);   // mantissa digits of 8, 8, 7 bits
    const int width = ro == 2 ? 7 : 8;
    const unsigned dm = (1u << width) - 1u;
    for (int x = 0; x < 2; ++x) {
      if (sm->st[x].done) continue;
      const unsigned pf = sm->st[x].prefix, mk = sm->st[x].mask;
      if (compact) {
        const unsigned n = sm->ncomp[x];
        const unsigned* b = buf + (x ? off1 : 0u);
        for (unsigned base = 0; base < n; base += NT) {
          const unsigned i = base + tid;
          const unsigned u = i < n ? b[i] : 0u;
          const bool v = i < n && (u & mk) == pf;
          hist_add(sm, x, (int)((u >> sh) & dm), v, fixed40(u));
        }
      } else {
        for (int base = 0; base < ndem; base += NT) {
          const int i = base + tid;
          const unsigned u = i < ndem ? __ldcg(src + (size_t)x * ndem + i) : 0u;
          const bool v = i < ndem && (u & mk) == pf;
          hist_add(sm, x, (int)((u >> sh) & dm), v, fixed40(u));
        }
      }
    }
    __syncthreads();
    if ((tid >> 5) < 2) pick_bin(sm, tid >> 5, sh, width, false, p);
  }
  __syncthreads();
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
  return res;
}

// After a CTA has written its a-values: the last of the unit's C CTAs to get
// here (global ticket) computes D_p for the unit.  Returns true in that CTA.
__device__ __forceinline__ bool last_of_unit(const DemandArgs& a, const Unit& u, int* flag_smem) {
  __threadfence();  // this thread's a-values before the ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* t = a.tickets + (size_t)u.r * (a.L * a.Hkv) + u.unit;
    const unsigned old = atomicAdd(t, 1u);
    const bool last = old == (unsigned)(a.C - 1);
    if (last) {
      *t = 0u;  // ready for the next call
      __threadfence();
    }
    *flag_smem = last ? 1 : 0;
  }
  __syncthreads();
  return *flag_smem != 0;
}

__device__ __forceinline__ void write_demand(const DemandArgs& a, const Unit& u, unsigned k) {
  const int x = threadIdx.x;
  if (x < 2) {
    const int units = a.L * a.Hkv;
    a.kout[((size_t)u.r * units + u.unit) * 2 + x] = (int32_t)k;
    atomicAdd(a.ksum + (size_t)u.r * 2 + x, (unsigned long long)k);
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
