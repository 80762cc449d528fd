// Boundary demand kernel for sm_103a: GrowPage Sec. 3.2 Eqs. 2, 7 and
// App. E.1 (scores of the calibrated summaries against every cached key,
// softmax over C_t, GQA mean, p-coverage demand D_p), plus the Eq. 9
// importance over the compression candidates, cached for Compress & Hold.
//
// Work unit: one (request, layer, KV head).  A unit is owned by one
// thread-block cluster of C CTAs; CTA c scores logical pages
// [c*ppc, (c+1)*ppc) and keeps every logit of its keys in shared memory,
// so K is read from HBM exactly once and no logit round-trips through
// global memory.  Distributed shared memory joins the CTAs:
//   1. scan     -- 16-byte streaming loads of K rows (each lane pair owns a
//                  key, each lane half of its 16-byte chunks, so one warp
//                  load covers whole 32-byte sectors), fp32 FMA against the
//                  2G summary rows broadcast from shared memory, lane-pair
//                  shuffle to finish the dot products;
//   2. softmax  -- per-row (max, sum of 2^(z-max)) over C_t and over the
//                  compression candidates, merged across the cluster;
//   3. values   -- a^S, a^L (mean over the G query heads) per key of C_t,
//                  and log2 max(a^S, a^L) per compression candidate,
//                  written to the importance cache;
//   4. D_p      -- radix select on the fp32 bit patterns of a^x (4 rounds
//                  of 8-bit digits) with per-bucket counts and exact
//                  fixed-point (2^-60) masses, histograms summed across the
//                  cluster, walking buckets from the top until the mass
//                  reaches p * total; then D_p = #(a > t) + ceil((p*total -
//                  mass(a > t)) / t).
// Logits are in base 2: the summaries arrive pre-scaled by log2(e)/sqrt(d).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdint>

#include "gp_kernels.h"

namespace cg = cooperative_groups;

namespace gp {
namespace {

constexpr int NT = 256;   // threads per CTA
constexpr int NW = 8;     // warps per CTA
constexpr int PAGE = 256; // tokens per page (b)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Probability -> exact fixed point with 60 fractional bits.
__device__ __forceinline__ unsigned long long to_fixed(float v) {
  return __float2ull_rn(v * 1.152921504606846976e18f);
}

// Add (count 1, mass w) of every valid lane to bin `bin`, one atomic pair
// per distinct bin in the warp.  All 32 lanes must call it.
__device__ __forceinline__ void warp_hist_add(unsigned* cnt, unsigned long long* mass,
                                              int bin, bool valid, unsigned long long w) {
  const int key = valid ? bin : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const unsigned l0 = (unsigned)(w & 0x1FFFFFull);
  const unsigned l1 = (unsigned)((w >> 21) & 0x1FFFFFull);
  const unsigned l2 = (unsigned)(w >> 42);
  const unsigned s0 = __reduce_add_sync(peers, l0);
  const unsigned s1 = __reduce_add_sync(peers, l1);
  const unsigned s2 = __reduce_add_sync(peers, l2);
  const int lane = threadIdx.x & 31;
  if (valid && lane == __ffs(peers) - 1) {
    atomicAdd(&cnt[bin], (unsigned)__popc(peers));
    atomicAdd(&mass[bin], (unsigned long long)s0 + ((unsigned long long)s1 << 21) +
                              ((unsigned long long)s2 << 42));
  }
}

struct SelState {
  unsigned prefix, mask, cnt_above, cnt_eq;
  unsigned long long mass_above, target;
  int bad;
};

template <bool BF16, int D, int ROWS>
struct Cfg {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int RB = D * ESZ;       // bytes per key row
  static constexpr int NCH = RB / 16;      // 16-byte chunks per row
  static constexpr int EPC = 16 / ESZ;     // elements per chunk
  static constexpr int HALF = NCH / 2;     // chunks per lane (lane pair per key)
  static constexpr int KPT = 2;            // keys per lane pair per group
  static constexpr int GROUP = 16 * KPT;   // keys per warp group
  static constexpr int GPP = PAGE / GROUP; // groups per page
  static_assert(NCH % 2 == 0, "row must hold an even number of chunks");
};

template <bool BF16, int EPC>
__device__ __forceinline__ void unpack(const uint4& v, float* f) {
  if constexpr (BF16) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
  } else {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
}

// Shared-memory carve-up (bytes, 16-aligned pieces).
template <int D, int ROWS>
struct Smem {
  size_t qs, z, mst, sst, lsm, lsl, hcnt, hmass, ccnt, cmass, redf, redd, sel, phys, total;
  __host__ __device__ Smem(int ppc) {
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 15) & ~size_t(15); return r; };
    qs = take(sizeof(float) * ROWS * D);
    z = take(sizeof(float) * (size_t)ppc * PAGE * ROWS);
    mst = take(sizeof(float) * 2 * ROWS);
    sst = take(sizeof(double) * 2 * ROWS);
    lsm = take(sizeof(float) * 2 * ROWS);
    lsl = take(sizeof(float) * 2 * ROWS);
    hcnt = take(sizeof(unsigned) * 2 * 2 * 256);
    hmass = take(sizeof(unsigned long long) * 2 * 2 * 256);
    ccnt = take(sizeof(unsigned) * 2 * 256);
    cmass = take(sizeof(unsigned long long) * 2 * 256);
    redf = take(sizeof(float) * NW * 2 * ROWS);
    redd = take(sizeof(double) * NW * 2 * ROWS);
    sel = take(sizeof(SelState) * 2);
    phys = take(sizeof(int) * 64);
    total = o;
  }
};

template <bool BF16, int D, int ROWS>
__global__ void __launch_bounds__(NT, 2) k_demand(DemandArgs a) {
  using C = Cfg<BF16, D, ROWS>;
  extern __shared__ __align__(16) unsigned char smem[];
  const Smem<D, ROWS> L(a.ppc);
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  float* zb = reinterpret_cast<float*>(smem + L.z);
  float* mst = reinterpret_cast<float*>(smem + L.mst);
  double* sst = reinterpret_cast<double*>(smem + L.sst);
  float* lsm = reinterpret_cast<float*>(smem + L.lsm);
  float* lsl = reinterpret_cast<float*>(smem + L.lsl);
  unsigned* hcnt = reinterpret_cast<unsigned*>(smem + L.hcnt);
  unsigned long long* hmass = reinterpret_cast<unsigned long long*>(smem + L.hmass);
  unsigned* ccnt = reinterpret_cast<unsigned*>(smem + L.ccnt);
  unsigned long long* cmass = reinterpret_cast<unsigned long long*>(smem + L.cmass);
  float* redf = reinterpret_cast<float*>(smem + L.redf);
  double* redd = reinterpret_cast<double*>(smem + L.redd);
  SelState* st = reinterpret_cast<SelState*>(smem + L.sel);
  int* phys = reinterpret_cast<int*>(smem + L.phys);

  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int csize = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.L * a.Hkv;
  const int wi = blockIdx.x / a.C;  // the cluster's work item; rank = blockIdx.x % C
  const int r = a.work[wi / units];
  const int unit = wi % units;
  const int layer = unit / a.Hkv, h = unit % a.Hkv;
  const DevReq rq = a.reqs[r];
  const int P = rq.num_pages;
  const int ndem = (P - 1) * PAGE;
  const int ncmp = P * PAGE - a.R;
  const int j0 = crank * a.ppc;
  const int npg = max(0, min(P, j0 + a.ppc) - j0);
  const int G = ROWS / 2;

  // ---- setup: summaries of this unit, physical pages of this CTA --------
  {
    const float* src = a.qt + ((size_t)r * units + unit) * ROWS * D;
    for (int i = tid; i < ROWS * D; i += NT) qs[i] = src[i];
    if (tid < npg) {
      int pg = a.bt[rq.bt_off + j0 + tid];
      if (pg < 0 || pg >= a.num_pages_total) {
        atomicOr(a.err, ERR_BAD_PAGE);
        pg = 0;
      }
      phys[tid] = pg;
    }
    if (tid < 2) {
      st[tid].prefix = 0; st[tid].mask = 0; st[tid].cnt_above = 0; st[tid].cnt_eq = 0;
      st[tid].mass_above = 0; st[tid].target = 0; st[tid].bad = 0;
    }
  }
  __syncthreads();

  // ---- 1. scan: z = qt . k for the CTA's keys ----------------------------
  {
    const int ngroups = npg * C::GPP;
    const int ngw = warp < ngroups ? (ngroups - warp + NW - 1) / NW : 0;
    const int total = ngw * C::HALF;
    const int t = lane >> 1, par = lane & 1;
    const size_t head_stride = (size_t)PAGE * C::RB;
    const unsigned char* kb = static_cast<const unsigned char*>(a.k_cache);
    const size_t layer_off = (size_t)layer * a.num_pages_total;

    auto row_ptr = [&](int step, int kk) -> const uint4* {
      const int gl = warp + NW * (step / C::HALF);     // local group
      const int s = step % C::HALF;
      const int pl = gl / C::GPP;
      const int slot = (gl % C::GPP) * C::GROUP + t + 16 * kk;
      const unsigned char* base =
          kb + ((layer_off + phys[pl]) * a.Hkv + h) * head_stride + (size_t)slot * C::RB;
      return reinterpret_cast<const uint4*>(base) + (2 * s + par);
    };

    float acc[C::KPT][ROWS];
    auto compute = [&](int step, const uint4* buf) {
      const int s = step % C::HALF;
      if (s == 0) {
#pragma unroll
        for (int kk = 0; kk < C::KPT; ++kk)
#pragma unroll
          for (int rr = 0; rr < ROWS; ++rr) acc[kk][rr] = 0.f;
      }
      float kf[C::KPT][C::EPC];
#pragma unroll
      for (int kk = 0; kk < C::KPT; ++kk) unpack<BF16, C::EPC>(buf[kk], kf[kk]);
      const int d0 = (2 * s + par) * C::EPC;
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) {
        const float4* qp = reinterpret_cast<const float4*>(qs + rr * D + d0);
#pragma unroll
        for (int e4 = 0; e4 < C::EPC / 4; ++e4) {
          const float4 q = qp[e4];
#pragma unroll
          for (int kk = 0; kk < C::KPT; ++kk) {
            float v = acc[kk][rr];
            v = fmaf(kf[kk][4 * e4 + 0], q.x, v);
            v = fmaf(kf[kk][4 * e4 + 1], q.y, v);
            v = fmaf(kf[kk][4 * e4 + 2], q.z, v);
            v = fmaf(kf[kk][4 * e4 + 3], q.w, v);
            acc[kk][rr] = v;
          }
        }
      }
      if (s == C::HALF - 1) {
        const int gl = warp + NW * (step / C::HALF);
#pragma unroll
        for (int kk = 0; kk < C::KPT; ++kk) {
          float out[ROWS / 2];
#pragma unroll
          for (int rr = 0; rr < ROWS / 2; ++rr) {
            const float send = par ? acc[kk][rr] : acc[kk][rr + ROWS / 2];
            const float mine = par ? acc[kk][rr + ROWS / 2] : acc[kk][rr];
            out[rr] = mine + __shfl_xor_sync(0xffffffffu, send, 1);
          }
          const int kl = gl * C::GROUP + t + 16 * kk;
          float* dst = zb + (size_t)kl * ROWS + par * (ROWS / 2);
          if constexpr (ROWS / 2 == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(out[0], out[1], out[2], out[3]);
          } else if constexpr (ROWS / 2 == 2) {
            *reinterpret_cast<float2*>(dst) = make_float2(out[0], out[1]);
          } else {
#pragma unroll
            for (int rr = 0; rr < ROWS / 2; ++rr) dst[rr] = out[rr];
          }
        }
      }
    };

    uint4 b0[C::KPT], b1[C::KPT], b2[C::KPT];
    auto load = [&](int step, uint4* buf) {
#pragma unroll
      for (int kk = 0; kk < C::KPT; ++kk) buf[kk] = ld_stream(row_ptr(step, kk));
    };
    if (total > 0) load(0, b0);
    if (total > 1) load(1, b1);
    for (int i = 0; i < total; i += 3) {
      if (i + 2 < total) load(i + 2, b2);
      compute(i, b0);
      if (i + 3 < total) load(i + 3, b0);
      if (i + 1 < total) compute(i + 1, b1);
      if (i + 4 < total) load(i + 4, b1);
      if (i + 2 < total) compute(i + 2, b2);
    }
  }
  __syncthreads();

  const int base_slot = j0 * PAGE;
  const int nloc = npg * PAGE;

  // ---- 2. softmax statistics per row over C_t (dem) and candidates (cmp) --
  {
    float md[ROWS], mc[ROWS];
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) { md[rr] = -FLT_MAX; mc[rr] = -FLT_MAX; }
    for (int kl = tid; kl < nloc; kl += NT) {
      const int i = base_slot + kl;
      const float* z = zb + (size_t)kl * ROWS;
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) {
        const float v = z[rr];
        if (i < ndem) md[rr] = fmaxf(md[rr], v);
        if (i < ncmp) mc[rr] = fmaxf(mc[rr], v);
      }
    }
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        md[rr] = fmaxf(md[rr], __shfl_xor_sync(0xffffffffu, md[rr], o));
        mc[rr] = fmaxf(mc[rr], __shfl_xor_sync(0xffffffffu, mc[rr], o));
      }
      if (lane == 0) { redf[warp * 2 * ROWS + rr] = md[rr]; redf[warp * 2 * ROWS + ROWS + rr] = mc[rr]; }
    }
    __syncthreads();
    if (tid < 2 * ROWS) {
      float m = -FLT_MAX;
      for (int w = 0; w < NW; ++w) m = fmaxf(m, redf[w * 2 * ROWS + tid]);
      mst[tid] = m;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) { md[rr] = mst[rr]; mc[rr] = mst[ROWS + rr]; }
    float sd[ROWS], sc[ROWS];
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) { sd[rr] = 0.f; sc[rr] = 0.f; }
    for (int kl = tid; kl < nloc; kl += NT) {
      const int i = base_slot + kl;
      const float* z = zb + (size_t)kl * ROWS;
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) {
        const float v = z[rr];
        if (i < ndem) sd[rr] += ex2(v - md[rr]);
        if (i < ncmp) sc[rr] += ex2(v - mc[rr]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
      double dd = sd[rr], dc = sc[rr];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        dd += __shfl_xor_sync(0xffffffffu, dd, o);
        dc += __shfl_xor_sync(0xffffffffu, dc, o);
      }
      if (lane == 0) { redd[warp * 2 * ROWS + rr] = dd; redd[warp * 2 * ROWS + ROWS + rr] = dc; }
    }
    __syncthreads();
    if (tid < 2 * ROWS) {
      double s = 0.0;
      for (int w = 0; w < NW; ++w) s += redd[w * 2 * ROWS + tid];
      sst[tid] = s;
    }
  }
  cluster.sync();
  // merge (max, sum) across the cluster: lse = M + log2(S), kept as (M, log2 S)
  if (tid < 2 * ROWS) {
    float M = -FLT_MAX;
    for (int c = 0; c < csize; ++c) {
      const double s = *cluster.map_shared_rank(sst + tid, c);
      const float m = *cluster.map_shared_rank(mst + tid, c);
      if (s > 0.0) M = fmaxf(M, m);
    }
    double S = 0.0;
    for (int c = 0; c < csize; ++c) {
      const double s = *cluster.map_shared_rank(sst + tid, c);
      const float m = *cluster.map_shared_rank(mst + tid, c);
      if (s > 0.0) S += s * exp2((double)(m - M));
    }
    lsm[tid] = S > 0.0 ? M : 0.f;
    lsl[tid] = S > 0.0 ? (float)log2(S) : 0.f;
  }
  __syncthreads();

  // ---- 3. per-key distributions and importance cache ---------------------
  {
    float* scores = a.scores + rq.score_off + (size_t)unit * ncmp;
    float* dbg = (a.dbg && rq.dbg_off >= 0) ? a.dbg + rq.dbg_off + (size_t)unit * 2 * ndem : nullptr;
    const float inv_g = 1.0f / (float)G;
    const float lg_g = lg2((float)G);
    for (int kl = tid; kl < nloc; kl += NT) {
      const int i = base_slot + kl;
      float* zp = zb + (size_t)kl * ROWS;
      float z[ROWS];
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) z[rr] = zp[rr];
      if (i < ndem) {
        float ax[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          float s = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int rr = x * G + g;
            s += ex2((z[rr] - lsm[rr]) - lsl[rr]);
          }
          ax[x] = s * inv_g;
        }
        zp[0] = ax[0];
        zp[1] = ax[1];
        if (dbg) {
          dbg[i] = ax[0];
          dbg[ndem + i] = ax[1];
        }
      }
      if (i < ncmp) {
        float best = -FLT_MAX;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          float tv[ROWS / 2];
          float m = -FLT_MAX;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int rr = ROWS + x * G + g;   // cmp statistics live at [ROWS, 2 ROWS)
            tv[g] = (z[x * G + g] - lsm[rr]) - lsl[rr];
            m = fmaxf(m, tv[g]);
          }
          float s = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) s += ex2(tv[g] - m);
          best = fmaxf(best, m + lg2(s) - lg_g);
        }
        scores[i] = best;
      }
    }
  }
  __syncthreads();

  // ---- 4. D_p by radix select over C_t (both summaries at once) ----------
  unsigned dres[2] = {0u, 0u};
  if (ndem > 0) {
    const int iters = npg;  // nloc / NT
    for (int ro = 0; ro < 4; ++ro) {
      const int buf = ro & 1;
      const int shift = 24 - 8 * ro;
      unsigned* hc = hcnt + buf * 512;
      unsigned long long* hm = hmass + buf * 512;
      hc[tid] = 0u; hc[256 + tid] = 0u;
      hm[tid] = 0ull; hm[256 + tid] = 0ull;
      __syncthreads();
      const unsigned pf0 = st[0].prefix, mk0 = st[0].mask;
      const unsigned pf1 = st[1].prefix, mk1 = st[1].mask;
      for (int it = 0; it < iters; ++it) {
        const int kl = tid + it * NT;
        const bool isdem = base_slot + kl < ndem;
        const float* zp = zb + (size_t)kl * ROWS;
        const float v0 = zp[0], v1 = zp[1];
        const unsigned u0 = __float_as_uint(v0), u1 = __float_as_uint(v1);
        warp_hist_add(hc, hm, (u0 >> shift) & 255u, isdem && ((u0 & mk0) == pf0), to_fixed(v0));
        warp_hist_add(hc + 256, hm + 256, (u1 >> shift) & 255u, isdem && ((u1 & mk1) == pf1),
                      to_fixed(v1));
      }
      cluster.sync();
      // sum the cluster's histograms
      {
        unsigned c0 = 0, c1 = 0;
        unsigned long long m0 = 0, m1 = 0;
        for (int c = 0; c < csize; ++c) {
          const unsigned* rc = cluster.map_shared_rank(hc, c);
          const unsigned long long* rm = cluster.map_shared_rank(hm, c);
          c0 += rc[tid]; c1 += rc[256 + tid];
          m0 += rm[tid]; m1 += rm[256 + tid];
        }
        ccnt[tid] = c0; ccnt[256 + tid] = c1;
        cmass[tid] = m0; cmass[256 + tid] = m1;
      }
      __syncthreads();
      if (warp < 2) {
        const int x = warp;
        const unsigned* cc = ccnt + 256 * x;
        const unsigned long long* cm = cmass + 256 * x;
        // lane l owns bins [255 - 8 l - 7, 255 - 8 l], walked from the top
        const int top = 255 - 8 * lane;
        unsigned lc = 0;
        unsigned long long lm = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) { lc += cc[top - k]; lm += cm[top - k]; }
        if (ro == 0) {
          unsigned long long tot = lm;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
          if (lane == 0) {
            unsigned long long tg = (unsigned long long)ceil(a.p * (double)tot);
            if (tg < 1) tg = 1;
            if (tg > tot) tg = tot;
            st[x].target = tg;
          }
          __syncwarp();
        }
        const unsigned long long need = st[x].target - st[x].mass_above;
        unsigned long long im = lm;
        unsigned ic = lc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long om = __shfl_up_sync(0xffffffffu, im, o);
          const unsigned oc = __shfl_up_sync(0xffffffffu, ic, o);
          if (lane >= o) { im += om; ic += oc; }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, im >= need);
        int src = hit ? __ffs(hit) - 1 : 31;
        if (lane == src) {
          unsigned long long cum = im - lm;
          unsigned cnt = ic - lc;
          int chosen = top - 7;
          bool found = false;
          for (int k = 0; k < 8; ++k) {
            const int bin = top - k;
            if (cum + cm[bin] >= need) { chosen = bin; found = true; break; }
            cum += cm[bin];
            cnt += cc[bin];
          }
          if (!found || !hit) st[x].bad = 1;
          st[x].prefix |= (unsigned)chosen << shift;
          st[x].mask |= 255u << shift;
          st[x].mass_above += cum;
          st[x].cnt_above += cnt;
          if (ro == 3) st[x].cnt_eq = cc[chosen];
        }
        __syncwarp();
      }
      __syncthreads();
    }
    if (tid < 2) {
      const SelState s = st[tid];
      const unsigned long long tf = to_fixed(__uint_as_float(s.prefix));
      const unsigned long long need = s.target - s.mass_above;
      unsigned j = s.cnt_eq;
      if (tf > 0) {
        const unsigned long long q = (need + tf - 1) / tf;
        if (q < j) j = (unsigned)q;
      }
      if (j < 1) j = 1;
      dres[tid] = s.cnt_above + j;
      if (s.bad) atomicOr(a.err, ERR_BAD_COUNT);
    }
  }

  // ---- 5. outputs ---------------------------------------------------------
  if (crank == 0 && tid < 2) {
    a.kout[((size_t)r * units + unit) * 2 + tid] = (int32_t)dres[tid];
    atomicAdd(a.ksum + (size_t)r * 2 + tid, (unsigned long long)dres[tid]);
  }
  cluster.sync();  // keep this CTA's shared memory alive for its peers
}

template <bool BF16, int D, int ROWS>
cudaError_t launch_t(const DemandArgs& a, cudaStream_t s) {
  auto kern = k_demand<BF16, D, ROWS>;
  const size_t smem = Smem<D, ROWS>(a.ppc).total;
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

}  // namespace

size_t demand_smem_bytes(int D, int G, int ppc) {
  if (D == 128 && G == 4) return Smem<128, 8>(ppc).total;
  if (D == 128 && G == 2) return Smem<128, 4>(ppc).total;
  if (D == 64 && G == 4) return Smem<64, 8>(ppc).total;
  if (D == 64 && G == 2) return Smem<64, 4>(ppc).total;
  return 0;
}

cudaError_t launch_demand(const DemandArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE || a.C < 1 || a.C > 16 || a.ppc < 1 || a.ppc > 64) return cudaErrorInvalidValue;
  const bool bf = !a.kv_f32;
  if (a.D == 128 && a.G == 4) return bf ? launch_t<true, 128, 8>(a, s) : launch_t<false, 128, 8>(a, s);
  if (a.D == 128 && a.G == 2) return bf ? launch_t<true, 128, 4>(a, s) : launch_t<false, 128, 4>(a, s);
  if (a.D == 64 && a.G == 4) return bf ? launch_t<true, 64, 8>(a, s) : launch_t<false, 64, 8>(a, s);
  if (a.D == 64 && a.G == 2) return bf ? launch_t<true, 64, 4>(a, s) : launch_t<false, 64, 4>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
