// Boundary demand kernel, CUDA-core variant (fp32 FMA): GrowPage Sec. 3.2
// Eqs. 2, 7 and App. E.1, plus the Eq. 9 importance cached for Compress &
// Hold.  It serves fp32 caches (and bf16 ones when forced, or when the K
// cache cannot be described by a tensor map); bf16 caches otherwise take the
// tcgen05 variant (k_demand_tc.cu).
//
// Work unit: one (request, layer, KV head), owned by a cluster of C CTAs;
// CTA c scores the balanced page range [c P / C, (c+1) P / C) (at most ppc
// pages) and keeps its logits in shared memory, so K is read from HBM once:
//   1. scan     -- 16-byte streaming loads of K rows (a lane pair per key,
//                  each lane half of the row's 16-byte chunks, so a warp load
//                  covers whole 32-byte sectors), fp32 FMA against the 2G
//                  summary rows broadcast from shared memory, a lane-pair
//                  shuffle to finish each dot product;
//   2. softmax  -- online (max, sum of 2^(z-max)) per row over C_t and over
//                  the last page's other candidates, pushed to every rank of
//                  the cluster through distributed shared memory and merged;
//   3. values   -- a^S, a^L per key of C_t and log2 importance per
//                  candidate, written to global memory;
//   4. D_p      -- the last CTA of the unit to finish runs the radix select
//                  of demand_common.cuh over the unit's a-values.
#include <cuda_bf16.h>

#include "demand_common.cuh"

namespace gp {
namespace {

using namespace dem;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <bool BF16, int D>
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

template <bool BF16>
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
  size_t qs, z, xg, part, lse, phys, dp, flag, total;
  __host__ __device__ Smem(int ppc) {
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 15) & ~size_t(15); return r; };
    qs = take(sizeof(float) * ROWS * D);
    z = take(sizeof(float) * (size_t)ppc * PAGE * ROWS);
    xg = take(sizeof(StatXchg));
    part = take(sizeof(float) * NW * 2 * 2 * ROWS);
    lse = take(sizeof(float) * 2 * ROWS);
    phys = take(sizeof(int) * 64);
    dp = take(sizeof(DpSmem));
    flag = take(sizeof(int) * 4);
    total = o;
  }
};

template <bool BF16, int D, int ROWS>
__global__ void __launch_bounds__(NT, 2) k_demand_ffma(const __grid_constant__ DemandArgs a) {
  using C = Cfg<BF16, D>;
  extern __shared__ __align__(16) unsigned char smem[];
  const Smem<D, ROWS> L(a.ppc);
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  float* zb = reinterpret_cast<float*>(smem + L.z);
  StatXchg* xg = reinterpret_cast<StatXchg*>(smem + L.xg);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* lse_dem = reinterpret_cast<float*>(smem + L.lse);
  float* lse_cmp = lse_dem + ROWS;
  int* phys = reinterpret_cast<int*>(smem + L.phys);
  DpSmem* dps = reinterpret_cast<DpSmem*>(smem + L.dp);
  int* flag = reinterpret_cast<int*>(smem + L.flag);

  cluster_arrive_relaxed();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Unit u = make_unit(a);
  const int units = a.L * a.Hkv;

  // ---- setup: summaries of this unit, physical pages of this CTA --------
  {
    const float* src = a.qt + ((size_t)u.r * units + u.unit) * ROWS * D;
    for (int i = tid; i < ROWS * D; i += NT) qs[i] = src[i];
    if (tid < u.npg) phys[tid] = checked_page(a, u, u.j0 + tid);
  }
  __syncthreads();

  // ---- 1. scan: z = qt . k for the CTA's keys ----------------------------
  {
    const int ngroups = u.npg * C::GPP;
    const int ngw = warp < ngroups ? (ngroups - warp + NW - 1) / NW : 0;
    const int total = ngw * C::HALF;
    const int t = lane >> 1, par = lane & 1;
    const size_t head_stride = (size_t)PAGE * C::RB;
    const unsigned char* kb = static_cast<const unsigned char*>(a.k_cache);
    const size_t layer_off = (size_t)u.layer * a.num_pages_total;

    auto row_ptr = [&](int step, int kk) -> const uint4* {
      const int gl = warp + NW * (step / C::HALF);  // local group
      const int s = step % C::HALF;
      const int pl = gl / C::GPP;
      const int slot = (gl % C::GPP) * C::GROUP + t + 16 * kk;
      const unsigned char* base = kb + ((layer_off + phys[pl]) * a.Hkv + u.h) * head_stride + (size_t)slot * C::RB;
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
      for (int kk = 0; kk < C::KPT; ++kk) unpack<BF16>(buf[kk], kf[kk]);
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
            out[rr] = mine + __shfl_xor_sync(FULL, send, 1);
          }
          const int kl = gl * C::GROUP + t + 16 * kk;
          float* dst = zb + (size_t)kl * ROWS + par * (ROWS / 2);
#pragma unroll
          for (int rr = 0; rr < ROWS / 2; ++rr) dst[rr] = out[rr];
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

  const int base_slot = u.j0 * PAGE;
  const int nloc = u.npg * PAGE;

  // ---- 2. softmax statistics: C_t keys (set 0) and the tail (set 1) -----
  {
    float m[2][ROWS], s[2][ROWS];
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
      m[0][rr] = m[1][rr] = NEG;
      s[0][rr] = s[1][rr] = 0.f;
    }
    for (int kl = tid; kl < nloc; kl += NT) {
      const int i = base_slot + kl;
      if (i >= u.ncmp) continue;
      const int set = i < u.ndem ? 0 : 1;
      const float* z = zb + (size_t)kl * ROWS;
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) {
        if (set == 0) online(m[0][rr], s[0][rr], z[rr]);
        else online(m[1][rr], s[1][rr], z[rr]);
      }
    }
#pragma unroll
    for (int set = 0; set < 2; ++set)
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) {
        warp_combine(m[set][rr], s[set][rr]);
        if (lane == 0) {
          part[((warp * 2 + set) * ROWS + rr) * 2 + 0] = m[set][rr];
          part[((warp * 2 + set) * ROWS + rr) * 2 + 1] = s[set][rr];
        }
      }
  }
  __syncthreads();
  float cm = NEG, cs = 0.f;
  if (tid < 2 * ROWS) {
    for (int w = 0; w < NW; ++w) combine(cm, cs, part[(w * 2 * ROWS + tid) * 2], part[(w * 2 * ROWS + tid) * 2 + 1]);
  }
  push_stats<ROWS>(xg, u.crank, a.C, cm, cs);
  merge_stats<ROWS>(xg, a.C, lse_dem, lse_cmp);
  __syncthreads();

  // ---- 3. per-key distributions and importance cache ---------------------
  {
    float* sc = a.scores + u.rq.score_off + (size_t)u.unit * u.ncmp;
    float* av = a.aval + u.rq.aval_off + (size_t)u.unit * 2 * u.ndem;
    for (int kl = tid; kl < nloc; kl += NT) {
      float z[ROWS];
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) z[rr] = zb[(size_t)kl * ROWS + rr];
      key_values<ROWS>(z, base_slot + kl, u.ndem, u.ncmp, lse_dem, lse_cmp, av, sc);
    }
  }

  // ---- 4. D_p, by the unit's last CTA -------------------------------------
  if (!last_of_unit(a, u, flag)) return;
  for (int x = 0; x < 2; ++x) {
    unsigned k = 0;
    if (u.ndem > 0) {
      const float* av = a.aval + u.rq.aval_off + ((size_t)u.unit * 2 + x) * u.ndem;
      k = coverage_demand<NT, 0>(av, u.ndem, a.pfix, reinterpret_cast<unsigned*>(zb), a.ppc * PAGE * ROWS, dps, a.err,
                                 tid, 0u, 0u);
    }
    if (tid == 0) write_demand(a, u.r, u.unit, x, k);
  }
}

template <bool BF16, int D, int ROWS>
cudaError_t launch_t(const DemandArgs& a, cudaStream_t s) {
  return launch_cluster(k_demand_ffma<BF16, D, ROWS>, a, Smem<D, ROWS>(a.ppc).total, s);
}

}  // namespace

cudaError_t launch_demand_ffma(const DemandArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE || a.C < 1 || a.C > 16 || a.ppc < 1 || a.ppc > 16) return cudaErrorInvalidValue;
  const bool bf = !a.kv_f32;
  if (a.D == 128 && a.G == 4) return bf ? launch_t<true, 128, 8>(a, s) : launch_t<false, 128, 8>(a, s);
  if (a.D == 128 && a.G == 2) return bf ? launch_t<true, 128, 4>(a, s) : launch_t<false, 128, 4>(a, s);
  if (a.D == 64 && a.G == 4) return bf ? launch_t<true, 64, 8>(a, s) : launch_t<false, 64, 8>(a, s);
  if (a.D == 64 && a.G == 2) return bf ? launch_t<true, 64, 4>(a, s) : launch_t<false, 64, 4>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
