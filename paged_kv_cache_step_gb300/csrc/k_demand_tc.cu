// Boundary demand kernel, tensor-core variant (tcgen05, sm_103a): GrowPage
// Sec. 3.2 Eqs. 2, 7 and App. E.1, plus the Eq. 9 importance cached for
// Compress & Hold, for bf16 caches and requests of at most 128 pages.
//
// Why the tensor core on an HBM-bound scan: each key meets 2G = 8 summary
// rows, 2 * 8 * d flops per 2 d bytes of K.  On CUDA cores that is 8 FMAs
// per loaded bf16 plus its unpacking, which at GB300's HBM rate keeps the
// FP32 pipes nearly saturated and leaves no issue slots for the softmax.
// The tensor core takes the products off the SM's pipes entirely.
//
// Exactness: K is bf16 already; each fp32 summary row q~ is split into three
// bf16 parts h1 + h2 + h3 (h1 = bf16(q~), h2 = bf16(q~ - h1), h3 =
// bf16(q~ - h1 - h2)), which represent q~ to fp32 precision.  One MMA with
// N = 3 * 2G (padded to a multiple of 16) gives K . h1, K . h2, K . h3 per key
// in fp32, summed afterwards.  The prep kernel writes these parts already in
// the 128-byte-swizzled K-major layout the MMA reads (one bulk copy).
//
// Per CTA (cluster rank c of the unit, logical pages [c*ppc, (c+1)*ppc)):
//   thread 0   : TMA producer and MMA issuer.  A tile is 128 keys x d of one
//                page (box 64 x 128, 128-byte swizzle), NSTAGE tiles in
//                flight through an mbarrier ring; each tile's accumulator
//                (128 lanes x N columns) stays in TMEM until the epilogue.
//   warps 4..7 : while the scan runs, read each finished tile from TMEM
//                (warp w owns lane quadrant w % 4) and fold its logits into
//                online (max, sum) statistics per row.
//   all        : push the statistics to every rank (DSMEM), merge, then
//                read TMEM again to write a^S, a^L and the importance.
//   last CTA   : of the unit (global ticket) computes D_p.
// Every wait is bounded; on expiry the CTA records ERR_TIMEOUT, drains its
// copies in flight and finishes with garbage rather than hanging.
#include <cuda.h>
#include <cuda_bf16.h>

#include "demand_common.cuh"

namespace gp {
namespace {

using namespace dem;

template <int D, int ROWS>
struct TcCfg {
  static constexpr int NB = (3 * ROWS + 15) / 16 * 16;  // MMA N: 3 parts x ROWS rows, padded
  static constexpr int HALVES = D / 64;                  // 128-byte swizzle spans per key row
  static constexpr int TILE_BYTES = 128 * D * 2;         // 128 keys of bf16
  static constexpr int HALF_BYTES = 128 * 128;           // one 64-element span of 128 keys
  static constexpr int BQ_BYTES = HALVES * NB * 128;
  static constexpr int KSTEPS = D / 16;
  static constexpr int NSTAGE = 3;
  static constexpr int MAX_TILES = 16;
  static constexpr uint32_t IDESC = (1u << 4)        // D: f32
                                    | (1u << 7)      // A: bf16
                                    | (1u << 10)     // B: bf16
                                    | ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

constexpr long long kWaitLimit = 1ll << 31;  // clock cycles (about one second)

// ---- PTX wrappers ----------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; gives up when the limit passes or *abort is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitLimit) return false;
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int NB>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v);

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Logits of the key in this thread's lane of tile t: sum of the three parts.
template <int NB, int ROWS>
__device__ __forceinline__ void tile_logits(uint32_t tmem, int quad, int t, float* z) {
  float v[NB];
  tmem_ld<NB>(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(t * NB), v);
#pragma unroll
  for (int r = 0; r < ROWS; ++r) z[r] = v[r] + (v[ROWS + r] + v[2 * ROWS + r]);
}

// Shared memory, after aligning the dynamic base to 1 KiB.
template <int D, int ROWS>
struct TcSmem {
  using T = TcCfg<D, ROWS>;
  static constexpr size_t STAGE = 0;
  static constexpr size_t BQ = STAGE + (size_t)T::NSTAGE * T::TILE_BYTES;
  static constexpr size_t BARS = BQ + T::BQ_BYTES;                    // full, empty, bq, ready[]
  static constexpr int NBARS = 2 * T::NSTAGE + 1 + T::MAX_TILES;
  static constexpr size_t XG = (BARS + 8 * NBARS + 15) & ~size_t(15);
  static constexpr size_t PART = XG + sizeof(StatXchg);              // [4 warps][2 sets][ROWS] (m, s)
  static constexpr size_t LSE = PART + sizeof(float) * 4 * 2 * ROWS * 2;
  static constexpr size_t MISC = LSE + sizeof(float) * 2 * ROWS;     // tmem holder, abort, flag, pages
  static constexpr size_t END = MISC + sizeof(int) * (4 + T::MAX_TILES);
  static constexpr size_t BYTES = END + 1024;                        // alignment slack
  static_assert(sizeof(DpSmem) + 1024 <= (size_t)T::NSTAGE * T::TILE_BYTES, "select scratch");
};

template <int D, int ROWS>
__global__ void __launch_bounds__(NT, 2) k_demand_tc(const __grid_constant__ DemandArgs a) {
  using T = TcCfg<D, ROWS>;
  using S = TcSmem<D, ROWS>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  StatXchg* xg = reinterpret_cast<StatXchg*>(smem + S::XG);
  float* part = reinterpret_cast<float*>(smem + S::PART);
  float* lse_dem = reinterpret_cast<float*>(smem + S::LSE);
  float* lse_cmp = lse_dem + ROWS;
  int* misc = reinterpret_cast<int*>(smem + S::MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = misc + 1;
  int* flag = misc + 2;
  int* phys = misc + 4;
  const uint32_t bar_full = sbase + (uint32_t)S::BARS;
  const uint32_t bar_empty = bar_full + 8 * T::NSTAGE;
  const uint32_t bar_bq = bar_empty + 8 * T::NSTAGE;
  const uint32_t bar_ready = bar_bq + 8;

  cluster_arrive_relaxed();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Unit u = make_unit(a);
  const int units = a.L * a.Hkv;
  const int ntiles = 2 * u.npg;
  const uint32_t ncols = (uint32_t)a.ppc * 2 * T::NB <= 32 ? 32u : (uint32_t)a.ppc * 2 * T::NB;

  if (tid == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_bq, 1);
    for (int t = 0; t < T::MAX_TILES; ++t) mbar_init(bar_ready + 8 * t, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort = 0;
    for (int j = 0; j < u.npg; ++j) phys[j] = checked_page(a, u, u.j0 + j);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // ---- scan ----------------------------------------------------------------
  if (warp == 0) {
    if (lane == 0) {
      const size_t layer_rows = (size_t)u.layer * a.num_pages_total;
      auto issue = [&](int t) {
        const int s = t % T::NSTAGE;
        const int y = (int)(((layer_rows + phys[t >> 1]) * a.Hkv + u.h) * PAGE + (t & 1) * 128);
        const uint32_t dst = sbase + (uint32_t)(S::STAGE + (size_t)s * T::TILE_BYTES);
        mbar_expect_tx(bar_full + 8 * s, T::TILE_BYTES);
#pragma unroll
        for (int hx = 0; hx < T::HALVES; ++hx) tma_load_2d(dst + hx * T::HALF_BYTES, &a.kmap, hx * 64, y, bar_full + 8 * s);
      };
      mbar_expect_tx(bar_bq, T::BQ_BYTES);
      bulk_load(sbase + (uint32_t)S::BQ, a.bq + ((size_t)u.r * units + u.unit) * T::BQ_BYTES, T::BQ_BYTES, bar_bq);
      int issued = 0;
      for (; issued < T::NSTAGE && issued < ntiles; ++issued) issue(issued);
      bool ok = mbar_wait(bar_bq, 0, abort);
      int t = 0;
      for (; ok && t < ntiles; ++t) {
        const int s = t % T::NSTAGE;
        if (!(ok = mbar_wait(bar_full + 8 * s, (t / T::NSTAGE) & 1, abort))) break;
        tc_fence_after();
        const uint32_t a0 = sbase + (uint32_t)(S::STAGE + (size_t)s * T::TILE_BYTES);
        const uint32_t b0 = sbase + (uint32_t)S::BQ;
#pragma unroll
        for (int k = 0; k < T::KSTEPS; ++k) {
          const uint32_t ad = a0 + (k >> 2) * T::HALF_BYTES + (k & 3) * 32;
          const uint32_t bd = b0 + (k >> 2) * (T::NB * 128) + (k & 3) * 32;
          mma_f16(tmem + (uint32_t)(t * T::NB), sw128_desc(ad), sw128_desc(bd), T::IDESC, k > 0 ? 1u : 0u);
        }
        mma_commit(bar_empty + 8 * s);
        mma_commit(bar_ready + 8 * t);
        // refill the stage of the previous tile once its MMAs are done
        if (t >= 1 && issued < ntiles) {
          const int tp = t - 1, sp = tp % T::NSTAGE;
          if (!(ok = mbar_wait(bar_empty + 8 * sp, (tp / T::NSTAGE) & 1, abort))) break;
          issue(issued++);
        }
      }
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
        // wait (bounded) for the copies still in flight before the memory is reused
        const int zero = 0;
        for (int tt = t; tt < issued; ++tt) mbar_wait(bar_full + 8 * (tt % T::NSTAGE), (tt / T::NSTAGE) & 1, &zero);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // online softmax statistics of the finished tiles
    const int quad = warp - 4;
    float m[2][ROWS], sm[2][ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      m[0][r] = m[1][r] = -INFINITY;
      sm[0][r] = sm[1][r] = 0.f;
    }
    for (int t = 0; t < ntiles; ++t) {
      // warp-uniform outcome: the TMEM load below is warp-collective
      if (!__all_sync(FULL, mbar_wait(bar_ready + 8 * t, 0, abort))) {
        if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
        break;
      }
      tc_fence_after();
      float z[ROWS];
      tile_logits<T::NB, ROWS>(tmem, quad, t, z);
      const int i = u.j0 * PAGE + t * 128 + 32 * quad + lane;
      if (i < u.ndem) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) online(m[0][r], sm[0][r], z[r]);
      } else if (i < u.ncmp) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) online(m[1][r], sm[1][r], z[r]);
      }
    }
#pragma unroll
    for (int set = 0; set < 2; ++set)
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        warp_combine(m[set][r], sm[set][r]);
        if (lane == 0) {
          part[((quad * 2 + set) * ROWS + r) * 2 + 0] = m[set][r];
          part[((quad * 2 + set) * ROWS + r) * 2 + 1] = sm[set][r];
        }
      }
  }
  __syncthreads();
  float cm = -INFINITY, cs = 0.f;
  if (tid < 2 * ROWS) {
    for (int q = 0; q < 4; ++q) combine(cm, cs, part[(q * 2 * ROWS + tid) * 2], part[(q * 2 * ROWS + tid) * 2 + 1]);
  }
  push_stats<ROWS>(xg, u.crank, a.C, cm, cs);
  merge_stats<ROWS>(xg, a.C, lse_dem, lse_cmp);
  __syncthreads();

  // ---- values: a^S, a^L and the importance of every key ----------------------
  {
    float* sc = a.scores + u.rq.score_off + (size_t)u.unit * u.ncmp;
    float* av = a.aval + u.rq.aval_off + (size_t)u.unit * 2 * u.ndem;
    const int quad = warp & 3;
    for (int t = warp >> 2; t < ntiles; t += 2) {
      if (!__all_sync(FULL, mbar_wait(bar_ready + 8 * t, 0, abort))) break;
      tc_fence_after();
      float z[ROWS];
      tile_logits<T::NB, ROWS>(tmem, quad, t, z);
      key_values<ROWS>(z, u.j0 * PAGE + t * 128 + 32 * quad + lane, u.ndem, u.ncmp, lse_dem, lse_cmp, av, sc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }

  // ---- D_p, by the unit's last CTA ---------------------------------------------
  if (!last_of_unit(a, u, flag)) return;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  unsigned k = 0;
  if (u.ndem > 0) {
    DpSmem* dps = reinterpret_cast<DpSmem*>(smem + S::STAGE);
    const size_t off = (sizeof(DpSmem) + 15) & ~size_t(15);
    unsigned* buf = reinterpret_cast<unsigned*>(smem + S::STAGE + off);
    const int cap = (int)(((size_t)T::NSTAGE * T::TILE_BYTES - off) / 4);
    const float* av = a.aval + u.rq.aval_off + (size_t)u.unit * 2 * u.ndem;
    k = coverage_demand(av, u.ndem, a.p, buf, cap, dps, a.err);
  }
  write_demand(a, u, k);
}

template <int D, int ROWS>
cudaError_t launch_t(const DemandArgs& a, cudaStream_t s) {
  using T = TcCfg<D, ROWS>;
  if (2 * a.ppc > T::MAX_TILES) return cudaErrorInvalidValue;
  // TMEM columns per CTA (a power of two >= 32); the CTAs an SM can hold must
  // never ask for more than its 512 columns, or a blocked allocation could
  // wait on a CTA that itself waits on its cluster.  Shared memory is padded
  // so that at most 512 / ncols CTAs fit on an SM.
  int ncols = 2 * a.ppc * T::NB;
  if (ncols < 32) ncols = 32;
  if (ncols & (ncols - 1)) return cudaErrorInvalidValue;
  const int fit = 512 / ncols;  // CTAs whose TMEM fits at once
  int dev = 0, sm_total = 0, reserved = 0, max_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_total, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  size_t smem = TcSmem<D, ROWS>::BYTES;
  // (fit + 1) CTAs of this size must not fit in one SM
  const size_t floor_bytes = (size_t)sm_total / (size_t)(fit + 1) - (size_t)reserved + 16;
  if (smem < floor_bytes) smem = floor_bytes;
  if (smem > (size_t)max_optin) return cudaErrorInvalidValue;
  return launch_cluster(k_demand_tc<D, ROWS>, a, smem, s);
}

}  // namespace

cudaError_t launch_demand_tc(const DemandArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE || a.kv_f32 || a.C < 1 || a.C > 16 || a.ppc < 1 || !a.bq) return cudaErrorInvalidValue;
  if (a.D == 128 && a.G == 4) return launch_t<128, 8>(a, s);
  if (a.D == 128 && a.G == 2) return launch_t<128, 4>(a, s);
  if (a.D == 64 && a.G == 4) return launch_t<64, 8>(a, s);
  if (a.D == 64 && a.G == 2) return launch_t<64, 4>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
