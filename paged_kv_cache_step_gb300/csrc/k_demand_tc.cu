// Boundary demand kernel, tensor-core variant (tcgen05, sm_103a): GrowPage
// Sec. 3.2 Eqs. 2, 7 and App. E.1, plus the Eq. 9 importance cached for
// Compress & Hold, for bf16 caches and requests of up to 256 pages.
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
// Persistent and warp-specialised: a cooperative grid of one CTA per SM.
// Each unit (request, layer, KV head) is split into parts of at most 10
// pages (tc_parts); CTA b takes parts b, b + grid, ... of the call's part
// list, which runs in unit order.  Roles:
//   warp 0      producer: per part, the unit's B operand (bulk copy) and the
//               part's K tiles (128 keys x d, box 64 x 128 with the 128-byte
//               swizzle) through an NSTAGE mbarrier ring, running ahead
//               across parts;
//   warp 1      MMA issuer: tcgen05.mma into a ring of TMEM accumulator
//               slots (a tile's accumulator is 128 lanes x N columns); a slot
//               is reused once the epilogue has read it, so the scan runs on
//               while the epilogue finishes the previous part;
//   warps 2..9  epilogue (warp w reads TMEM lane quadrant w % 4; two warps
//               per quadrant split the tiles): as tiles finish, it sums the
//               three partial products into each key's 2G logits, stores
//               them in a compact per-part TMEM region (2G columns per 128
//               keys, two parts deep), releases the accumulator slot and
//               folds online softmax statistics; then a reduce-scatter
//               butterfly over the warp, the part's statistics to global
//               memory and a count per unit.  It runs one part ahead: once
//               every part of the previous part's unit has counted in, the
//               merge, then that part's a^S, a^L and the importance of every
//               key to global memory, and a ticket per unit;
//   warps 10..15 selector: the CTA of part (2 unit + x) mod parts computes D_p
//               of summary x of the unit once all its parts' tickets are in
//               -- the exact select of demand_common.cuh, on the SM's
//               otherwise idle issue slots; a CTA's last part's selects are
//               left to the whole CTA once its scan is over.
// Progress: every CTA is resident (cooperative launch) and meets its units
// in increasing order, so the lowest unfinished unit always has all its
// parts' statistics on the way.  Every wait is bounded; on expiry the CTA
// records ERR_TIMEOUT, raises a shared abort flag that ends every role's
// loop, drains its copies in flight and finishes with garbage rather than
// hanging.
#include <cuda.h>
#include <cuda_bf16.h>

#include "demand_common.cuh"
#include "tc_ptx.cuh"

namespace gp {
namespace {

using namespace dem;
using namespace tc;

constexpr int NTHR = 512;       // 16 warps
constexpr int EPI_W0 = 2;       // epilogue warps 2..9: two per TMEM lane quadrant
constexpr int EPI_NW = 8;
constexpr int EPI_NTH = 32 * EPI_NW;
constexpr int SEL_W0 = 10;      // selector warps 10..15
constexpr int SEL_NTH = 32 * (16 - SEL_W0);
constexpr int BAR_EPI = 1;      // named barriers
constexpr int BAR_SEL = 2;
constexpr int QLEN = 32;        // select queue
constexpr long long kWaitLimit = 1ll << 31;  // clock cycles (about one second)
#ifndef GP_TC_STAGE_BYTES
#define GP_TC_STAGE_BYTES (96 * 1024)  // bytes of K tiles in flight per CTA (one CTA per SM)
#endif

template <int D, int ROWS>
struct TcCfg {
  static constexpr int NB = (3 * ROWS + 15) / 16 * 16;  // MMA N: 3 parts x ROWS rows, padded
  static constexpr int HALVES = D / 64;                  // 128-byte swizzle spans per key row
  static constexpr int TILE_BYTES = 128 * D * 2;         // 128 keys of bf16
  static constexpr int HALF_BYTES = 128 * 128;           // one 64-element span of 128 keys
  static constexpr int BQ_BYTES = HALVES * NB * 128;
  static constexpr int KSTEPS = D / 16;
  static constexpr int NSTAGE = GP_TC_STAGE_BYTES / TILE_BYTES;  // K in flight per SM
  static constexpr int TPU = 2 * TC_MAX_PPC;             // tiles per unit and CTA at most (10 pages)
  static constexpr int WSLOTS = (512 - 2 * TPU * ROWS) / NB;  // accumulator slots; the rest holds
  static constexpr int CBASE = WSLOTS * NB;              // two units of compact logits from here
  static_assert(CBASE + 2 * TPU * ROWS <= 512 && WSLOTS >= 4, "TMEM layout");
  static constexpr uint32_t IDESC = (1u << 4)        // D: f32
                                    | (1u << 7)      // A: bf16
                                    | (1u << 10)     // B: bf16
                                    | ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

// ---- PTX wrappers (the shared ones are in tc_ptx.cuh) -------------------------
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
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync %0, %1;" ::"n"(BAR_EPI), "n"(EPI_NTH) : "memory"); }
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <int R>
__device__ __forceinline__ void tmem_st_rows(uint32_t taddr, const float* z);
template <>
__device__ __forceinline__ void tmem_st_rows<8>(uint32_t taddr, const float* z) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(z[0])), "r"(__float_as_uint(z[1])), "r"(__float_as_uint(z[2])),
               "r"(__float_as_uint(z[3])), "r"(__float_as_uint(z[4])), "r"(__float_as_uint(z[5])),
               "r"(__float_as_uint(z[6])), "r"(__float_as_uint(z[7]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_st_rows<4>(uint32_t taddr, const float* z) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(__float_as_uint(z[0])), "r"(__float_as_uint(z[1])), "r"(__float_as_uint(z[2])),
               "r"(__float_as_uint(z[3]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
template <int R>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float* z);
template <>
__device__ __forceinline__ void tmem_ld_rows<8>(uint32_t taddr, float* z) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) z[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld_rows<4>(uint32_t taddr, float* z) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) z[i] = __uint_as_float(r[i]);
}

// Logits of the key in this thread's lane of the tile at TMEM column `col`.
template <int NB, int ROWS>
__device__ __forceinline__ void tile_logits(uint32_t tmem, int quad, int col, float* z) {
  float v[NB];
  tmem_ld<NB>(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)col, v);
#pragma unroll
  for (int r = 0; r < ROWS; ++r) z[r] = v[r] + (v[ROWS + r] + v[2 * ROWS + r]);
}

// Per-part facts every role derives from the part index p.
struct UnitInfo {
  int r, unit, layer, h, P, ndem, ncmp, npg, j0;
  int part, nparts;  // this part of the unit, and how many it has
  int w;             // unit index within the launch (work slot * units + unit)
  size_t g;          // unit index within the call: r * units + unit
  DevReq rq;
};
__device__ __forceinline__ UnitInfo unit_info(const DemandArgs& a, int p) {
  UnitInfo u;
  const int units = a.L * a.Hkv;
  int lo = 0, hi = a.n_work;  // the work slot i with part_base[i] <= p < part_base[i + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.part_base[mid] <= p) lo = mid; else hi = mid;
  }
  u.r = a.work[lo];
  u.rq = a.reqs[u.r];
  u.P = u.rq.num_pages;
  u.nparts = tc_parts(u.P);
  const int local = p - a.part_base[lo];
  u.unit = local / u.nparts;
  u.w = lo * units + u.unit;
  u.part = (u.w + local % u.nparts) % u.nparts;
  u.layer = u.unit / a.Hkv;
  u.h = u.unit % a.Hkv;
  u.g = (size_t)u.r * units + u.unit;
  u.ndem = (u.P - 1) * PAGE;
  u.ncmp = u.P * PAGE - a.R;
  u.j0 = (u.part * u.P) / u.nparts;
  u.npg = ((u.part + 1) * u.P) / u.nparts - u.j0;
  return u;
}

struct XStat {
  float m, s;
};

// Shared memory, after aligning the dynamic base to 1 KiB.  The select
// buffer takes whatever is left of the dynamic allocation.
template <int D, int ROWS>
struct TcSmem {
  using T = TcCfg<D, ROWS>;
  static constexpr size_t STAGE = 0;
  static constexpr size_t BQ = STAGE + (size_t)T::NSTAGE * T::TILE_BYTES;  // 2 buffers
  static constexpr size_t XG = BQ + 2 * (size_t)T::BQ_BYTES;               // XStat [32 parts][16]
  static_assert(TC_MAX_PARTS <= 32, "merge buffer");
  static constexpr size_t BARS = XG + sizeof(XStat) * 32 * 16;
  // full[NSTAGE], empty[NSTAGE], bqfull[2], bqempty[2], mmadone, sel, ready[W], wfree[W]
  static constexpr int NBARS = 2 * T::NSTAGE + 6 + 2 * T::WSLOTS;
  static constexpr size_t PART = BARS + 8 * (size_t)NBARS;                 // [EPI_NW][16] XStat
  static constexpr size_t LSE = PART + sizeof(XStat) * EPI_NW * 16;        // lse_dem[8], lse_cmp[8]
  static constexpr size_t MISC = LSE + sizeof(float) * 16;                 // ints, see kernel
  static constexpr size_t DPS = (MISC + sizeof(int) * (16 + QLEN + 16) + 15) & ~size_t(15);
  static constexpr size_t SEL = (DPS + sizeof(DpSmem) + 15) & ~size_t(15);
  static constexpr size_t MIN_SEL_BYTES = 8 * 1024;
  static constexpr size_t MIN_BYTES = SEL + MIN_SEL_BYTES + 1024;          // + alignment slack
};

template <int D, int ROWS>
__global__ void __launch_bounds__(NTHR, 1) k_demand_tc(const __grid_constant__ DemandArgs a, int smem_bytes) {
  using T = TcCfg<D, ROWS>;
  using S = TcSmem<D, ROWS>;
  constexpr int NSTAT = 2 * ROWS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  XStat* xg = reinterpret_cast<XStat*>(smem + S::XG);         // [part][stat] of the unit being merged
  XStat* part = reinterpret_cast<XStat*>(smem + S::PART);
  float* lse_dem = reinterpret_cast<float*>(smem + S::LSE);
  float* lse_cmp = lse_dem + 8;
  int* misc = reinterpret_cast<int*>(smem + S::MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort = misc + 1;
  volatile int* q_head = misc + 2;
  volatile int* q_tail = misc + 3;
  volatile int* q_done = misc + 4;
  volatile int* sel_item = misc + 5;
  volatile int* flag = misc + 6;   // exchange outcome of the current part (epilogue)
  volatile int* epi_fail = misc + 8;  // an epilogue warp's tile wait gave up (sticky)
  int* phys = misc + 16;                                      // [16]
  volatile int* queue = misc + 32;                            // [QLEN]
  DpSmem* dps = reinterpret_cast<DpSmem*>(smem + S::DPS);
  unsigned* selbuf = reinterpret_cast<unsigned*>(smem + S::SEL);
  const int sel_cap =
      (int)(((size_t)smem_bytes - (size_t)(smem - smem_raw) - S::SEL) / sizeof(unsigned));

  const uint32_t bar_full = sbase + (uint32_t)S::BARS;
  const uint32_t bar_empty = bar_full + 8 * T::NSTAGE;
  const uint32_t bar_bqfull = bar_empty + 8 * T::NSTAGE;
  const uint32_t bar_bqempty = bar_bqfull + 16;
  const uint32_t bar_mmadone = bar_bqempty + 16;
  const uint32_t bar_sel = bar_mmadone + 8;
  const uint32_t bar_ready = bar_sel + 8;
  const uint32_t bar_wfree = bar_ready + 8 * T::WSLOTS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;  // CTA cta takes parts cta, cta + ncta, ...
  const int total_parts = a.n_parts;

  if (tid == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_bqfull + 8 * b, 1);
      mbar_init(bar_bqempty + 8 * b, 1);
    }
    mbar_init(bar_mmadone, 1);
    mbar_init(bar_sel, 1);
    for (int t = 0; t < T::WSLOTS; ++t) {
      mbar_init(bar_ready + 8 * t, 1);
      mbar_init(bar_wfree + 8 * t, 4);  // the four quadrant warps that read the slot
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort = 0;
    *q_head = 0;
    *q_tail = 0;
    *q_done = 0;
    *epi_fail = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // The next queued select (2 p + x: summary x of part p's unit) this CTA
  // computes, once every part of the unit has written its a-values; -1 when
  // the queue is empty and the
  // epilogue has finished (or stop_at_done and the epilogue has finished),
  // or on abort.  Called by one thread.
  auto take_item = [&](bool stop_at_done) -> int {
    int item = -1;
    const long long t0 = clock64();
    while (true) {
      const int h = *q_head, tl = *q_tail;
      if (*q_done && stop_at_done) break;
      if (h != tl) {
        item = queue[tl % QLEN];
        break;
      }
      if (*q_done) {
        __threadfence_block();
        if (*q_head == tl) break;
        continue;
      }
      if (*abort) break;
      if (clock64() - t0 > kWaitLimit) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
        break;
      }
      __nanosleep(200);
    }
    if (item >= 0) {
      const UnitInfo u = unit_info(a, item >> 1);
      const unsigned* tk = a.tickets + u.g;
      const long long t1 = clock64();
      while (ld_acquire(tk) < (unsigned)u.nparts) {
        if (*abort || clock64() - t1 > kWaitLimit) {
          atomicOr(a.err, ERR_TIMEOUT);
          *abort = 1;
          item = -1;
          break;
        }
        __nanosleep(100);
      }
    }
    return item;
  };

  if (warp == 0) {
    // ---- producer --------------------------------------------------------
    if (lane == 0) {
      int gt = 0, last_gt[T::NSTAGE], last_bq[2] = {-1, -1};
      for (int s = 0; s < T::NSTAGE; ++s) last_gt[s] = -1;
      bool ok = true;
      for (int kk = 0; ok; ++kk) {
        const int pi = cta + kk * ncta;
        if (pi >= total_parts) break;
        const UnitInfo u = unit_info(a, pi);
        const int b2 = kk & 1;
        if (kk >= 2 && !(ok = mbar_wait(bar_bqempty + 8 * b2, ((kk >> 1) - 1) & 1, abort))) break;
        mbar_expect_tx(bar_bqfull + 8 * b2, T::BQ_BYTES);
        bulk_load(sbase + (uint32_t)(S::BQ + (size_t)b2 * T::BQ_BYTES),
                  a.bq + u.g * T::BQ_BYTES, T::BQ_BYTES, bar_bqfull + 8 * b2);
        last_bq[b2] = kk;
        for (int j = 0; j < u.npg; ++j) {
          int pg = a.bt[u.rq.bt_off + u.j0 + j];
          if (pg < 0 || pg >= a.num_pages_total) {
            atomicOr(a.err, ERR_BAD_PAGE);
            pg = 0;
          }
          phys[j] = pg;
        }
        const size_t layer_rows = (size_t)u.layer * a.num_pages_total;
        for (int t = 0; t < 2 * u.npg; ++t, ++gt) {
          const int s = gt % T::NSTAGE;
          if (gt >= T::NSTAGE && !(ok = mbar_wait(bar_empty + 8 * s, ((gt / T::NSTAGE) - 1) & 1, abort))) break;
          const int y = (int)(((layer_rows + phys[t >> 1]) * a.Hkv + u.h) * PAGE + (t & 1) * 128);
          const uint32_t dst = sbase + (uint32_t)(S::STAGE + (size_t)s * T::TILE_BYTES);
          mbar_expect_tx(bar_full + 8 * s, T::TILE_BYTES);
#pragma unroll
          for (int hx = 0; hx < T::HALVES; ++hx)
            tma_load_2d(dst + hx * T::HALF_BYTES, &a.kmap, hx * 64, y, bar_full + 8 * s);
          last_gt[s] = gt;
        }
      }
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
      }
      // every copy issued has landed before the CTA moves on (bounded)
      const int zero = 0;
      for (int s = 0; s < T::NSTAGE; ++s)
        if (last_gt[s] >= 0) mbar_wait(bar_full + 8 * s, (last_gt[s] / T::NSTAGE) & 1, &zero);
      for (int b = 0; b < 2; ++b)
        if (last_bq[b] >= 0) mbar_wait(bar_bqfull + 8 * b, (last_bq[b] >> 1) & 1, &zero);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer --------------------------------------------------------
    if (lane == 0) {
      int gt = 0;
      bool ok = true;
      for (int kk = 0; ok; ++kk) {
        const int pi = cta + kk * ncta;
        if (pi >= total_parts) break;
        const UnitInfo u = unit_info(a, pi);
        const int b2 = kk & 1;
        if (!(ok = mbar_wait(bar_bqfull + 8 * b2, (kk >> 1) & 1, abort))) break;
        const uint32_t b0 = sbase + (uint32_t)(S::BQ + (size_t)b2 * T::BQ_BYTES);
        for (int t = 0; t < 2 * u.npg; ++t, ++gt) {
          const int s = gt % T::NSTAGE, ws = gt % T::WSLOTS;
          if (gt >= T::WSLOTS && !(ok = mbar_wait(bar_wfree + 8 * ws, ((gt / T::WSLOTS) - 1) & 1, abort))) break;
          if (!(ok = mbar_wait(bar_full + 8 * s, (gt / T::NSTAGE) & 1, abort))) break;
          tc_fence_after();
          const uint32_t a0 = sbase + (uint32_t)(S::STAGE + (size_t)s * T::TILE_BYTES);
          const uint32_t col = (uint32_t)(ws * T::NB);
#pragma unroll
          for (int k = 0; k < T::KSTEPS; ++k) {
            const uint32_t ad = a0 + (k >> 2) * T::HALF_BYTES + (k & 3) * 32;
            const uint32_t bd = b0 + (k >> 2) * (T::NB * 128) + (k & 3) * 32;
            mma_f16(tmem + col, sw128_desc(ad), sw128_desc(bd), T::IDESC, k > 0 ? 1u : 0u);
          }
          mma_commit(bar_empty + 8 * s);
          mma_commit(bar_ready + 8 * ws);
        }
        if (ok) mma_commit(bar_bqempty + 8 * b2);
      }
      if (!ok) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
      }
      // all MMAs issued have completed before TMEM is released (bounded)
      mma_commit(bar_mmadone);
      const int zero = 0;
      mbar_wait(bar_mmadone, 0, &zero);
    }
    __syncwarp();
  } else if (warp >= EPI_W0 && warp < SEL_W0) {
    // ---- epilogue ------------------------------------------------------------
    // Skewed by one part: part k+1's tiles are folded and its statistics
    // published before part k's merge waits on the other CTAs, so the
    // accumulator slots keep draining while the exchange completes.  Every
    // early exit is decided from shared flags written before a barrier, so
    // all epilogue threads leave together.
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const int half = (warp - EPI_W0) >> 2;      // tiles t with t % 2 == half
    const int ew = warp - EPI_W0;               // 0..7
    const int et = tid - 32 * EPI_W0;           // 0..255
    const uint32_t lanes = (uint32_t)(32 * quad) << 16;
    int gt0 = 0;  // global index of the part's first tile, in the MMA issuer's order

    // Fold part kk's tiles (compact logits into TMEM region kk & 1, online
    // statistics), then publish its statistics and count it in.
    auto fold_publish = [&](int kk, const UnitInfo& u) -> bool {
      const int ntiles = 2 * u.npg;
      const uint32_t cbase = tmem + lanes + (uint32_t)(T::CBASE + (kk & 1) * T::TPU * ROWS);
      float m[NSTAT], sm[NSTAT];
#pragma unroll
      for (int e = 0; e < NSTAT; ++e) {
        m[e] = NEG;
        sm[e] = 0.f;
      }
      bool ok = true;
      for (int t = half; t < ntiles; t += 2) {
        // warp-uniform outcome: the TMEM load below is warp-collective
        const int gt = gt0 + t, ws = gt % T::WSLOTS;
        if (!(ok = __all_sync(FULL, mbar_wait(bar_ready + 8 * ws, (gt / T::WSLOTS) & 1, abort)))) break;
        tc_fence_after();
        float z[ROWS];
        tile_logits<T::NB, ROWS>(tmem, quad, ws * T::NB, z);
        // keep the logits, hand the accumulator slot back to the MMA issuer
        tmem_st_rows<ROWS>(cbase + (uint32_t)(t * ROWS), z);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_wfree + 8 * ws);
        const int i = u.j0 * PAGE + t * 128 + 32 * quad + lane;
        if (i < u.ndem) {
#pragma unroll
          for (int r = 0; r < ROWS; ++r) online(m[r], sm[r], z[r]);
        } else if (i < u.ncmp) {
#pragma unroll
          for (int r = 0; r < ROWS; ++r) online(m[ROWS + r], sm[ROWS + r], z[r]);
        }
      }
      gt0 += ntiles;
      if (!ok && lane == 0) {
        atomicOr(a.err, ERR_TIMEOUT);
        *abort = 1;
        *epi_fail = 1;
      }
      {
        float om, os;
        int idx;
        warp_reduce_stats<NSTAT>(m, sm, lane, om, os, idx);
        if ((lane & (32 / NSTAT - 1)) == 0) part[ew * 16 + idx] = XStat{om, os};
      }
      epi_sync();
      if (*epi_fail) return false;  // written only before the barrier: every epilogue thread agrees
      // the part's statistics to global memory (8 bytes each), then its count
      if (et < NSTAT) {
        float cm = NEG, cs = 0.f;
#pragma unroll
        for (int q = 0; q < EPI_NW; ++q) combine(cm, cs, part[q * 16 + et].m, part[q * 16 + et].s);
        __stcg(a.xstat + u.g * (size_t)(TC_MAX_PARTS * 16) + u.part * 16 + et, make_float2(cm, cs));
      }
      epi_sync();
      if (et == 0) {
        __threadfence();
        atomicAdd(a.xcount + u.g, 1u);
      }
      return true;
    };

    // Once every part of its unit has counted in: merge the statistics, write
    // part kk's a^S, a^L and importance from TMEM region kk & 1, take a
    // ticket and queue the selects this CTA owns.
    auto finish = [&](int kk, int pi, const UnitInfo& u) -> bool {
      if (et == 0) {
        bool in = true;
        const long long t0 = clock64();
        while (ld_acquire(a.xcount + u.g) < (unsigned)u.nparts) {
          if (*abort || clock64() - t0 > kWaitLimit) {
            in = false;
            break;
          }
          __nanosleep(64);
        }
        if (!in) {
          atomicOr(a.err, ERR_TIMEOUT);
          *abort = 1;
        }
        *flag = in ? 1 : 0;
      }
      epi_sync();
      if (*flag == 0) return false;
      // the unit's statistics through L2 (other CTAs wrote them), then the
      // merge into base-2 log-sum-exps over C_t and over C_cmp
      const float2* xs_g = a.xstat + u.g * (size_t)(TC_MAX_PARTS * 16);
      for (int i = et; i < u.nparts * NSTAT; i += EPI_NTH) {
        const float2 v = __ldcg(xs_g + (i / NSTAT) * 16 + i % NSTAT);
        xg[(i / NSTAT) * 16 + i % NSTAT] = XStat{v.x, v.y};
      }
      epi_sync();
      if (et < ROWS) {
        float md, sd, mt, stl;
        merge_ranks(&xg[et].m, &xg[et].s, u.nparts, 32, &md, &sd);
        merge_ranks(&xg[ROWS + et].m, &xg[ROWS + et].s, u.nparts, 32, &mt, &stl);
        lse_pair(md, sd, mt, stl, lse_dem + et, lse_cmp + et);
      }
      epi_sync();
      // a^S, a^L and the importance of every key of this warp's tiles
      {
        const uint32_t cbase = tmem + lanes + (uint32_t)(T::CBASE + (kk & 1) * T::TPU * ROWS);
        float* sc = a.scores + u.rq.score_off + (size_t)u.unit * u.ncmp;
        float* av = a.aval + u.rq.aval_off + (size_t)u.unit * 2 * u.ndem;
        for (int t = half; t < 2 * u.npg; t += 2) {
          float z[ROWS];
          tmem_ld_rows<ROWS>(cbase + (uint32_t)(t * ROWS), z);
          key_values<ROWS>(z, u.j0 * PAGE + t * 128 + 32 * quad + lane, u.ndem, u.ncmp, lse_dem, lse_cmp, av, sc);
        }
      }
      tc_fence_before();
      epi_sync();
      if (et == 0) {
        // the CTA's a-values (ordered by the barrier above) before its ticket
        __threadfence();
        atomicAdd(a.tickets + u.g, 1u);
        // D_p of summary x is computed by the CTA of part (2 unit + x) mod
        // parts, which spreads the selects over the CTAs: queue it for this
        // CTA's selector warps
        for (int x = 0; x < 2; ++x) {
          if ((2 * u.w + x) % u.nparts != u.part) continue;
          const long long t0 = clock64();
          while (*q_head - *q_tail >= QLEN) {
            if (*abort || clock64() - t0 > kWaitLimit) {
              atomicOr(a.err, ERR_TIMEOUT);
              *abort = 1;
              break;
            }
          }
          if (*abort) break;
          // this CTA's last part: no scan is left to hide its select behind,
          // so the selector warps stop here and the whole CTA drains it
          if (pi + ncta >= total_parts) {
            *q_done = 1;
            __threadfence_block();
          }
          queue[*q_head % QLEN] = 2 * pi + x;
          __threadfence_block();
          *q_head = *q_head + 1;
        }
      }
      return true;
    };

    if (cta < total_parts) {
      int pi = cta;
      UnitInfo cur = unit_info(a, pi);
      bool live = fold_publish(0, cur);
      for (int kk = 0; live; ++kk) {
        const int pn = pi + ncta;
        UnitInfo nxt;
        const bool more = pn < total_parts;
        if (more) {
          nxt = unit_info(a, pn);
          if (!fold_publish(kk + 1, nxt)) break;
        }
        if (!finish(kk, pi, cur)) break;
        if (!more) break;
        cur = nxt;
        pi = pn;
      }
    }
    if (et == 0) {
      __threadfence_block();
      *q_done = 1;
    }
  } else if (warp >= SEL_W0) {
    // ---- selector ------------------------------------------------------------
    // Runs queued selects while the scan goes on; the ones still queued when
    // the epilogue finishes are left to the whole CTA (drain below).
    const int st = tid - 32 * SEL_W0;
    uint32_t sel_par = 0u;  // phase of the staging barrier
    while (true) {
      if (st == 0) *sel_item = take_item(true);
      sel_sync<SEL_NTH, BAR_SEL>();
      const int item = *sel_item;
      if (item < 0) break;
      const int x = item & 1;
      const UnitInfo u = unit_info(a, item >> 1);
      unsigned k = 0;
      if (u.ndem > 0) {
        const float* av = a.aval + u.rq.aval_off + ((size_t)u.unit * 2 + x) * u.ndem;
        k = coverage_demand<SEL_NTH, BAR_SEL>(av, u.ndem, a.pfix, selbuf, sel_cap, dps, a.err, st, bar_sel, sel_par);
        if (sel_resident(u.ndem, sel_cap)) sel_par ^= 1u;
      }
      if (st == 0) write_demand(a, u.r, u.unit, x, k);
      sel_sync<SEL_NTH, BAR_SEL>();
      if (st == 0) *q_tail = *q_tail + 1;
    }
    if (st == 0) misc[7] = (int)sel_par;
  }
  (void)phys;

  // ---- drain: selects still queued when the scan ended, with the whole CTA --
  tc_fence_before();
  __syncthreads();
  {
    uint32_t par = (uint32_t)misc[7];
    while (true) {
      if (tid == 0) *sel_item = take_item(false);
      __syncthreads();
      const int item = *sel_item;
      if (item < 0) break;
      const int x = item & 1;
      const UnitInfo u = unit_info(a, item >> 1);
      unsigned k = 0;
      if (u.ndem > 0) {
        const float* av = a.aval + u.rq.aval_off + ((size_t)u.unit * 2 + x) * u.ndem;
        k = coverage_demand<NTHR, 0>(av, u.ndem, a.pfix, selbuf, sel_cap, dps, a.err, tid, bar_sel, par);
        if (sel_resident(u.ndem, sel_cap)) par ^= 1u;
      }
      if (tid == 0) write_demand(a, u.r, u.unit, x, k);
      __syncthreads();
      if (tid == 0) *q_tail = *q_tail + 1;
    }
  }

  // ---- teardown ----------------------------------------------------------------
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// The kernel's launch attribute (set once) and its dynamic shared memory:
// the whole opt-in amount, so that one CTA owns an SM, its TMEM (512
// columns) and the select buffer.  0 if the device cannot hold the layout.
template <int D, int ROWS>
size_t prepare_t() {
  using S = TcSmem<D, ROWS>;
  static size_t smem = 0;
  if (smem) return smem;
  int dev = 0, max_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      (size_t)max_optin < S::MIN_BYTES) {
    cudaGetLastError();
    return 0;
  }
  if (cudaFuncSetAttribute(k_demand_tc<D, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  smem = (size_t)max_optin;
  return smem;
}

// CTAs the device holds at once (one per SM at this shared-memory size).
template <int D, int ROWS>
int resident_t() {
  static int n = -1;
  if (n >= 0) return n;
  const size_t smem = prepare_t<D, ROWS>();
  int dev = 0, sms = 0, per_sm = 0;
  if (!smem || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_demand_tc<D, ROWS>, NTHR, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  n = sms * per_sm;
  return n;
}

template <int D, int ROWS>
cudaError_t launch_t(const DemandArgs& a, cudaStream_t s) {
  if (a.n_parts < 1 || !a.part_base || !a.xstat || !a.xcount) return cudaErrorInvalidValue;
  const size_t smem = prepare_t<D, ROWS>();
  int grid = resident_t<D, ROWS>();
  if (!smem || grid < 1) return cudaErrorInvalidValue;
  if (grid > a.n_parts) grid = a.n_parts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(NTHR, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // the parts of a unit wait on one another: every CTA must be resident
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_demand_tc<D, ROWS>, a, (int)smem);
}

}  // namespace

int demand_tc_resident(int D, int G) {
  if (D == 128 && G == 4) return resident_t<128, 8>();
  if (D == 128 && G == 2) return resident_t<128, 4>();
  if (D == 64 && G == 4) return resident_t<64, 8>();
  if (D == 64 && G == 2) return resident_t<64, 4>();
  return 0;
}

cudaError_t launch_demand_tc(const DemandArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE || a.kv_f32 || !a.bq) return cudaErrorInvalidValue;
  if (a.D == 128 && a.G == 4) return launch_t<128, 8>(a, s);
  if (a.D == 128 && a.G == 2) return launch_t<128, 4>(a, s);
  if (a.D == 64 && a.G == 4) return launch_t<64, 8>(a, s);
  if (a.D == 64 && a.G == 2) return launch_t<64, 4>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gp
