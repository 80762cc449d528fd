// Compress & Hold kernel for sm_103a: GrowPage Sec. 3.3 Eqs. 9-10 and
// App. E.2, one CTA per (request, layer, KV head).
//
//  selection  -- importance s = max(a^S, a^L) comes from the cache the demand
//                kernel wrote (log2 domain; the order is the same).  The
//                protected recent window [P b - R, P b) is always kept.
//                Block-local: warp w takes logical blocks w, w+8, ... and
//                keeps the top k_loc' of each (bit-serial radix select on
//                order-preserving 32-bit keys: one warp reduction per bit).
//                Global: a CTA-wide bit-serial radix select keeps the top
//                K_t - |S_loc| of the remaining candidates.  Equal scores are
//                resolved towards the lower slot.
//  compaction -- order-preserving stream compaction: the k-th kept slot moves
//                to logical slot k of the target block table (ballot/popc +
//                word prefix scan).  The chunks (64 slots, 32 for 512-byte
//                rows) that move any row are listed in order; one thread
//                streams their K and V rows into a ring of CSTAGES shared-
//                memory stages with bulk async copies, and the CTA writes
//                each chunk's moving rows from there.  Source and target
//                tables differ only in pages replaced by copy-on-write
//                (fresh pages), so in-place moves only ever go to a lower
//                logical slot: a chunk's writes land below the next chunk's
//                first slot, never on a later chunk's rows, and each chunk is
//                written only after its own copy has landed.  That makes the
//                in-place pass race-free with several chunks in flight.
//                Rows whose physical location does not change are neither
//                read nor written.
//  hole-fill  -- an order-destroying variant (not the paper's compaction):
//                kept rows of the first P-1 pages stay where they are and
//                the last page's kept rows fill the holes, the k-th of them
//                the k-th hole; at most a page of rows moves per unit.
#include <cstdint>

#include "gp_kernels.h"

namespace gp {
namespace {

constexpr int NT = 256;
constexpr int NWARP = 8;
constexpr int PAGE = 256;
constexpr int MAX_WORDS = 256 * PAGE / 32;  // 256 pages
#ifndef GP_CMP_STAGES
#define GP_CMP_STAGES 2  // chunks of K and V in flight per CTA (two CTAs fit an SM)
#endif
constexpr int CSTAGES = GP_CMP_STAGES;
constexpr int STAGE_BYTES = 32 * 1024;      // K and V rows of one chunk
// Drains (waits for copies already issued, before the CTA's shared memory
// goes away) always use the full limit, whatever a.wait_limit says.
constexpr long long kDrainLimit = kDefaultWaitLimit;

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
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase of an mbarrier; false when `limit` clock cycles
// passed first.  try_wait may suspend the thread for a while by itself, so a
// limit far below the default polls with the non-blocking test_wait instead,
// checking the clock first: then the limit alone decides when the wait gives
// up, and a limit of 0 gives up at once.
constexpr long long kPollBelow = 1ll << 20;
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, long long limit) {
  if (limit < kPollBelow) {
    const long long t0 = clock64();
    while (clock64() - t0 < limit)
      if (bar_test(bar, parity)) return true;
    return false;
  }
  if (bar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!bar_try(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

__device__ __forceinline__ unsigned okey(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void warp_inc(unsigned* hist, unsigned bin, bool valid) {
  const int key = valid ? (int)bin : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  if (valid && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
}

// In a 256-bin count histogram, find the bin holding the need-th largest key
// (walking from bin 255 down).  Returns the bin and the count strictly above
// it.  Called by one full warp.
__device__ __forceinline__ void find_bin(const unsigned* hist, unsigned need, unsigned& bin_out,
                                         unsigned& above_out, bool& ok) {
  const int lane = threadIdx.x & 31;
  const int top = 255 - 8 * lane;
  unsigned lc = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) lc += hist[top - k];
  unsigned ic = lc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned oc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) ic += oc;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, ic >= need);
  const int src = hit ? __ffs(hit) - 1 : 31;
  unsigned chosen = 0, above = 0;
  bool found = false;
  if (lane == src) {
    unsigned cum = ic - lc;
    chosen = (unsigned)(top - 7);
    for (int k = 0; k < 8; ++k) {
      const unsigned b = (unsigned)(top - k);
      if (cum + hist[b] >= need) { chosen = b; found = true; break; }
      cum += hist[b];
    }
    above = cum;
  }
  bin_out = __shfl_sync(0xffffffffu, chosen, src);
  above_out = __shfl_sync(0xffffffffu, above, src);
  ok = __shfl_sync(0xffffffffu, found, src) && hit != 0;
}

// Exclusive prefix of popc(words[0..nw)) into pre[]; all threads call it.
__device__ void word_prefix(const unsigned* words, unsigned* pre, int nw, unsigned* red) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nw + NT - 1) / NT;
  const int w0 = tid * per;
  unsigned local = 0;
  for (int k = 0; k < per; ++k)
    if (w0 + k < nw) local += __popc(words[w0 + k]);
  unsigned inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  unsigned wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += red[w];
  unsigned run = wbase + inc - local;
  for (int k = 0; k < per; ++k) {
    if (w0 + k < nw) {
      pre[w0 + k] = run;
      run += __popc(words[w0 + k]);
    }
  }
  __syncthreads();
}

template <int RB>
__global__ void __launch_bounds__(NT, 1) k_compress(CompressArgs a) {
  extern __shared__ __align__(128) unsigned char stage_mem[];  // CSTAGES x STAGE_BYTES
  __shared__ __align__(8) unsigned long long full_bar[CSTAGES];
  __shared__ int s_nlist;
  __shared__ int s_stage0;  // uses of stage 0's barrier before the compaction (0 or 1)
  __shared__ unsigned keep[MAX_WORDS];
  __shared__ unsigned loc[MAX_WORDS];     // block-local picks (Eq. 10, S_loc)
  __shared__ unsigned tmp[MAX_WORDS];     // tie bits
  __shared__ unsigned pre[MAX_WORDS];     // exclusive word prefixes
  __shared__ unsigned whist[NWARP][256];
  __shared__ unsigned red[NWARP];
  __shared__ int s_old[PAGE], s_new[PAGE];
  __shared__ int s_hole[PAGE];            // hole-fill mode: the holes in order
  __shared__ int s_fast;                  // the selection's fast path applied
  __shared__ int s_nholes;
  __shared__ unsigned s_sel[4];           // prefix, mask, above, flags
  __shared__ int s_abort;                 // 1: a wait gave up; 2: the keep count is wrong

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units = a.L * a.Hkv;
  const int wi = blockIdx.x / units;
  const int unit = blockIdx.x % units;
  const int layer = unit / a.Hkv, h = unit % a.Hkv;
  const int r = a.work[wi];
  const DevReq rq = a.reqs[r];
  const int P = rq.num_pages;
  const int N = P * PAGE;
  const int words = N / 32;
  const int ncmp = N - a.R;
  const int kt = (P - a.drop) * PAGE - a.R;          // K_t (Eq. 10); Shrink drops two pages' worth
  const unsigned target_kept = (unsigned)((P - a.drop) * PAGE);

  if (tid == 0) {
    s_abort = 0;
    s_stage0 = 0;
    for (int st = 0; st < CSTAGES; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full_bar[st])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // the stage barriers exist before any thread waits on them
  for (int j = tid; j < P; j += NT) {
    s_old[j] = a.old_bt[rq.bt_off + j];
    s_new[j] = a.new_bt[rq.bt_off + j];
  }

  if (a.keep_in) {
    const unsigned* src = a.keep_in + rq.mask_off + (size_t)unit * words;
    for (int w = tid; w < words; w += NT) keep[w] = src[w];
    __syncthreads();
  } else {
    // The unit's importance values, staged in the (still idle) chunk stages
    // with one bulk copy when they fit: every pass below then reads shared
    // memory instead of making dependent trips to L2.
    const float* sc = a.scores + rq.score_off + (size_t)unit * ncmp;
    if ((size_t)ncmp * 4 <= (size_t)CSTAGES * STAGE_BYTES && (ncmp & 3) == 0 &&
        (reinterpret_cast<uintptr_t>(sc) & 15) == 0) {
      const uint32_t bar = smem_addr(&full_bar[0]);
      if (tid == 0) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)(ncmp * 4))
                     : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_addr(stage_mem)),
                     "l"(sc), "r"((uint32_t)(ncmp * 4)), "r"(bar)
                     : "memory");
      }
      if (!bar_wait(bar, 0u, a.wait_limit)) atomicOr(&s_abort, 1);
      sc = reinterpret_cast<const float*>(stage_mem);
      // phase 0 of stage 0's barrier is used: the compaction starts at phase 1
      if (tid == 0) s_stage0 = 1;
    }
    for (int w = tid; w < words; w += NT) loc[w] = 0u;
    __syncthreads();
    // ---- Eq. 10, global part: TopK_{K_t - |S_loc|}(C \ S_loc), then the keep words
    auto global_keep = [&]() {
      unsigned nloc = 0;
      for (int w = tid; w < words; w += NT) nloc += __popc(loc[w]);
  #pragma unroll
      for (int o = 16; o > 0; o >>= 1) nloc += __shfl_xor_sync(0xffffffffu, nloc, o);
      if (lane == 0) red[warp] = nloc;
      if (tid == 0) { s_sel[0] = 0; s_sel[1] = 0; s_sel[2] = 0; s_sel[3] = 0; }
      __syncthreads();
      unsigned tot_loc = 0;
      for (int w = 0; w < NWARP; ++w) tot_loc += red[w];
      const int need_g = kt - (int)tot_loc;
      const int iters = (ncmp + NT - 1) / NT;
      // radix select (8-bit digits) of the need_g-th largest key among the
      // candidates outside S_loc
      unsigned* hist = whist[0];
      if (need_g > 0) {
        for (int ro = 0; ro < 4; ++ro) {
          const int shift = 24 - 8 * ro;
          hist[tid] = 0u;
          __syncthreads();
          const unsigned prefix = s_sel[0], mask = s_sel[1];
          for (int it0 = 0; it0 < iters; it0 += 8) {
            // eight independent loads in flight, then their histogram updates
            unsigned kb[8];
            bool vb[8];
  #pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int s = tid + (it0 + j) * NT;
              vb[j] = it0 + j < iters && s < ncmp;
              kb[j] = 0u;
              if (vb[j]) {
                vb[j] = !((loc[s >> 5] >> (s & 31)) & 1u);
                kb[j] = okey(sc[s]);
                vb[j] = vb[j] && ((kb[j] & mask) == prefix);
              }
            }
  #pragma unroll
            for (int j = 0; j < 8; ++j) warp_inc(hist, (kb[j] >> shift) & 255u, vb[j]);
          }
          __syncthreads();
          if (warp == 0) {
            unsigned bin, ab;
            bool ok;
            find_bin(hist, (unsigned)need_g - s_sel[2], bin, ab, ok);
            if (lane == 0) {
              if (!ok) atomicOr(a.err, ERR_BAD_COUNT);
              s_sel[0] |= bin << shift;
              s_sel[1] |= 255u << shift;
              s_sel[2] += ab;
              if (ro == 3) s_sel[3] = hist[bin];
            }
          }
          __syncthreads();
        }
      }
      const unsigned T = s_sel[0];
      const unsigned need_eq = need_g > 0 ? (unsigned)need_g - s_sel[2] : 0u;
      const bool all_ties = need_g > 0 && s_sel[3] == need_eq;
      const bool rank_ties = need_g > 0 && !all_ties;
      // ties at T beyond need_eq are ranked in slot order (lower slot first):
      // tie bits per word, then their exclusive prefix counts
      if (rank_ties) {
        for (int w = warp; w < words; w += NWARP) {
          const int s = w * 32 + lane;
          bool eq = false;
          if (s < ncmp && !((loc[w] >> lane) & 1u)) eq = okey(sc[s]) == T;
          const unsigned b = __ballot_sync(0xffffffffu, eq);
          if (lane == 0) tmp[w] = b;
        }
        __syncthreads();
        word_prefix(tmp, pre, words, red);
      }
      // final keep words: local picks | global picks | recent window
      for (int w = warp; w < words; w += NWARP) {
        const int s = w * 32 + lane;
        bool kp = (loc[w] >> lane) & 1u;
        if (!kp && s < ncmp && need_g > 0) {
          const unsigned k = okey(sc[s]);
          if (k > T) {
            kp = true;
          } else if (k == T) {
            kp = all_ties || (pre[w] + __popc(tmp[w] & ((1u << lane) - 1u))) < need_eq;
          }
        }
        if (s >= ncmp) kp = true;
        const unsigned b = __ballot_sync(0xffffffffu, kp);
        if (lane == 0) keep[w] = b;
      }
      __syncthreads();
    };
    const int quota = min(a.k_loc, kt / P);
    // Fast path, exact whenever it applies: take the global top-K_t of ALL
    // candidates first.  Its drop set D0 is a suffix of the (score desc,
    // slot asc) order, so each block's kept part is a prefix of the block.
    // If every block keeps at least its quota k_loc', each block's top
    // k_loc' (S_loc) lies outside D0, and the Eq. 10 drop set -- the bottom
    // of C minus S_loc -- is D0 itself.  Otherwise Eq. 10 runs in full.
    global_keep();
    if (tid == 0) s_fast = 1;
    __syncthreads();
    for (int j = warp; j < P; j += NWARP) {
      const int lo = j * PAGE, hi = min(lo + PAGE, ncmp);
      const int kj = min(quota, hi - lo);
      if (kj <= 0) continue;
      unsigned c = 0;
      if (lane < PAGE / 32) {
        const int w = (lo >> 5) + lane, s0 = w * 32;
        if (s0 < hi) {
          const int nb = min(32, hi - s0);
          c = __popc(keep[w] & (nb == 32 ? 0xffffffffu : ((1u << nb) - 1u)));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0 && c < (unsigned)kj) s_fast = 0;
    }
    __syncthreads();
    if (!s_fast) {
      // ---- Eq. 10, block-local part: TopK_{k_loc'}(B_j) per logical block ----
      // Bit-serial radix select of each block's kj-th largest key: at each bit
      // the keys that match the prefix and have the bit set are counted with
      // warp ballots.  A warp takes GB blocks at once, so their
      // independent reduction chains overlap.  Afterwards prefix = that key
      // and above = the number of keys above it.
      constexpr int GB = 4;
      for (int j0 = warp; j0 < P; j0 += NWARP * GB) {
        unsigned key[GB][8], prefix[GB], above[GB], need[GB];
        bool val[GB][8];
        int kjv[GB];
  #pragma unroll
        for (int g = 0; g < GB; ++g) {
          const int j = j0 + g * NWARP;
          const int lo = j * PAGE;
          const int hi = min(lo + PAGE, ncmp);
          kjv[g] = j < P ? max(0, min(quota, hi - lo)) : 0;
  #pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = lo + 32 * e + lane;
            val[g][e] = j < P && s < hi;
            key[g][e] = val[g][e] ? okey(sc[s]) : 0u;
          }
          prefix[g] = 0u;
          above[g] = 0u;
          need[g] = (unsigned)kjv[g];
        }
        unsigned mask = 0u;
        for (int bit = 31; bit >= 0; --bit) {
          const unsigned m2 = mask | (1u << bit);
          unsigned tot[GB];
  #pragma unroll
          for (int g = 0; g < GB; ++g) {
            const unsigned p2 = prefix[g] | (1u << bit);
            unsigned c = 0;
  #pragma unroll
            for (int e = 0; e < 8; ++e)
              c += (unsigned)__popc(__ballot_sync(0xffffffffu, val[g][e] && (key[g][e] & m2) == p2));
            tot[g] = c;
          }
  #pragma unroll
          for (int g = 0; g < GB; ++g) {
            if (tot[g] >= need[g]) {
              prefix[g] |= 1u << bit;
            } else {
              need[g] -= tot[g];
              above[g] += tot[g];
            }
          }
          mask = m2;
        }
  #pragma unroll
        for (int g = 0; g < GB; ++g) {
          if (kjv[g] <= 0) continue;
          const int lo = (j0 + g * NWARP) * PAGE;
          const unsigned need_eq = (unsigned)kjv[g] - above[g];
          unsigned run = 0;
  #pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool gt = val[g][e] && key[g][e] > prefix[g];
            const bool eq = val[g][e] && key[g][e] == prefix[g];
            const unsigned be = __ballot_sync(0xffffffffu, eq);
            const unsigned rank = run + __popc(be & ((1u << lane) - 1u));
            run += __popc(be);
            const unsigned bw = __ballot_sync(0xffffffffu, gt || (eq && rank < need_eq));
            if (lane == 0) loc[(lo >> 5) + e] = bw;
          }
        }
      }
      __syncthreads();

      __syncthreads();
      global_keep();
    }
  }

  // ---- validate: exactly (P-1) b slots kept ------------------------------
  {
    unsigned c = 0;
    for (int w = tid; w < words; w += NT) c += __popc(keep[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) red[warp] = c;
    __syncthreads();
    if (tid == 0) {
      unsigned tot = 0;
      for (int w = 0; w < NWARP; ++w) tot += red[w];
      if (s_abort) {
        atomicOr(a.err, ERR_TIMEOUT);  // the selection ran on scores still being staged
      } else if (tot != target_kept) {
        s_abort = 2;
        atomicOr(a.err, a.keep_in ? ERR_BAD_MASK : ERR_BAD_COUNT);
      }
    }
    __syncthreads();
  }
  if (a.keep_out) {
    uint32_t* dst = a.keep_out + rq.mask_off + (size_t)unit * words;
    for (int w = tid; w < words; w += NT) dst[w] = keep[w];
  }
  if (s_abort) {
    // a staging copy of the scores may still be in flight (bounded wait)
    if (tid == 0 && s_stage0) bar_wait(smem_addr(&full_bar[0]), 0u, kDrainLimit);
    __syncthreads();
    return;
  }
  if (a.select_only) return;  // the keep masks were all that was asked for

  // ---- compaction ---------------------------------------------------------
  word_prefix(keep, pre, words, red);
  // hole-fill mode: the holes (slots of [0, (P-1) b) not kept), in order;
  // the k-th kept slot of the last page fills the k-th hole
  const int lastp = (P - 1) * PAGE;
  if (a.fill) {
    if (warp == 0) {
      int nh = 0;
      for (int w = 0; w < lastp / 32; ++w) {
        const bool hole = !((keep[w] >> lane) & 1u);
        const unsigned b = __ballot_sync(0xffffffffu, hole);
        if (hole && nh + __popc(b & ((1u << lane) - 1u)) < PAGE) s_hole[nh + __popc(b & ((1u << lane) - 1u))] = w * 32 + lane;
        nh += __popc(b);
      }
      if (lane == 0) {
        if (nh > PAGE) atomicOr(a.err, ERR_BAD_COUNT);
        s_nholes = min(nh, PAGE);
      }
    }
    __syncthreads();
  }
  const int kept_first = lastp - (a.fill ? s_nholes : 0);  // kept slots of the first P-1 pages
  constexpr int CR = (16384 / RB) < 64 ? (16384 / RB) : 64;  // rows per chunk: K and V of it fill a stage
  constexpr int PIECES = RB / 16;                            // 16-byte pieces per row
  static_assert(2 * CR * RB <= STAGE_BYTES && PAGE % CR == 0 && CR % 32 == 0, "chunk shape");
  const size_t head_stride = (size_t)PAGE * RB;
  unsigned char* kc = static_cast<unsigned char*>(a.k_cache);
  unsigned char* vc = static_cast<unsigned char*>(a.v_cache);
  const size_t lbase = (size_t)layer * a.num_pages_total;
  const int nchunks = N / CR;
  // Logical slot i's target slot, or -1 when the row is not kept or stays where it is.
  auto target = [&](int i) -> int {
    const int w = i >> 5, bit = i & 31;
    const unsigned word = keep[w];
    if (!((word >> bit) & 1u)) return -1;
    int dst;
    if (a.fill) {
      // kept rows of the first P-1 pages stay; the last page's kept rows fill the holes
      const int rank = (int)(pre[w] + __popc(word & ((1u << bit) - 1u))) - kept_first;
      dst = i < lastp ? i : s_hole[min(PAGE - 1, max(0, rank))];
    } else {
      dst = (int)(pre[w] + __popc(word & ((1u << bit) - 1u)));
    }
    return (s_old[i >> 8] == s_new[dst >> 8] && (i & 255) == (dst & 255)) ? -1 : dst;
  };
  // chunks that move any row, in order (loc is free once the keep words exist)
  unsigned* list = loc;
  for (int w = tid; w < (nchunks + 31) / 32; w += NT) tmp[w] = 0u;
  __syncthreads();
  for (int c = warp; c < nchunks; c += NWARP) {
    bool mv = false;
    for (int r = lane; r < CR; r += 32) mv |= target(c * CR + r) >= 0;
    const bool any = __any_sync(0xffffffffu, mv);
    if (lane == 0 && any) atomicOr(&tmp[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  if (warp == 0) {
    int n = 0;
    for (int base = 0; base < nchunks; base += 32) {
      const bool f = base + lane < nchunks && ((tmp[(base >> 5)] >> lane) & 1u);
      const unsigned b = __ballot_sync(0xffffffffu, f);
      if (f) list[n + __popc(b & ((1u << lane) - 1u))] = (unsigned)(base + lane);
      n += __popc(b);
    }
    if (lane == 0) s_nlist = n;
  }
  __syncthreads();
  const int nlist = s_nlist;
  // one thread streams chunk k of the list into stage k % CSTAGES
  auto issue = [&](int k) {
    const int c = (int)list[k], st = k % CSTAGES;
    const int i0 = c * CR;
    const int sp = s_old[i0 >> 8];
    const uint32_t bar = smem_addr(&full_bar[st]);
    const size_t src = ((lbase + (size_t)sp) * a.Hkv + h) * head_stride + (size_t)(i0 & 255) * RB;
    const bool ok = sp >= 0 && sp < a.num_pages_total && ((reinterpret_cast<uintptr_t>(kc + src) |
                                                          reinterpret_cast<uintptr_t>(vc + src)) & 15) == 0;
    if (!ok) {
      // a bad source: record it and complete the phase without data
      atomicOr(a.err, ERR_BAD_PAGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      return;
    }
    const uint32_t dk = smem_addr(stage_mem + (size_t)st * STAGE_BYTES);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"((uint32_t)(2 * CR * RB))
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dk),
                 "l"(kc + src), "r"((uint32_t)(CR * RB)), "r"(bar)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dk + (uint32_t)(CR * RB)),
                 "l"(vc + src), "r"((uint32_t)(CR * RB)), "r"(bar)
                 : "memory");
  };
  // parity of the phase that chunk k completes on its stage's barrier
  const int stage0_used = s_stage0;
  auto phase = [&](int k) -> uint32_t {
    return (uint32_t)(((k / CSTAGES) + (k % CSTAGES == 0 ? stage0_used : 0)) & 1);
  };
  if (tid == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stages held the scores
    for (int k = 0; k < CSTAGES && k < nlist; ++k) issue(k);
  }
  unsigned moved_rows = 0;
  int done = 0;  // chunks consumed
  for (int k = 0; k < nlist; ++k) {
    const int st = k % CSTAGES;
    if (!bar_wait(smem_addr(&full_bar[st]), phase(k), a.wait_limit)) atomicOr(&s_abort, 1);
    __syncthreads();
    if (s_abort) break;  // every thread reads it after the barrier: all leave together
    const int c = (int)list[k];
    const unsigned char* sk = stage_mem + (size_t)st * STAGE_BYTES;
    for (int pidx = tid; pidx < CR * PIECES; pidx += NT) {
      const int row = pidx / PIECES, q = pidx % PIECES;
      const int i = c * CR + row;
      const int dst = target(i);
      if (dst < 0) continue;
      const int dp = s_new[dst >> 8];
      if (dp < 0 || dp >= a.num_pages_total) {
        atomicOr(a.err, ERR_BAD_PAGE);
        continue;
      }
      const size_t doff = ((lbase + s_new[dst >> 8]) * a.Hkv + h) * head_stride + (size_t)(dst & 255) * RB + q * 16;
      *reinterpret_cast<uint4*>(kc + doff) = *reinterpret_cast<const uint4*>(sk + (size_t)row * RB + q * 16);
      *reinterpret_cast<uint4*>(vc + doff) =
          *reinterpret_cast<const uint4*>(sk + (size_t)CR * RB + (size_t)row * RB + q * 16);
      if (q == 0) ++moved_rows;
    }
    done = k + 1;
    __syncthreads();  // the stage has been read: refill it with chunk k + CSTAGES
    if (tid == 0 && k + CSTAGES < nlist) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(k + CSTAGES);
    }
  }
  if (s_abort) {
    // copies still in flight land before the CTA's shared memory goes away (bounded)
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      for (int k = done; k < nlist && k < done + CSTAGES; ++k)
        bar_wait(smem_addr(&full_bar[k % CSTAGES]), phase(k), kDrainLimit);
    }
    __syncthreads();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) moved_rows += __shfl_xor_sync(0xffffffffu, moved_rows, o);
  if (lane == 0 && moved_rows) atomicAdd(a.moved, (unsigned long long)moved_rows);
}

}  // namespace

template <int RB>
cudaError_t launch_rb(const CompressArgs& a, cudaStream_t s) {
  static bool attr = false;
  const int smem = CSTAGES * STAGE_BYTES;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(k_compress<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_compress<RB><<<dim3(a.n_work * a.L * a.Hkv), NT, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE || a.wait_limit < 0) return cudaErrorInvalidValue;
  switch (a.D * a.elt) {
    case 128: return launch_rb<128>(a, s);
    case 256: return launch_rb<256>(a, s);
    case 512: return launch_rb<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gp
