// Compress & Hold kernel for sm_103a: GrowPage Sec. 3.3 Eqs. 9-10 and
// App. E.2, one CTA per (request, layer, KV head).
//
//  selection  -- importance s = max(a^S, a^L) comes from the cache the demand
//                kernel wrote (log2 domain; the order is the same).  The
//                protected recent window [P b - R, P b) is always kept.
//                Block-local: warp w takes logical blocks w, w+8, ... and
//                keeps the top k_loc' of each (radix select on
//                order-preserving 32-bit keys, per-warp 256-bin
//                histograms).  Global: a CTA-wide radix select keeps the top
//                K_t - |S_loc| of the remaining candidates.  Equal scores are
//                resolved towards the lower slot.
//  compaction -- order-preserving stream compaction: the k-th kept slot moves
//                to logical slot k of the target block table (ballot/popc +
//                word prefix scan).  Source and target tables differ only in
//                pages replaced by copy-on-write (fresh pages), so in-place
//                moves only ever go to a lower logical slot; each 64-slot
//                chunk is read completely into registers before any of its
//                rows is written, which makes the in-place pass race-free.
//                Rows whose physical location does not change are skipped.
#include <cstdint>

#include "gp_kernels.h"

namespace gp {
namespace {

constexpr int NT = 256;
constexpr int NWARP = 8;
constexpr int PAGE = 256;
constexpr int MAX_WORDS = 256 * PAGE / 32;  // 256 pages

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
__global__ void __launch_bounds__(NT) k_compress(CompressArgs a) {
  __shared__ unsigned keep[MAX_WORDS];
  __shared__ unsigned loc[MAX_WORDS];     // block-local picks (Eq. 10, S_loc)
  __shared__ unsigned tmp[MAX_WORDS];     // tie bits
  __shared__ unsigned pre[MAX_WORDS];     // exclusive word prefixes
  __shared__ unsigned whist[NWARP][256];
  __shared__ unsigned red[NWARP];
  __shared__ int s_old[PAGE], s_new[PAGE];
  __shared__ unsigned s_sel[4];           // prefix, mask, above, flags
  __shared__ int s_abort;

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
  const int kt = (P - 1) * PAGE - a.R;
  const unsigned target_kept = (unsigned)((P - 1) * PAGE);

  if (tid == 0) s_abort = 0;
  for (int j = tid; j < P; j += NT) {
    s_old[j] = a.old_bt[rq.bt_off + j];
    s_new[j] = a.new_bt[rq.bt_off + j];
  }

  if (a.keep_in) {
    const unsigned* src = a.keep_in + rq.mask_off + (size_t)unit * words;
    for (int w = tid; w < words; w += NT) keep[w] = src[w];
    __syncthreads();
  } else {
    const float* sc = a.scores + rq.score_off + (size_t)unit * ncmp;
    for (int w = tid; w < words; w += NT) loc[w] = 0u;
    __syncthreads();
    // ---- Eq. 10, block-local part: TopK_{k_loc'}(B_j) per logical block ----
    const int quota = min(a.k_loc, kt / P);
    for (int j = warp; j < P; j += NWARP) {
      const int lo = j * PAGE;
      const int hi = min(lo + PAGE, ncmp);
      const int kj = min(quota, hi - lo);
      if (kj <= 0) continue;
      unsigned key[8];
      bool val[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int s = lo + 32 * e + lane;
        val[e] = s < hi;
        key[e] = val[e] ? okey(sc[s]) : 0u;
      }
      unsigned prefix = 0, mask = 0, above = 0;
      for (int ro = 0; ro < 4; ++ro) {
        const int shift = 24 - 8 * ro;
        for (int q = lane; q < 256; q += 32) whist[warp][q] = 0u;
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          warp_inc(whist[warp], (key[e] >> shift) & 255u, val[e] && ((key[e] & mask) == prefix));
        __syncwarp();
        unsigned bin, ab;
        bool ok;
        find_bin(whist[warp], (unsigned)kj - above, bin, ab, ok);
        if (!ok && lane == 0) atomicOr(a.err, ERR_BAD_COUNT);
        prefix |= bin << shift;
        mask |= 255u << shift;
        above += ab;
        __syncwarp();
      }
      const unsigned need_eq = (unsigned)kj - above;
      unsigned run = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool gt = val[e] && key[e] > prefix;
        const bool eq = val[e] && key[e] == prefix;
        const unsigned be = __ballot_sync(0xffffffffu, eq);
        const unsigned rank = run + __popc(be & ((1u << lane) - 1u));
        run += __popc(be);
        const unsigned bw = __ballot_sync(0xffffffffu, gt || (eq && rank < need_eq));
        if (lane == 0) loc[(lo >> 5) + e] = bw;
      }
    }
    __syncthreads();
    // ---- Eq. 10, global part: TopK_{K_t - |S_loc|}(C \ S_loc) ----------------
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
    unsigned* hist = whist[0];
    if (need_g > 0) {
      for (int ro = 0; ro < 4; ++ro) {
        const int shift = 24 - 8 * ro;
        hist[tid] = 0u;
        __syncthreads();
        const unsigned prefix = s_sel[0], mask = s_sel[1];
        for (int it = 0; it < iters; ++it) {
          const int s = tid + it * NT;
          bool v = s < ncmp;
          unsigned k = 0;
          if (v) {
            v = !((loc[s >> 5] >> (s & 31)) & 1u);
            k = okey(sc[s]);
            v = v && ((k & mask) == prefix);
          }
          warp_inc(hist, (k >> shift) & 255u, v);
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
      if (tot != target_kept) {
        s_abort = 1;
        atomicOr(a.err, a.keep_in ? ERR_BAD_MASK : ERR_BAD_COUNT);
      }
    }
    __syncthreads();
  }
  if (a.keep_out) {
    uint32_t* dst = a.keep_out + rq.mask_off + (size_t)unit * words;
    for (int w = tid; w < words; w += NT) dst[w] = keep[w];
  }
  if (s_abort) return;

  // ---- compaction ---------------------------------------------------------
  word_prefix(keep, pre, words, red);
  constexpr int PIECES = RB / 16;          // 16-byte pieces per row
  constexpr int ROWS_PASS = NT / PIECES;   // rows per pass
  constexpr int E = 64 / ROWS_PASS;        // passes per 64-slot chunk
  const size_t head_stride = (size_t)PAGE * RB;
  unsigned char* kc = static_cast<unsigned char*>(a.k_cache);
  unsigned char* vc = static_cast<unsigned char*>(a.v_cache);
  const size_t lbase = (size_t)layer * a.num_pages_total;
  const int q = tid % PIECES;
  unsigned moved_rows = 0;
  const int nchunks = N / 64;
  for (int c = 0; c < nchunks; ++c) {
    uint4 kv[E], vv[E];
    size_t doff[E];
    bool mv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = c * 64 + tid / PIECES + e * ROWS_PASS;
      const int w = i >> 5, bit = i & 31;
      const unsigned word = keep[w];
      mv[e] = false;
      doff[e] = 0;
      if ((word >> bit) & 1u) {
        const int dst = (int)(pre[w] + __popc(word & ((1u << bit) - 1u)));
        const int sp = s_old[i >> 8], so = i & 255;
        const int dp = s_new[dst >> 8], dof = dst & 255;
        if (sp != dp || so != dof) {
          mv[e] = true;
          const size_t soff = ((lbase + sp) * a.Hkv + h) * head_stride + (size_t)so * RB + q * 16;
          doff[e] = ((lbase + dp) * a.Hkv + h) * head_stride + (size_t)dof * RB + q * 16;
          kv[e] = *reinterpret_cast<const uint4*>(kc + soff);
          vv[e] = *reinterpret_cast<const uint4*>(vc + soff);
          if (q == 0) ++moved_rows;
        }
      }
    }
    __syncthreads();  // every source row of this chunk is in registers
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (mv[e]) {
        *reinterpret_cast<uint4*>(kc + doff[e]) = kv[e];
        *reinterpret_cast<uint4*>(vc + doff[e]) = vv[e];
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) moved_rows += __shfl_xor_sync(0xffffffffu, moved_rows, o);
  if (lane == 0 && moved_rows) atomicAdd(a.moved, (unsigned long long)moved_rows);
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  if (a.n_work == 0) return cudaSuccess;
  if (a.b != PAGE) return cudaErrorInvalidValue;
  const int rb = a.D * a.elt;
  const dim3 grid(a.n_work * a.L * a.Hkv);
  switch (rb) {
    case 128: k_compress<128><<<grid, NT, 0, s>>>(a); break;
    case 256: k_compress<256><<<grid, NT, 0, s>>>(a); break;
    case 512: k_compress<512><<<grid, NT, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gp
