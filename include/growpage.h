/*
 * growpage.h -- C ABI of a GB300-native (sm_103a) capacity-boundary engine
 * for GrowPage ("GrowPage: On-Demand KV Budgeting for Efficient LLM
 * Reasoning Serving", arXiv 2609.03494) over a paged KV cache.
 *
 * What the engine computes (paper sections in brackets):
 *   - every decode step: the dual-timescale query summaries      [Sec. 3.2 Eq. 6, App. E.1]
 *   - at a capacity boundary: calibration + RoPE of both summaries,
 *     scores against every cached key through the block table,
 *     softmax, GQA mean and the p-coverage demand D_p per
 *     (layer, KV head), and the request-level trend Delta          [Sec. 3.2 Eqs. 7-8, App. E.1 Eq. 12]
 *   - the decision Grow by One Page vs Compress & Hold             [Sec. 3.2, Sec. 4.2]
 *   - Grow: append a fresh page to the block table                 [Sec. 3.3, Sec. 4.2]
 *   - Compress & Hold: importance max(a^S, a^L), protected recent
 *     window, block-local + global top-k, and copy-on-write
 *     compaction of the retained K/V into (P-1) b slots            [Sec. 3.3 Eqs. 9-10, App. E.2]
 *   - a refcounted page pool and a slot pool for the summaries    [Sec. 4.2, App. E.1 Eq. 11, App. E.2]
 *
 * Conventions
 *   - Every call returns gp_status; nothing throws across the ABI.  The
 *     text of the last failure is available from gp_last_error().
 *   - Device pointers ("_dev") are CUDA device addresses owned by the caller
 *     (for example PyTorch tensors); host pointers are plain memory owned by
 *     the caller.  The engine owns the summary pool, its scratch buffers, the
 *     page refcounts, the free-page list and the slot list.
 *   - All device work is issued on the stream given to gp_create, in call
 *     order.  gp_boundary_demand synchronises that stream before returning
 *     (the decision is a host decision, Sec. 4.2); the other hot-path calls
 *     are asynchronous.
 *   - Allocation failures (GP_ERR_NO_PAGES, GP_ERR_NO_SLOTS) leave every
 *     piece of state unchanged.
 *   - A context is not thread-safe; use one per host thread.
 *
 * Layouts
 *   K and V caches: [L][num_pages][Hkv][page_size][head_dim] of kv_dtype,
 *     so one (layer, page, KV head) tile is page_size * head_dim contiguous
 *     elements (64 KiB for bf16, d = 128, page_size = 256).
 *   Query summaries (engine-owned, fp64): [L][max_slots][2][Hq][head_dim],
 *     index 0 = short (beta_s), 1 = long (beta_l)  (App. E.1 Eq. 11).  fp64
 *     because the long summary's 1 - beta_l = 0.001 increments and the
 *     large logits of concentrated heads need more than fp32's 24 bits to
 *     keep importance scores within 1e-5 relative.
 *   Queries: [L][n][Hq][head_dim] of q_dtype, normalised and pre-RoPE.
 *   Query head j belongs to KV head j / (Hq / Hkv).
 *
 * EMA convention (fixed here because the paper's pages disagree): the stored
 * beta is the decay, the weight on the previous summary:
 *   qbar <- beta * qbar + (1 - beta) * q,  beta_s = 0.9 < beta_l = 0.999.
 */
#ifndef GROWPAGE_H
#define GROWPAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GP_OK = 0,
  GP_ERR_INVALID = 1,     /* bad argument; nothing changed */
  GP_ERR_NO_PAGES = 2,    /* the free pool cannot supply the pages; nothing changed */
  GP_ERR_NO_SLOTS = 3,    /* no free summary slot; nothing changed */
  GP_ERR_CUDA = 4,        /* a CUDA runtime call failed (text in gp_last_error) */
  GP_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (about one second of SM
                             clock); the kernel drained its copies and returned, so the
                             context stays usable, but that launch's outputs are
                             unspecified */
  GP_ERR_STATE = 6,       /* call out of order (e.g. compress without a fresh demand) */
  GP_ERR_UNSUPPORTED = 7  /* shape outside what the kernels were built for */
} gp_status;

typedef enum { GP_DTYPE_BF16 = 0, GP_DTYPE_F32 = 1 } gp_dtype;
/* Capacity-control policies (GrowPage Sec. 3.2; the alternatives of App. H.1):
 * GROWPAGE  Grow iff Delta > tau, else Compress & Hold;
 * FIXED     never Grow (GrowPage-Fixed);
 * RANDOM    Compress & Hold with probability random_compress, else Grow,
 *           whatever Delta (GrowPage-Random); the draw of the engine's k-th
 *           decision (k = 0, 1, ... since gp_create) is
 *           u_k = (splitmix64(random_seed * 2^32 + k) >> 11) * 2^-53;
 * INVERSE   Grow iff Delta <= tau, else Compress & Hold (GrowPage-Inverse);
 * SHRINK    Eq. 13: Shrink iff Delta < shrink_threshold, Grow iff Delta > tau,
 *           else Compress & Hold; Shrink only while the request holds more
 *           than shrink_floor_pages pages (App. H.1: 1024 tokens), else
 *           Compress & Hold. */
typedef enum {
  GP_POLICY_GROWPAGE = 0,
  GP_POLICY_FIXED = 1,
  GP_POLICY_RANDOM = 2,
  GP_POLICY_INVERSE = 3,
  GP_POLICY_SHRINK = 4
} gp_policy;
typedef enum { GP_ACT_GROW = 0, GP_ACT_COMPRESS = 1, GP_ACT_SHRINK = 2 } gp_action_kind;
/* Working-set metric of the demand estimation.
 *   TOP_P:   K^x = D_p(a^x) over C_t (Eq. 2, Eq. 7), the method's metric.
 *   ENTROPY: the ablation of Sec. 5.3 (Table 2) that puts attention entropy
 *            in its place.  The pages give no formula; the engine takes the
 *            entropy's effective support size E^x = exp(H(a^x)),
 *            H(a) = -sum_i a_i ln a_i over C_t (1 for a point mass, |C_t| for
 *            the uniform distribution), and uses it where K^x stands in
 *            Eq. 8.  D_p is still computed and reported. */
typedef enum { GP_METRIC_TOP_P = 0, GP_METRIC_ENTROPY = 1 } gp_metric;

/* Engine configuration.  Defaults (gp_config_default) follow the paper:
 * page_size 256, recent_window 16, k_loc 64, beta_s 0.9, beta_l 0.999,
 * p 0.99, tau 0, max_slots 512 (Sec. 3.2, Sec. 5.1, App. D, App. E.1). */
typedef struct gp_config {
  int32_t num_layers;        /* L */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv; Hq / Hkv in {1, 2, 4, 8} */
  int32_t head_dim;          /* d: 64 or 128 */
  int32_t page_size;         /* b: 256 (the only size the kernels support) */
  int32_t kv_dtype;          /* gp_dtype of the K/V caches */
  int32_t q_dtype;           /* gp_dtype of the query inputs */
  int32_t max_slots;         /* M: rows of the summary pool */
  int32_t num_pages;         /* physical pages in the K/V caches */
  int32_t max_pages_per_req; /* block-table capacity; at most 256 */
  int32_t recent_window;     /* R: always-kept recent tokens, 0 <= R < b */
  int32_t k_loc;             /* Eq. 10 per-block quota */
  int32_t reserve_pages;     /* Grow only while free pages > reserve (Sec. 4.2) */
  int32_t policy;            /* gp_policy */
  double beta_s;             /* short-summary decay */
  double beta_l;             /* long-summary decay */
  double p;                  /* coverage target of D_p, 0 < p < 1 */
  double tau;                /* decision threshold on Delta */
  double rope_theta;         /* rotate-half RoPE base */
  /* policy variants (App. H.1); defaults 0.7, -0.005, 4 pages, 0 */
  double random_compress;    /* RANDOM: probability of Compress & Hold */
  double shrink_threshold;   /* SHRINK: Shrink iff Delta < this */
  int32_t shrink_floor_pages;/* SHRINK: no Shrink at or below this many pages */
  uint32_t random_seed;      /* RANDOM: seed of the counter-based draws */
  int32_t demand_metric;     /* gp_metric; default TOP_P */
} gp_config;

/* One request as the caller's scheduler sees it.  block_table is a HOST
 * array owned by the caller, capacity max_pages_per_req, holding num_pages
 * physical page ids in logical order.  gp_grow_page and gp_compress_hold
 * rewrite it in place.  pos is the current decode position (tokens
 * generated so far, evicted ones included); RoPE of the summaries uses it. */
typedef struct gp_request {
  int32_t slot;
  int32_t num_pages;
  int32_t* block_table;
  int64_t pos;
} gp_request;

/* Result of the demand estimation for one request (Eqs. 7-8):
 * sum_k_short = sum over (layer, KV head) of K^S, likewise sum_k_long;
 * num_candidates = |C_t| = (P - 1) * b; num_units = L * Hkv;
 * delta = (sum_k_short - sum_k_long) / (num_candidates * num_units).
 * Under GP_METRIC_ENTROPY, eff_short / eff_long = sums over the units of
 * exp(H(a^S)) / exp(H(a^L)) (in unit order), and
 * delta = (eff_short - eff_long) / (num_candidates * num_units); under
 * TOP_P both are 0. */
typedef struct gp_demand {
  int64_t sum_k_short;
  int64_t sum_k_long;
  int32_t num_candidates;
  int32_t num_units;
  double delta;
  double eff_short;
  double eff_long;
} gp_demand;

typedef struct gp_action {
  int32_t kind;      /* gp_action_kind */
  int32_t fallback;  /* 1: Delta asked for Grow but the pool could not grant it */
  int32_t forced;    /* 1: P == 1, nothing to compress, Grow forced */
} gp_action;

typedef struct gp_stats_t {
  int64_t demand_calls;
  int64_t demand_requests;
  int64_t grow;
  int64_t compress;
  int64_t fallback;
  int64_t forced_grow;
  int64_t cow_pages;       /* shared pages replaced by copy-on-write */
  int64_t moved_rows;      /* (layer, head, token) rows moved by compaction */
  int64_t shrink;          /* Shrink decisions (policy SHRINK) */
} gp_stats_t;

typedef struct gp_ctx gp_ctx;

/* ---- lifecycle --------------------------------------------------------- */

/* Fill *cfg with the paper's defaults (shape fields zero). */
gp_status gp_config_default(gp_config* cfg);

/* Create an engine.  k_cache / v_cache: device base addresses of the caller's
 * caches (layout above), which must stay alive and unmoved for the engine's
 * lifetime.  stream: a cudaStream_t (NULL = legacy default stream).
 * If k_cache and v_cache are both NULL the context is host-only: pages,
 * refcounts, slots and decisions work, no CUDA call is made, and the device
 * calls return GP_ERR_STATE.  On success *out owns the engine. */
gp_status gp_create(const gp_config* cfg, void* k_cache, void* v_cache,
                    void* stream, gp_ctx** out);
gp_status gp_destroy(gp_ctx* ctx);
const char* gp_last_error(const gp_ctx* ctx);
const char* gp_status_string(gp_status st);

/* ---- page pool with refcounts (Sec. 4.2, App. E.2) -----------------------
 * Pages index the caller's caches.  Allocation is deterministic: the lowest
 * free id.  gp_page_ref shares a page (prefix caching); gp_page_unref drops
 * one reference and frees the page at zero; an unref of a free page is
 * GP_ERR_INVALID. */
gp_status gp_page_alloc(gp_ctx* ctx, int32_t* page);
gp_status gp_page_ref(gp_ctx* ctx, int32_t page);
gp_status gp_page_unref(gp_ctx* ctx, int32_t page);
gp_status gp_page_refcount(const gp_ctx* ctx, int32_t page, int32_t* rc);
gp_status gp_free_page_count(const gp_ctx* ctx, int32_t* n);

/* ---- summary slots (App. E.1) --------------------------------------------
 * A slot is bound to a running request; its first gp_update_summaries must
 * pass first = 1, which overwrites stale values (no clearing needed). */
gp_status gp_slot_acquire(gp_ctx* ctx, int32_t* slot);
gp_status gp_slot_release(gp_ctx* ctx, int32_t slot);

/* ---- hot path -------------------------------------------------------------
 * gp_update_summaries: Sec. 3.2 Eq. 6 with the App. E.1 initialisation, for
 * n requests of one decode step.  slots_dev: int32[n] device; q_dev:
 * [L][n][Hq][d] q_dtype device; first_dev: uint8[n] device (1 = slot's first
 * step).  Asynchronous.  Slot ids out of range are skipped and reported as
 * GP_ERR_INVALID by the next synchronising call. */
gp_status gp_update_summaries(gp_ctx* ctx, int32_t n, const int32_t* slots_dev,
                              const void* q_dev, const uint8_t* first_dev);

/* gp_boundary_demand: for n requests at a capacity boundary (each holding
 * num_pages full pages), App. E.1 Eq. 12 calibration against q_cur, RoPE at
 * pos, scores of both summaries against every key of the request through
 * its block table, softmax over C_t = [0, (P-1) b) and D_p per (layer, KV
 * head) (Eqs. 2 and 7), and Delta (Eq. 8).  q_cur_dev: [L][n][Hq][d] q_dtype
 * device (the same q_t just passed to gp_update_summaries).  out: host
 * gp_demand[n].  It also caches, per (layer, KV head), the importance
 * max(a^S, a^L) of Eq. 9 over [0, P b - R) for a following
 * gp_compress_hold.  Synchronises the stream. */
gp_status gp_boundary_demand(gp_ctx* ctx, int32_t n, const gp_request* reqs,
                             const void* q_cur_dev, gp_demand* out);

/* gp_boundary_demand_noalloc: the same demand estimation as
 * gp_boundary_demand (same kernels, same results) for callers that must not
 * allocate memory -- for example a serving process that reserves all of its
 * GPU memory at start-up so that no request can fail later on an
 * out-of-memory error and no cudaMalloc/cudaFree synchronises the device
 * mid-flight.  The paper has no counterpart to this call.
 * It calls no cudaMalloc, cudaFree or other allocating routine: every
 * temporary (request descriptors, block tables, calibrated summaries and
 * their tensor-core operands, importance values, a-values, arrival tickets,
 * per-unit D_p and their sums) lives in one file-scope device array of
 * 64 MiB that every GPU loading the library holds until the process exits.
 * A call needing more is rejected with GP_ERR_INVALID and a message naming
 * the size; n is at most 512.  The need: per request, its importance values
 * and a-values, L * Hkv * (4 (P b - R) + 8 (P - 1) b) bytes (about
 * 12 L Hkv P b; each region rounded up to 256 bytes), plus per (layer, KV
 * head) of every request 16 * 8 * 26 bytes of partial softmax statistics,
 * 8 G d bytes of calibrated summaries, (d / 64) * 128 * ceil(6 G / 16) * 16
 * bytes of tensor-core operand and 16 bytes of counters -- about 15.3 KiB at
 * d = 128, G = 4 -- plus small descriptor arrays.  On the first call on a device, with that device current, the
 * array's address is looked up once (cudaGetSymbolAddress); make that first
 * call before any stream capture.  All calls share the array and its host
 * staging, which keep the last call's contents: calls that overlap on the
 * GPU, or run on several host threads at once, race.  Inputs and outputs
 * are the caller's: out is host gp_demand[n]; k_units, if not NULL, is host
 * int32[n][L * Hkv][2] receiving K^S, K^L per (layer, KV head).  It does not
 * prepare a following gp_compress_hold: the demand records that an earlier
 * gp_boundary_demand left for these slots are dropped, so a
 * gp_compress_hold of them returns GP_ERR_STATE until the next
 * gp_boundary_demand.  Device-side errors are reported as by gp_synchronize.
 * Contexts with demand_metric GP_METRIC_ENTROPY are refused
 * (GP_ERR_UNSUPPORTED); eff_short and eff_long are 0.
 * Synchronises the stream. */
gp_status gp_boundary_demand_noalloc(gp_ctx* ctx, int32_t n, const gp_request* reqs,
                                     const void* q_cur_dev, gp_demand* out,
                                     int32_t* k_units);

/* gp_decide: per the configured policy (gp_policy above; GROWPAGE: Grow iff
 * Delta > tau, else Compress & Hold, Sec. 3.2).  Delta is compared as
 * delta = (sum_k_short - sum_k_long) / (num_candidates * num_units) in
 * double (for tau == 0 the Grow test is the exact integer one); under
 * GP_METRIC_ENTROPY as (eff_short - eff_long) / (num_candidates *
 * num_units), compared with tau in double.  P == 1
 * forces Grow; a Grow that would leave the pool at or below reserve_pages
 * (counting earlier grants of this call) becomes a fallback Compress
 * (Sec. 4.2, App. H.2).  Host only. */
gp_status gp_decide(gp_ctx* ctx, int32_t n, const gp_request* reqs,
                    const gp_demand* demand, gp_action* out);

/* gp_grow_page: Grow by One Page -- take the lowest free page (refcount 1)
 * and append it to req->block_table (num_pages + 1).  GP_ERR_NO_PAGES or a
 * full block table leave the request unchanged.  Host only. */
gp_status gp_grow_page(gp_ctx* ctx, gp_request* req);

/* Device-side errors of the asynchronous calls below (a failed check inside a
 * kernel, or a bounded wait that gave up) are reported by the next call that
 * synchronises with the engine -- gp_synchronize, gp_boundary_demand or an
 * inspection call -- as GP_ERR_INVALID or GP_ERR_TIMEOUT.  The host-side state
 * of the failed call (block tables, refcounts, the pool) was committed when it
 * returned GP_OK; the K/V rows of the units it was compacting are then
 * unspecified.  Errors found before the launch (arguments, GP_ERR_NO_PAGES, a
 * launch that fails) change nothing.
 *
 * gp_compress_hold: Compress & Hold for n requests, each of which must have
 * been passed to the last gp_boundary_demand with the same slot, pages and
 * block table (else GP_ERR_STATE).  Per (layer, KV head): importance
 * (Eq. 9), the recent R tokens always kept, block-local top-k_loc' with
 * k_loc' = min(k_loc, |B_j|, floor(K_t / P)) plus global top-(K_t - |S_loc|)
 * (Eq. 10, K_t = (P-1) b - R, equal scores: lower slot first), then stable
 * compaction: the k-th kept slot moves to logical slot k.  Copy-on-write
 * (App. E.2): every page with refcount > 1 is first replaced in the block
 * table by a fresh page (lowest id first, ascending logical order) and the
 * request's reference to the shared page is dropped after the copy.
 * num_pages is unchanged; logical slots [(P-1) b, P b) become free.
 * GP_ERR_NO_PAGES (not enough fresh pages for copy-on-write) changes
 * nothing.  Asynchronous on the stream. */
gp_status gp_compress_hold(gp_ctx* ctx, int32_t n, gp_request* reqs);

/* gp_shrink: Shrink (App. H.1, Eq. 13) for n requests prepared like those of
 * gp_compress_hold (a gp_boundary_demand on the same slot, pages and block
 * table): the same selection and copy-on-write as Compress & Hold, but with
 * K_t = (P-2) b - R, so two pages' worth of history is compacted into
 * logical slots [0, (P-2) b); the last page of the (new) block table is
 * then returned to the pool (its reference dropped) and num_pages becomes
 * P - 1, which leaves one page of free slots [(P-2) b, (P-1) b).  Needs
 * P >= 3 (else GP_ERR_INVALID).  GP_ERR_NO_PAGES (copy-on-write) changes
 * nothing.  Asynchronous on the stream. */
gp_status gp_shrink(gp_ctx* ctx, int32_t n, gp_request* reqs);

/* gp_compress_fill: Compress & Hold with hole-fill compaction -- NOT the
 * paper's compaction, an order-destroying variant that moves far fewer
 * bytes.  Selection and copy-on-write as gp_compress_hold (same keep
 * masks), but the kept slots of the first P-1 logical pages stay where they
 * are and the kept slots of the last page fill the holes (dropped slots of
 * the first P-1 pages): the k-th kept slot of the last page (ascending) goes
 * to the k-th hole (ascending).  Logical order and block locality are not
 * preserved; num_pages is unchanged and logical slots [(P-1) b, P b) become
 * free.  At most one page of rows moves per (layer, KV head).
 * Asynchronous on the stream. */
gp_status gp_compress_fill(gp_ctx* ctx, int32_t n, gp_request* reqs);

/* gp_compact_kv: the compaction step of Compress & Hold for a caller-given
 * index set (App. E.2), with the same copy-on-write handling.
 * keep_masks_dev: device uint32, per request [L][Hkv][ceil(P b / 32)] bit
 * masks (bit i%32 of word i/32 = keep slot i), requests concatenated in
 * order; each (layer, KV head) must keep exactly (P-1) b slots (else the
 * masks are rejected with GP_ERR_INVALID at the next synchronising call and
 * that unit is not moved).  Asynchronous. */
gp_status gp_compact_kv(gp_ctx* ctx, int32_t n, gp_request* reqs,
                        const uint32_t* keep_masks_dev);

/* gp_decode_attention: one layer of a decode step -- attention over each
 * request's paged cache with the summary update fused in, where the paper
 * integrates it (Sec. 4.1: the decode attention kernel updates the query
 * summaries in passing).  For request r and query head g (KV head g / G):
 *   the summaries of (layer, slot, g) are updated from the PRE-RoPE query q
 *   exactly as gp_update_summaries does (first_dev[r]: both set to q);
 *   z_i = RoPE_pos(q) . k_i / sqrt(d) over the first num_tokens[r] logical
 *   slots (keys are stored rotated, rotate-half at rope_theta), a =
 *   softmax(z), out[r][g] = sum_i a_i v_i.
 * q_dev: device [n][Hq][d] in q_dtype; first_dev: device uint8 [n];
 * num_tokens: HOST int32 [n], 0 <= num_tokens[r] <= num_pages * 256 (0 gives
 * a zero output); the cache slots past num_tokens[r] may hold any bits, NaN
 * and inf included: they do not reach the output.  out_dev: device fp32
 * [n][Hq][d], 4-byte aligned.  Requests need not be at a boundary.  bf16
 * caches with d = 128 and 2 or 4 query heads per KV head run on the
 * tensor-core kernel, everything else (or everything, under
 * gp_set_scan_kernel(CUDA_CORE)) on the CUDA-core one; both give the same
 * results within fp32 tolerances.  With a compaction pending on the side stream (see
 * gp_set_compaction_stream), the call makes the engine stream wait for it
 * only if one of its requests holds a page that compaction reads or writes;
 * otherwise the attention runs concurrently with it (App. E.3).
 * Asynchronous on the engine stream. */
gp_status gp_decode_attention(gp_ctx* ctx, int32_t layer, int32_t n, const gp_request* reqs,
                              const int32_t* num_tokens, const void* q_dev, const uint8_t* first_dev,
                              float* out_dev);

/* ---- asynchronous compaction (App. E.3: compaction overlapped with decoding)
 * gp_set_compaction_stream: from now on the compaction of gp_compress_hold,
 * gp_shrink, gp_compress_fill and gp_compact_kv runs on `stream` (a caller
 * CUDA stream; NULL: the engine stream again).  Each such call makes the
 * side stream wait for the work the engine stream holds at that point, then
 * returns without waiting for the compaction; the block tables and the page
 * pool are updated on the host as before.  While it runs, gp_update_summaries
 * (which touches no K/V), gp_decode_attention of requests that share no page
 * with it, and the caller's work on other streams may overlap it; every
 * later engine call that reads K/V or the engine's scratch (demand,
 * compaction, inspection, gp_stats, gp_synchronize, gp_destroy) first waits
 * for it on the host.  Before reading the compacted requests' K/V, the
 * caller makes its own stream wait with gp_wait_compaction.  The pages such
 * a call releases (shared pages replaced by copy-on-write, the page Shrink
 * returns) are back in the pool when it returns, while the side stream may
 * still read them: a caller that writes into a page the pool hands out
 * (gp_page_alloc, gp_grow_page) makes the writing stream wait with
 * gp_wait_compaction first.  Waits for a pending compaction first. */
gp_status gp_set_compaction_stream(gp_ctx* ctx, void* stream);
/* gp_wait_compaction: `stream` (NULL: the engine stream) waits for the last
 * compaction launched on the side stream (no-op if none ever was).  It
 * enqueues the wait and returns at once. */
gp_status gp_wait_compaction(gp_ctx* ctx, void* stream);

/* ---- inspection (tests, benchmarks) ---------------------------------------
 * All of these synchronise the stream.  req_idx indexes the request list of
 * the last gp_boundary_demand (k, probabilities, scores) or of the last
 * gp_compress_hold (keep masks). */

/* K^S, K^L per unit: k_out host int32[L * Hkv * 2] ([unit][x]). */
gp_status gp_debug_demand_k(gp_ctx* ctx, int32_t req_idx, int32_t* k_out);
/* Importance log2 max(a^S, a^L) over [0, P b - R): host float[L*Hkv][P b - R]. */
gp_status gp_debug_scores(gp_ctx* ctx, int32_t req_idx, float* out);
/* Demand distributions a^S, a^L over C_t: host float[L*Hkv][2][(P-1) b]
 * (the kernels keep them for the D_p select of every demand call). */
gp_status gp_debug_probs(gp_ctx* ctx, int32_t req_idx, float* out);
/* Keep masks of the last gp_compress_hold: host uint32[L*Hkv][ceil(P b/32)]. */
gp_status gp_debug_keep_mask(gp_ctx* ctx, int32_t req_idx, uint32_t* out);
/* Effective support sizes exp(H(a^S)), exp(H(a^L)) per unit of the last
 * demand call: host double[L * Hkv * 2] ([unit][x]).  GP_ERR_STATE unless
 * the context's demand_metric is GP_METRIC_ENTROPY. */
gp_status gp_debug_entropy(gp_ctx* ctx, int32_t req_idx, double* out);
/* Summaries of one slot: host double[L][2][Hq][d]. */
gp_status gp_read_summaries(gp_ctx* ctx, int32_t slot, double* out);

/* gp_synchronize: waits for every piece of engine work (the engine stream,
 * the speculative selection, a side-stream compaction) and reports the
 * device-side errors of earlier asynchronous calls: GP_ERR_TIMEOUT if only
 * bounded waits gave up, GP_ERR_INVALID if a device-side check failed (the
 * text names the error bits), GP_OK otherwise.  The error word is cleared. */
gp_status gp_synchronize(gp_ctx* ctx);

/* gp_debug_attention_plan: the work split gp_decode_attention gives the
 * tensor-core attention kernel for n requests attending to num_tokens[r]
 * tokens on a device of `sms` SMs, computed on the host without launching
 * anything (also on a host-only context).  Every (request, KV head) pair's
 * attended pages are laid end to end and cut into one even range per SM;
 * each range's pieces are one CTA's items.  items_out: host int32
 * [max_items][8], per item (request, KV head, piece, pieces of the pair,
 * first page, tiles of 128 keys, first item of the pair, CTA), items of a
 * CTA consecutive and CTAs in order.  *n_items, *n_ctas: the counts (set
 * also when max_items is too small, which returns GP_ERR_INVALID).  Host
 * only. */
gp_status gp_debug_attention_plan(gp_ctx* ctx, int32_t n, const int32_t* num_tokens, int32_t sms,
                                  int32_t max_items, int32_t* items_out, int32_t* n_items, int32_t* n_ctas);

/* ---- test hooks -------------------------------------------------------------
 * gp_debug_set_wait_limit: the limit, in SM clock cycles, of the bounded copy
 * waits of later launches of `kernel` (GP_KERNEL_COMPRESS: the compaction;
 * GP_KERNEL_SELECT: the speculative selection); 0 makes each such wait give
 * up at once, a negative value restores the default of 2^31 (about one
 * second).  A wait that gives up makes its CTA wait for the copies it already
 * issued (always with the default limit), record a timeout and return;
 * gp_synchronize then reports GP_ERR_TIMEOUT.  Other kernels:
 * GP_ERR_UNSUPPORTED.  Host only; for tests of the timeout path.
 * gp_debug_fail_next_launch: the next launch of `kernel` (GP_KERNEL_*) fails
 * without running, as a failed launch would (GP_ERR_CUDA); -1 clears it.
 * Host only; for tests of the rollback paths. */
gp_status gp_debug_set_wait_limit(gp_ctx* ctx, int32_t kernel, int64_t cycles);
gp_status gp_debug_fail_next_launch(gp_ctx* ctx, int32_t kernel);

/* Which kernels do the cache-wide contractions: the scan of
 * gp_boundary_demand and the scores and weighted values of
 * gp_decode_attention.  AUTO (default): the tensor-core (tcgen05) kernels
 * where they apply -- the scan for bf16 caches (every request length up to
 * the 256-page block-table limit), attention for bf16 caches with d = 128
 * and 2 or 4 query heads per KV head -- and the CUDA-core (fp32 FMA)
 * kernels otherwise: fp32 caches, other attention shapes, or a K or V cache
 * no tensor map can describe (base not 16-byte aligned, or 2^31 or more key
 * rows).  CUDA_CORE forces the latter everywhere; TENSOR_CORE makes calls the
 * tensor-core kernels cannot serve fail with GP_ERR_UNSUPPORTED.  Both give
 * the same results within the tolerances of fp32 arithmetic.  Host only. */
#define GP_SCAN_AUTO 0
#define GP_SCAN_CUDA_CORE 1
#define GP_SCAN_TENSOR_CORE 2
gp_status gp_set_scan_kernel(gp_ctx* ctx, int32_t kind);

/* Where Compress & Hold's Eq. 10 selection runs (Sec. 3.3).  SPECULATIVE:
 * after every gp_boundary_demand, on an engine-owned stream, while the host
 * reads the sums and decides, so that a following Compress & Hold (or hole
 * fill) only moves rows.  IN_COMPACTION: at the head of each (layer, KV
 * head) unit's compaction CTA, where the copies of the other units' CTAs
 * keep HBM busy.  AUTO (default): speculative for demand calls of at most
 * 4 x (SM count) units that Compress & Hold could take, in the compaction
 * above that.  The keep masks are the same either way.  Host only. */
#define GP_SELECT_AUTO 0
#define GP_SELECT_SPECULATIVE 1
#define GP_SELECT_IN_COMPACTION 2
gp_status gp_set_selection_mode(gp_ctx* ctx, int32_t mode);

/* Per-kernel device time: when enabled, every kernel launch is bracketed by
 * CUDA events on the engine stream.  names: GP_KERNEL_* below.  The query
 * synchronises and returns the summed milliseconds and launch count since
 * the last reset. */
#define GP_KERNEL_EMA 0
#define GP_KERNEL_PREP 1
#define GP_KERNEL_DEMAND 2
#define GP_KERNEL_COMPRESS 3
#define GP_KERNEL_ATTENTION 4
#define GP_KERNEL_SELECT 5
#define GP_KERNEL_ENTROPY 6
#define GP_KERNEL_COUNT 7
gp_status gp_set_timing(gp_ctx* ctx, int32_t enabled);
gp_status gp_kernel_time(gp_ctx* ctx, int32_t kernel, double* ms, int64_t* launches);
gp_status gp_reset_timing(gp_ctx* ctx);

gp_status gp_stats(const gp_ctx* ctx, gp_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* GROWPAGE_H */
