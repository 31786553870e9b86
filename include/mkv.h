/*
 * mkv.h -- C ABI of the mixed-format paged decode-attention library
 * (GB300 / sm_103a).
 *
 * What it implements
 * ------------------
 * The decode hot path of "Minima-KV: Retention-Preserving KV Cache
 * Compression with Mixed-Format Paged Attention" (arXiv 2608.23834).  From
 * the abstract (mlsanity.com paper page): Recent and protected Anchor pages
 * remain in FP8, older non-anchor pages move to packed TQ3, every
 * live-request page remains addressable, and format-specific kernels compute
 * partial attention states that a globally normalised online-softmax merge
 * combines, so decode runs over the heterogeneous cache without a cache-sized
 * dense shadow.  The setupai.cc summary ("Technical Deep Dive") adds that the
 * mixed formats share PagedAttention's block structure and that TQ3 is a
 * 3-bit format.
 *
 * Calls: mkv_pool_create (page pool + page table + tier tags),
 * mkv_append_tokens (FP8 quantise into the tail page), mkv_demote_pages
 * (FP8 -> TQ3 repack), mkv_decode_attention (FP8 partials + TQ3 partials +
 * LSE merge).  Beyond the pages: mkv_append_decode (append fused into the
 * decode kernel), mkv_decode_attention_multi (several causal query tokens
 * per request), mkv_decode_attention_noalloc, mkv_dequantize_pages (dense
 * export), plan inspection, and failure-detection hooks
 * (mkv_check_device_errors, mkv_selftest_wait_timeout, mkv_inject_plan_slot).
 * Every step runs in this library's CUDA kernels; there is no CPU or dense
 * fallback.
 *
 * ============================================================ Storage formats
 * The pages name FP8 and TQ3 but define neither; this section is the
 * library's definition.  Notation: d = head_dim (256), P = page_size (a
 * multiple of 16), a "row" = one token, one kv head, K or V.
 *
 * FP8 row (Recent, Anchor): E4M3 "fn" codes (OCP FP8; bias 7, max 448, no
 * infinities) plus one IEEE fp16 scale per row:
 *     s      = fp16_rn( fp32_rn( max_i |x_i| / 448 ) )
 *     code_i = e4m3_rn_satfinite( fp32_rn( x_i / s ) )   (all +0 when s == 0)
 *     x_hat_i = value(code_i) * s                         (exact in fp32)
 * Inputs x are fp32 or bf16; divisions are IEEE fp32 round-to-nearest-even.
 *
 * TQ3 row (Stale): produced from the FP8-dequantised row x_hat by
 *     y     = R x_hat,  R = H_d D / sqrt(d)
 *             H_d: Sylvester Hadamard matrix, natural order;
 *             D = diag(sign_i): sign_i = -1 iff bit (i mod 64) of output
 *             floor(i/64) of SplitMix64(rotation_seed) is 1 (signs first,
 *             then H; the same R for K and V, all layers and heads)
 *     sigma = fp16_rn( ||x_hat||_2 / sqrt(d) )
 *     u_i   = y_i / sigma  (0 when sigma == 0)
 *     code_i = #{k in 1..7 : tau_k <= u_i}          (0..7, ties to upper)
 *     x_tilde = R^T ( sigma * L[code] )
 * Codebook: L_k = fp16_rn(c_k), c_0 < ... < c_7 the 8-level Lloyd-Max
 * quantiser of N(0,1) (fp64 fixed point); tau_k = (L_{k-1} + L_k) / 2
 * (exact).  mkv_tq3_codebook() returns the values.
 *
 * Page layout: one (layer, slot) page holds P tokens.  For kv head
 * h = 0..H_kv-1 in order: a K plane, then a V plane.  A plane is the code
 * bytes followed by P little-endian fp16 scales in token order.
 *   FP8 plane codes (P*d bytes):
 *     K: byte t*d + j                      (row-major)
 *     V: byte (t/2)*2d + 2j + (t%2)        (rows of a token pair interleaved)
 *   TQ3 plane codes (P*3d/8 bytes, 3 bits per code): 12-byte units of
 *   32 codes = three little-endian 32-bit words W0, W1, W2:
 *     bits [4i, 4i+3) of W_k = code (8k + i)           i = 0..7, k = 0..2
 *     bit  4i+3       of W_k = bit k of code (24 + i)
 *     K: unit t*(d/32) + j/32, code j%32
 *     V: unit (t/2)*(d/16) + j/16, code 2*(j%16) + (t%2)
 * Sizes per page, d = 256, 4 kv heads: FP8 P*2064 B (132,096 at P = 64),
 * TQ3 P*784 B (50,176 at P = 64); slot s of layer l is at
 * arena + (l * slots + s) * page_bytes.
 *
 * ============================================================ Attention
 * For a request of length n, query head h (kv head floor(h/G), G =
 * H_q/H_kv): s_t = q_h . k_t / sqrt(d) over all n tokens (FP8 or TQ3
 * dequantised per the page's tier), out = sum_t softmax(s)_t v_t (fp32),
 * lse = ln sum_t exp(s_t) (fp32).  TQ3 pages are scored in the rotated
 * domain with q' = R q and their output is rotated back once (R^T) after
 * the TQ3 partials are merged.
 *
 * ============================================================ Conventions
 * Ownership: every device buffer (pool memory, q, k, v, out, lse) belongs to
 * the caller; the pool keeps non-owning pointers into device_buf, which must
 * outlive it.  Host arrays are read only during the call.
 * Streams: GPU work is enqueued on the stream passed in (NULL = legacy default
 * stream); calls return without waiting unless stated.  Slots freed by
 * demotion or release are reused in stream order, so a pool must be driven
 * from one stream (or the caller orders its streams).
 * Errors: every call returns an mkv_status; no C++ exception crosses the ABI;
 * mkv_last_error() gives a thread-local message.  A failing call changes no
 * pool state.  Non-finite inputs are undefined behaviour (not checked).
 * Threads: a pool is not thread-safe.
 */
#ifndef MKV_H_
#define MKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (CUDA runtime) / CUstream (driver). */
typedef struct CUstream_st* mkv_stream_t;

typedef enum {
  MKV_OK = 0,
  MKV_ERR_INVALID_ARGUMENT = 1, /* bad pointer, id, shape, dtype or range */
  MKV_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. d != 256) */
  MKV_ERR_OUT_OF_PAGES = 3,     /* no free slot in the needed arena */
  MKV_ERR_INVALID_STATE = 4,    /* illegal tier transition or page state */
  MKV_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
  MKV_ERR_DEVICE_CHECK = 6,     /* a kernel reported a failed check or timeout */
  MKV_ERR_CAPACITY = 7          /* a per-call limit of the pool was exceeded */
} mkv_status;

/* Tier tags (the pages' three-tier hierarchy R / A / S).  R and A pages are
 * FP8, S pages are TQ3. */
typedef enum {
  MKV_TIER_NONE = 0,
  MKV_TIER_RECENT = 1,
  MKV_TIER_ANCHOR = 2,
  MKV_TIER_STALE = 3
} mkv_tier;

typedef enum { MKV_F32 = 0, MKV_BF16 = 1 } mkv_dtype;

/* mkv_pool_config.flags */
#define MKV_POOL_HOST_ONLY 1 /* bookkeeping only: no device memory is touched and
                                GPU calls validate, update state and skip the
                                launch (used by host-logic tests) */

typedef struct {
  int32_t num_layers;        /* layers sharing one page table */
  int32_t num_q_heads;       /* H_q */
  int32_t num_kv_heads;      /* H_kv; G = H_q / H_kv must be 1..8 */
  int32_t head_dim;          /* d; the kernels support 256 */
  int32_t page_size;         /* P tokens per page: 64 or 128 */
  int32_t fp8_slots;         /* FP8 arena capacity in pages (per layer) */
  int32_t tq3_slots;         /* TQ3 arena capacity in pages (per layer) */
  int32_t max_seqs;          /* sequence ids are 0..max_seqs-1 */
  int32_t max_pages_per_seq; /* longest sequence = this * page_size tokens */
  int32_t max_batch;         /* most sequences in one decode/append call (0: max_seqs) */
  int32_t flags;             /* MKV_POOL_* */
  int32_t reserved;          /* must be 0 */
  uint64_t rotation_seed;    /* SplitMix64 seed of the TQ3 rotation signs */
} mkv_pool_config;

typedef struct mkv_pool mkv_pool;

typedef struct {
  int64_t recent_pages, anchor_pages, stale_pages; /* live logical pages per tier */
  int64_t live_tokens;                             /* sum of sequence lengths */
  int64_t fp8_bytes, tq3_bytes;                    /* live page bytes, all layers */
  double kv_bytes_per_live_token;                  /* (fp8+tq3 bytes) / live tokens */
  int32_t fp8_slots_free, tq3_slots_free;
  int64_t device_bytes;                            /* size of the pool's device buffer */
  int64_t workspace_bytes;                         /* partial-state workspace inside it */
} mkv_stats;

/* ---------------------------------------------------------------- pool */

/* Bytes of device memory a pool with this config needs (arenas, page-table
 * and plan regions, partial-state workspace).  No device access. */
mkv_status mkv_pool_required_bytes(const mkv_pool_config* cfg, size_t* device_bytes);

/* Create a pool over the caller's device buffer (>= required bytes, 256-byte
 * aligned; may be NULL with MKV_POOL_HOST_ONLY).  Zero-fills the FP8 arena on
 * `stream` so every stored byte is a finite FP8 value.  *out receives the
 * handle.  Pages: the paged cache extends PagedAttention ("PagedAttention
 * Integration", setupai.cc "Technical Deep Dive"). */
mkv_status mkv_pool_create(const mkv_pool_config* cfg, void* device_buf, size_t bytes,
                           mkv_stream_t stream, mkv_pool** out);

/* Destroy the handle (host memory only; the device buffer stays the caller's).
 * The caller must make sure no work that uses the pool is still running. */
mkv_status mkv_pool_destroy(mkv_pool* pool);

/* ---------------------------------------------------------------- sequences */

/* Host bookkeeping: sequence seq_ids[i] grows by n_new[i] >= 0 tokens; every
 * page it opens takes a free FP8 slot and is tagged RECENT.  All-or-nothing:
 * MKV_ERR_OUT_OF_PAGES (or a bad id / length past max_pages_per_seq) leaves
 * every sequence unchanged.  The caller then writes the new tokens of every
 * layer with mkv_append_tokens before they are attended to. */
mkv_status mkv_seq_extend(mkv_pool* pool, int32_t n, const int32_t* seq_ids, const int32_t* n_new);

/* Drop a sequence: its slots return to the free lists (reused in stream
 * order) and its length becomes 0. */
mkv_status mkv_seq_release(mkv_pool* pool, int32_t seq);

/* Length in tokens and number of pages of a sequence. */
mkv_status mkv_seq_info(const mkv_pool* pool, int32_t seq, int32_t* length, int32_t* num_pages);

/* Tier and physical slot of logical page `page` of `seq`. */
mkv_status mkv_page_info(const mkv_pool* pool, int32_t seq, int32_t page, mkv_tier* tier,
                         int32_t* slot);

/* ---------------------------------------------------------------- write path */

/* FP8 append / quantise (Recent pages stay in FP8: abstract, mlsanity.com).
 * For layer `layer`, write the last n_new[i] tokens of each sequence
 * seq_ids[i] (the tokens the preceding mkv_seq_extend added).  k, v: device
 * arrays [sum_i n_new[i], H_kv, d] of `dtype`, rows in call order.
 * Each row is quantised as "FP8 row" above into its page.  Enqueued on
 * `stream`.  Errors: INVALID_ARGUMENT (ids, layer, dtype, n_new larger than
 * the sequence), INVALID_STATE (a target page is not FP8). */
mkv_status mkv_append_tokens(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids,
                             const int32_t* n_new, const void* k, const void* v, mkv_dtype dtype,
                             mkv_stream_t stream);

/* Re-tag an FP8 page: MKV_TIER_ANCHOR protects it from demotion ("protected
 * Anchor pages remain in FP8", abstract), MKV_TIER_RECENT unprotects it.
 * INVALID_STATE for a TQ3 page or for MKV_TIER_STALE (use demotion). */
mkv_status mkv_set_tier(mkv_pool* pool, int32_t seq, int32_t page, mkv_tier tier);

/* FP8 -> TQ3 demotion ("older non-anchor pages move to packed TQ3",
 * abstract): for each (seq_ids[i], pages[i]), re-encode the page of every
 * layer as "TQ3 row" above into a fresh TQ3 slot, tag it STALE and free its
 * FP8 slot (stream-ordered reuse).  All-or-nothing checks first:
 * INVALID_STATE for an Anchor page, a TQ3 page, a partial (not full) page or
 * a page listed twice; OUT_OF_PAGES when the TQ3 arena is short. */
mkv_status mkv_demote_pages(mkv_pool* pool, int32_t n, const int32_t* seq_ids, const int32_t* pages,
                            mkv_stream_t stream);

/* ---------------------------------------------------------------- decode */

/* Mixed-format decode attention for one layer ("Format-specific kernels
 * compute partial attention states and combine them through a globally
 * normalized online-softmax merge", abstract).  q: device [n, H_q, d] of
 * `dtype`; out: device fp32 [n, H_q, d]; lse: device fp32 [n, H_q] (natural
 * log).  Attends over all tokens of each sequence (length >= 1).
 * Workspace use is O(#splits x H_q x d), independent of context length.
 * Errors: INVALID_ARGUMENT (n > max_batch, empty sequence, repeated id,
 * layer, dtype, NULL pointers). */
mkv_status mkv_decode_attention(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids,
                                const void* q, mkv_dtype dtype, float* out, float* lse,
                                mkv_stream_t stream);

/* Several query tokens per request over the mixed-format cache (chunked
 * prefill, or verifying speculative tokens).  The pages describe one query
 * token per step; this call extends the same attention, partial states and
 * merge causally: the last nq tokens of each sequence (already appended, so
 * the sequence holds len >= nq tokens) are the queries, and query token i
 * (position len - nq + i) attends to tokens 0 .. len - nq + i: the
 * attention of mkv_decode_attention run nq times over the growing prefix
 * (bit-identical to it for nq = 1; within rounding for nq >= 2).
 * q: device [n, nq, H_q, d] of `dtype`; out: device fp32 [n, nq, H_q, d];
 * lse: device fp32 [n, nq, H_q].  The pages that hold the query tokens must
 * be FP8 (they are the newest, so Recent).  With nq >= 2 the query tokens
 * go in pairs: the plan holds n * ceil(nq / 2) batch entries, entry
 * b * ceil(nq / 2) + j reading request b's prefix up to its query token
 * min(2j + 1, nq - 1) for query tokens 2j and 2j + 1 together (each block is
 * dequantised once for both; token 2j masks the prefix's last token).
 * Errors: those of mkv_decode_attention; INVALID_ARGUMENT for
 * nq < 1, n * nq > max_batch or a sequence shorter than nq; INVALID_STATE
 * when a query token sits in a TQ3 page. */
mkv_status mkv_decode_attention_multi(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids,
                                      int32_t nq, const void* q, mkv_dtype dtype, float* out, float* lse,
                                      mkv_stream_t stream);

/* One decode step of one layer: append each sequence's newest token (FP8,
 * as mkv_append_tokens with n_new = 1) and run mixed-format decode attention
 * over all its tokens (as mkv_decode_attention), in one call and one kernel
 * launch fewer (the append runs inside the partial-attention kernel).  The
 * newest token must already be counted by mkv_seq_extend and sit in an FP8
 * page.  k, v: device [n, H_kv, d] of kv_dtype (row i is seq_ids[i]'s token);
 * q, out, lse as in mkv_decode_attention.  Errors: those of the two calls. */
mkv_status mkv_append_decode(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids, const void* k,
                             const void* v, mkv_dtype kv_dtype, const void* q, mkv_dtype q_dtype, float* out,
                             float* lse, mkv_stream_t stream);

/* Materialising export: dequantise pages [page0, page0 + npages) of one
 * sequence and layer into dense rows -- the "materializing quality profile"
 * of the pages (abstract, mlsanity.com) as a debugging and quality tool, not
 * part of decode.  FP8 rows give x_hat (exact), TQ3 rows x_tilde = R^T (sigma
 * L[code]) (fp32 FWHT).  k_out, v_out: device [npages * P, H_kv, d] of
 * out_dtype (MKV_F32 or MKV_BF16, round-to-nearest-even); token slots past
 * the sequence length are written as 0.  Enqueued on `stream`. */
mkv_status mkv_dequantize_pages(mkv_pool* pool, int32_t layer, int32_t seq, int32_t page0, int32_t npages,
                                void* k_out, void* v_out, mkv_dtype out_dtype, mkv_stream_t stream);

/* ---------------------------------------------------------------- inspection */

/* Live pages and bytes per tier and KV bytes per live token (the pages'
 * deployment accounting, abstract: 18.3 KiB per live token on their model). */
mkv_status mkv_pool_stats(const mkv_pool* pool, mkv_stats* stats);

/* Copy the raw bytes of one (layer, seq, page) into host_dst (cap bytes
 * available; needs the page size of its tier).  Synchronises `stream`.
 * *tier and *n_valid (tokens written) are filled when non-NULL. */
mkv_status mkv_export_page(mkv_pool* pool, int32_t layer, int32_t seq, int32_t page, void* host_dst,
                           size_t cap, mkv_tier* tier, int32_t* n_valid, mkv_stream_t stream);

/* The pool's rotation signs (d entries, +1 / -1). */
mkv_status mkv_rotation_signs(const mkv_pool* pool, int8_t* host_dst, int32_t cap);

/* The stored TQ3 codebook: levels[8] (fp16 values, ascending) and
 * thresholds[7].  Library constant, computed at load time by the library's
 * own Lloyd-Max iteration. */
mkv_status mkv_tq3_codebook(float* levels8, float* thresholds7);

/* Decode plan for a batch (host only, no device access): the number of
 * partial-state splits the decode kernels would use, and per split 9 ints
 * {batch index, kv head, tier (1 = FP8, 3 = TQ3), first page entry, page
 * count, tokens, CTA, first block, blocks}, CTA by CTA.  Blocks are counted
 * within the split's (request, kv head, tier) group: 16 FP8 or 32 TQ3 tokens
 * each, page by page, so two consecutive splits may share one page.
 * chunks (cap splits of 9 ints) may be NULL to query the count. */
mkv_status mkv_plan_decode(mkv_pool* pool, int32_t n, const int32_t* seq_ids, int32_t* chunks,
                           int32_t cap, int32_t* n_chunks);

/* The same for mkv_decode_attention_multi with nq query tokens per request:
 * with nq = 1 the decode plan; with nq >= 2 split records use batch index
 * b * ceil(nq / 2) + j for query tokens 2j and 2j + 1 of request b (the
 * prefix up to query token min(2j + 1, nq - 1)).  Errors: those of
 * mkv_decode_attention_multi. */
mkv_status mkv_plan_decode_multi(mkv_pool* pool, int32_t n, const int32_t* seq_ids, int32_t nq, int32_t* chunks,
                                 int32_t cap, int32_t* n_chunks);

/* Synchronise `stream` and report (and clear) the pool's device error word:
 * MKV_ERR_DEVICE_CHECK if a kernel flagged a failed check or a bounded wait
 * that ran out. */
mkv_status mkv_check_device_errors(mkv_pool* pool, mkv_stream_t stream);

/* Failure-detection self-test (not from the pages).  Enqueues on `stream` a
 * one-CTA kernel that waits on an mbarrier nothing arrives on, with the
 * decode kernel's rule for a wait that runs out: after limit_cycles SM clocks
 * (1 .. 4e9; 2e6 is about 1 ms) it records the timeout bit in the pool's
 * device error word and returns.  The next mkv_check_device_errors then
 * reports MKV_ERR_DEVICE_CHECK and clears the word; the CUDA context and the
 * pool stay usable.  Nothing faults, traps or spins without a bound.
 * Errors: INVALID_ARGUMENT (limit), UNSUPPORTED on a host-only pool. */
mkv_status mkv_selftest_wait_timeout(mkv_pool* pool, int64_t limit_cycles, mkv_stream_t stream);

/* Fault injection for tests (not from the pages): overwrite the physical slot
 * of page entry `entry` of the device copy of the current decode plan, the
 * one the last decode call planned, with `slot`.  The next decode call with
 * the same batch reuses that plan (mkv_append_decode, which writes through
 * the plan's slots, always plans again).  The decode kernel checks every slot
 * before it copies a block: a slot outside the arena skips the copy, stops
 * the CTA's remaining work and sets the error word, so the call's outputs
 * are undefined and the next mkv_check_device_errors reports
 * MKV_ERR_DEVICE_CHECK.  Nothing faults.  Any later change to the pool, or
 * another batch, plans again from the host tables.  Synchronises `stream`.
 * Errors: INVALID_ARGUMENT (entry), INVALID_STATE (no current plan),
 * UNSUPPORTED on a host-only pool. */
mkv_status mkv_inject_plan_slot(mkv_pool* pool, int32_t entry, int32_t slot, mkv_stream_t stream);

/* Instrumentation: when `start` / `stop` (cudaEvent_t handles owned by the
 * caller) are non-NULL, the next mkv_decode_attention call records `start`
 * right before its partial-attention kernel and `stop` right after it, on the
 * call's stream, then forgets them.  Lets a caller time that kernel alone. */
mkv_status mkv_set_timing_events(mkv_pool* pool, void* start, void* stop);

/* Decode attention that allocates nothing (no counterpart in the paper; this
 * is a convenience of this library).  Same arguments, result and errors as
 * mkv_decode_attention, but the partial-state scratch of the call lives in a
 * fixed 8 MiB array compiled into the library (a file-scope __device__ array
 * that every GPU using the library holds until the process exits) instead of
 * the pool's workspace.  It is meant for callers that may not allocate device
 * memory at call time -- for example code running under a framework whose
 * caching allocator owns the whole device, or code that must not trigger a
 * cudaMalloc in the middle of a step -- and it calls no cudaMalloc, cudaFree
 * or other allocating routine.
 * Limit: splits x G x (2 + d) x 4 bytes of partial states must fit in 8 MiB
 * (1,354 splits at G = 6, d = 256); larger batches return MKV_ERR_CAPACITY
 * and launch nothing.  The size is known only once the batch is planned, so
 * a refused call leaves the pool's plan for these ids built and its upload
 * enqueued on the stream, as a mkv_decode_attention call would.
 * Device: the call must be made with the pool's device current (else
 * MKV_ERR_INVALID_ARGUMENT).  Every call looks the array's address up for
 * that device (cudaGetSymbolAddress; the first lookup in a process may load
 * the library's device code, so make the first call before any stream
 * capture).  All calls share the one array, which keeps the
 * last call's contents; nothing in it needs to start at zero (every partial
 * state is written in full before it is read).  Calls whose GPU work
 * overlaps -- on different streams, or from different pools -- race on the
 * array and must be ordered by the caller. */
mkv_status mkv_decode_attention_noalloc(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids,
                                        const void* q, mkv_dtype dtype, float* out, float* lse,
                                        mkv_stream_t stream);

/* Page relevance: for each request b of `seq_ids` and each of its pages j,
 *   mass[b * mass_stride + j] = (1 / Hq) sum_h sum_{t in page j}
 *                               exp(q_h . k_t / sqrt(d) - lse_h),
 * the softmax weight the page's tokens receive, averaged over the query
 * heads (kv head floor(h/G); TQ3 pages scored in the rotated domain).  The
 * pages protect Anchor pages by "age and relevance" (insight.aitobox.com
 * post, "执行摘要") without defining relevance; this attention mass is the
 * library's definition, the signal of a relevance-based Anchor policy.
 * q: [n, Hq, d] device (dtype), the query of a decode step of `layer`;
 * lse: [n, Hq] fp32 device, that decode call's lse for the same q (so a
 * request's masses sum to 1 up to rounding).  mass: [n, mass_stride] fp32
 * device; entries past a sequence's page count are left untouched;
 * mass_stride >= the longest sequence's page count (else
 * INVALID_ARGUMENT).  Reads K only; one 128-thread block per page.  Async on
 * `stream`; shares the demotion staging region, so a later mkv_demote_pages
 * on another stream must be ordered by the caller. */
mkv_status mkv_page_relevance(mkv_pool* pool, int32_t layer, int32_t n, const int32_t* seq_ids, const void* q,
                              mkv_dtype q_dtype, const float* lse, float* mass, int32_t mass_stride,
                              mkv_stream_t stream);

/* ------------------------------------------------------------ step graph
 * One decode step over every layer as a single CUDA graph launch.  The
 * pages describe one query token per request and step, attended over the
 * whole paged cache layer by layer (Minima-KV abstract, mlsanity.com paper
 * page); a serving loop repeats exactly that launch sequence every step, so
 * it can be recorded once and replayed.  The graph holds, for each layer l in
 * order, what mkv_append_decode (k, v given) or mkv_decode_attention (k, v
 * NULL) would enqueue: the partial-attention kernel (with the fused append)
 * and the LSE merge.
 *
 * mkv_step_graph_create: records the graph for the batch `seq_ids[0..n)` on
 * caller-owned device buffers that stay fixed for the graph's life, one per
 * layer (arrays of num_layers pointers): q[l] [n, Hq, d] (q_dtype), k[l],
 * v[l] [n, Hkv, d] (kv_dtype) or k = v = NULL, out[l] [n, Hq, d] fp32,
 * lse[l] [n, Hq] fp32.  Plans the batch and uploads the plan on `stream`;
 * the recording itself runs on a private stream and executes nothing.
 * The kernels read their per-CTA piece ranges from the pool's device plan,
 * so one recording serves every later plan of the same batch.  Errors: as
 * mkv_append_decode / mkv_decode_attention, plus MKV_ERR_UNSUPPORTED on a
 * host-only pool and MKV_ERR_CUDA when capture or instantiation fails.
 *
 * mkv_step_graph_launch: one step.  The caller first writes the step's
 * inputs into the fixed buffers and makes the pool's host updates
 * (mkv_seq_extend, mkv_demote_pages) as for the per-layer calls.  The call
 * re-plans if the pool changed (host work, then an upload in stream order)
 * and launches the graph on `stream`; asynchronous like the per-layer calls.
 * The batch must still be valid (same ids, none released).
 *
 * mkv_step_graph_destroy: frees the graph (not the buffers).  A pool must
 * outlive its graphs. */
typedef struct mkv_step_graph mkv_step_graph;
mkv_status mkv_step_graph_create(mkv_pool* pool, int32_t n, const int32_t* seq_ids, const void* const* q,
                                 const void* const* k, const void* const* v, mkv_dtype q_dtype, mkv_dtype kv_dtype,
                                 float* const* out, float* const* lse, mkv_stream_t stream, mkv_step_graph** graph);
mkv_status mkv_step_graph_launch(mkv_step_graph* graph, mkv_stream_t stream);
mkv_status mkv_step_graph_destroy(mkv_step_graph* graph);

/* Thread-local text of the last error (never NULL). */
const char* mkv_last_error(void);

/* Library version string. */
const char* mkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MKV_H_ */
