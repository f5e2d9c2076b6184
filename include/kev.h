/*
 * kev.h -- C ABI of libkev: packed, question-isolated attention on one GB300 (sm_103a).
 *
 * N questions are packed into one token sequence of T tokens.  Question i owns the
 * half-open interval [begin_i, end_i) of packed positions.  Prefill attention is causal
 * AND block diagonal: token t of question i attends to token u iff u lies in the same
 * interval and u <= t (Kev architecture article, icman.com.cn news 75864, §2.1 end and
 * §2.3; Kev pipeline article, gsyq.cn news 368355, §2.2 "visible domain").  Each
 * question's K/V rows go into its own slot of a preallocated pool (Kev pipeline article,
 * §2.2 "KV cache slot pool").  A decode step appends one K/V row per live question and
 * attends over its whole slot (inference-engine notes, sakurs2.com, §2.2); questions that
 * stopped early are dropped from the step (Kev pipeline article, §1.2, §2.3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is caller-owned DEVICE memory, contiguous, 16-byte aligned.
 *    The library allocates nothing and keeps no mutable global state (the one exception is
 *    the fixed scratch of kev_decode_attn_static, below), so calls on different streams
 *    with different buffers are independent.  The cache is passed in
 *    and out as an argument, never held by the library (KV-cache isolation article,
 *    hnwysp.cn news 130224, §3.3 and §4.3).
 *  - Everything is enqueued on `stream`; no entry point synchronises the host except
 *    kev_read_status.
 *  - Layouts (row-major, last index fastest):
 *        q        [T, H_q, d]          out  [T, H_q, d]
 *        k, v     [T, H_kv, d]
 *        pool_k, pool_v  [n_slots, H_kv, slot_cap, d]
 *        q_new [N, H_q, d], k_new/v_new [N, H_kv, d], decode out [N, H_q, d]
 *    q-head h reads kv-head h / (H_q / H_kv) (grouped-query attention).
 *  - Element type: KEV_BF16 (bf16 storage, fp32 accumulation, bf16 output rounded to
 *    nearest even) or KEV_FP32 (fp32 storage and arithmetic, no TF32).
 *    Supported head dims: bf16 d in {64, 128} (tensor cores); fp32 any d that is a multiple of 16
 *    from 16 to 256 (CUDA cores); the RoPE entry points take d in {64, 128}.  H_q must be a
 *    multiple of H_kv, G = H_q/H_kv <= 16.
 *  - Errors.  Arguments the host can check (null or misaligned pointers, negative sizes,
 *    unsupported shapes, too small a workspace) are returned at once and nothing is
 *    launched.  Data-dependent errors (intervals, slot ids, lengths) are found on the
 *    device before anything is written: the call's kernels then write nothing, and the
 *    code is stored in *dev_status (if dev_status is not NULL) in stream order.
 *    kev_read_status turns it into a kev_status.
 *  - Scale: kev_attn_shape.scale == 0 means 1/sqrt(d).
 *  - A call takes at most KEV_MAX_QUESTIONS questions (else KEV_ERR_UNSUPPORTED).
 */
#ifndef KEV_H
#define KEV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KEV_MAX_QUESTIONS 4096

typedef struct CUstream_st* kev_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  KEV_OK = 0,
  KEV_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, negative size, workspace too small */
  KEV_ERR_UNSUPPORTED = 2,   /* dtype, head dim or group size this library does not implement */
  KEV_ERR_INTERVALS = 3,     /* (device) an interval is reversed, outside [0,T] or overlaps another */
  KEV_ERR_SLOT = 4,          /* (device) slot id outside [0,n_slots) or shared by two live questions */
  KEV_ERR_SLOT_OVERFLOW = 5, /* (device) a question longer than slot_cap, or no room for a decode row */
  KEV_ERR_TIMEOUT = 6,       /* (device) a bounded wait inside a kernel gave up; outputs are invalid */
  KEV_ERR_CUDA = 7,          /* a CUDA runtime call failed (launch error, no device, ...) */
  KEV_ERR_POSITION = 8,      /* (device) a position at or past the RoPE table's max_pos */
  KEV_ERR_PREFIX = 9,        /* (device) a cached prefix length negative or not a multiple of 128 */
  KEV_ERR_SAMPLING = 10,     /* (device) a live temperature negative / not finite, or a uniform outside [0,1) */
  KEV_ERR_ADAPTER = 11       /* (device) a LoRA adapter id outside [-1, n_adapters) */
} kev_status;

typedef enum { KEV_BF16 = 0, KEV_FP32 = 1 } kev_dtype;

/* Half-open interval [begin, end) of packed-token indices owned by one question. */
typedef struct {
  int32_t begin;
  int32_t end;
} kev_interval;

typedef struct {
  int32_t h_q;   /* query heads */
  int32_t h_kv;  /* key/value heads; h_q % h_kv == 0 */
  int32_t d_h;   /* head dimension: bf16 64 or 128; fp32 a multiple of 16 up to 256 */
  int32_t dtype; /* kev_dtype */
  float scale;   /* softmax scale; 0 => 1/sqrt(d_h) */
} kev_attn_shape;

/* ---------------------------------------------------------------------------------------
 * Prefill
 * ------------------------------------------------------------------------------------- */

/* Bytes of device workspace kev_prefill_attn / kev_build_segments / kev_kv_write need for
 * at most `n_questions` questions packed into `total_tokens` tokens.  0 on bad arguments. */
size_t kev_prefill_workspace_size(int32_t n_questions, int32_t total_tokens, const kev_attn_shape* shape);

/* Segment descriptors (step 1 of prefill; exported for tests and debugging).
 *
 * Validates the intervals (0 <= begin <= end <= T; non-empty intervals pairwise disjoint)
 * and, if slot_ids != NULL, the slots (every id in [0, n_slots); every length <= slot_cap;
 * non-empty questions on distinct slots -- two live questions sharing one cache is the
 * shared-state bug of the KV-cache isolation article, §2.3, §6.1).  Then writes into
 * `workspace`: the status word, cu_seqlens[N+1] (prefix sums of the lengths in interval
 * order, the varlen form of the block-diagonal mask, Kev architecture article §5.2, §6.4)
 * and the prefill work list: one item per (question, 128-row query tile, q-head block),
 * covering key tiles [0, m] of its own question only, so no tile that is masked across
 * questions or above the causal diagonal is ever scheduled.  Items are ordered longest
 * first.  Interval order is free and intervals need not cover [0, T): tokens in no
 * interval are keys for nobody and their output rows are written as 0.
 *   intervals  device kev_interval[n_questions]
 *   slot_ids   device int32[n_questions] or NULL (no slot checks)
 *   workspace  device, kev_prefill_workspace_size(...) bytes, 256-byte aligned */
kev_status kev_build_segments(const kev_interval* intervals, int32_t n_questions, int32_t total_tokens,
                              const int32_t* slot_ids, int32_t n_slots, int32_t slot_cap,
                              const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, kev_stream_t stream);

/* Host copy of the work list built by kev_build_segments (synchronises `stream`).
 * Each item is {question, q_row_begin, q_rows, first_head | (n_heads << 16) | (two_tiles << 30)}:
 * without two_tiles, n_heads consecutive q-heads of one kv group over one query tile (2 for
 * bf16, whose kernel runs two query tiles that share every K/V tile; 1 for fp32); with
 * two_tiles (bf16, when a group of an odd size leaves one q-head over), that q-head's query
 * tiles starting at q_row_begin and q_row_begin + 128, q_rows being the second tile's rows.
 * Items come longest first.  Returns the item count, or -1 on error (or when the list is in
 * unit form, below).  Writes at most `max_items` items to `items_out` (host int32[4*max_items]).
 * This item form is built for fp32, for bf16 with d_h = 64 and for the chunked prefill. */
int32_t kev_read_work_list(const void* workspace, size_t workspace_bytes, int32_t* items_out,
                           int32_t max_items, kev_stream_t stream);

/* Host copy of the work list in unit form, built by kev_build_segments for bf16 with d_h = 128
 * (synchronises `stream`): the work of the CTA-pair kernel, whose MMAs are 256 query rows tall,
 * 128 from each CTA of a pair.  Each unit is 8 int32: {question, kv_head, nkv_A | (nkv_B << 16),
 * 0, a0, a1, b0, b1}.  A "half" (a0 ... b1) is (m << 8) | h: query tile m of the question (rows
 * begin + 128 m ...) with q-head kv_head * G + h, or -1 for none.  Tile A is halves a0, a1 (one
 * per CTA), tile B halves b0, b1; tiles A and B share every K/V tile.  nkv_t is the key tiles
 * tile t runs: the larger of its halves' m + 1, or 0 when both are -1.  Per question and kv head,
 * the halves pair the q-heads (2e, 2e+1) of one query tile; with an odd group the last q-head
 * pairs its tiles m and m + 1 (m even); units take these pairs two by two in order of key-tile
 * count.  Units come longest first.  Returns the unit count, or -1 on error (or when the list is
 * in item form).  Writes at most `max_units` units to `units_out` (host int32[8*max_units]). */
int32_t kev_read_work_units(const void* workspace, size_t workspace_bytes, int32_t* units_out,
                            int32_t max_units, kev_stream_t stream);

/* Attention over a work list already built in `workspace` by kev_build_segments with the
 * same intervals/slots (step 2 of prefill), plus the slot write when slot_ids != NULL:
 *   out[t, h, :] = softmax_u(scale q[t,h].k[u,g] over allowed u) v[u,g]    (g = h / G)
 *   pool_{k,v}[slot_i, g, j, :] = {k,v}[begin_i + j, g, :]   for j < L_i   (bit copy)
 * Rows of tokens in no interval are written as zeros.  Pool positions >= L_i and slots no
 * question uses are not touched. */
kev_status kev_prefill_from_segments(const void* q, const void* k, const void* v, int32_t total_tokens,
                                     const kev_interval* intervals, int32_t n_questions,
                                     const int32_t* slot_ids, void* pool_k, void* pool_v,
                                     int32_t n_slots, int32_t slot_cap, void* out,
                                     const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, kev_stream_t stream);

/* Full prefill: kev_build_segments followed by kev_prefill_from_segments.
 * Pass slot_ids = NULL (and NULL pools) to skip the slot write. */
kev_status kev_prefill_attn(const void* q, const void* k, const void* v, int32_t total_tokens,
                            const kev_interval* intervals, int32_t n_questions,
                            const int32_t* slot_ids, void* pool_k, void* pool_v,
                            int32_t n_slots, int32_t slot_cap, void* out,
                            const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, kev_stream_t stream);

/* Slot write alone (validation of kev_build_segments, then the bit copy above).
 * Uses the same workspace as prefill. */
kev_status kev_kv_write(const void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                        int32_t n_questions, const int32_t* slot_ids, void* pool_k, void* pool_v,
                        int32_t n_slots, int32_t slot_cap, const kev_attn_shape* shape,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Decode
 * ------------------------------------------------------------------------------------- */

/* Bytes of decode workspace for up to `n_questions` questions in slots of `slot_cap`.
 * The workspace must be zero-filled once before its first use (e.g. cudaMemsetAsync);
 * every call that ends in KEV_OK leaves its counters at zero again (after a call whose
 * device status is KEV_ERR_TIMEOUT, zero it again).  Two calls in flight at the same time
 * must not share one workspace. */
size_t kev_decode_workspace_size(int32_t n_questions, int32_t slot_cap, const kev_attn_shape* shape);

/* One decode step over the slot pool (inference-engine notes §2.2; Kev pipeline article
 * §2.2-§2.3).  For every live question i (active[i] != 0), with n = lens[i]:
 *   pool_{k,v}[slot_ids[i], g, n, :] = {k,v}_new[i, g, :]                (append first)
 *   out[i, h, :] = softmax_j(scale q_new[i,h] . pool_k[slot, g, j]) pool_v[slot, g, j],
 *                  j = 0..n  (n + 1 positions; no mask: every cached position is visible)
 * Dropped questions (active[i] == 0) take no part: nothing is read or written for them,
 * their out rows keep their contents and their slot ids are not checked.
 * `lens` is read, never written (see kev_decode_advance).
 * Device-detected errors: KEV_ERR_SLOT (live slot id out of range or shared by two live
 * questions), KEV_ERR_SLOT_OVERFLOW (lens[i] < 0 or lens[i] >= slot_cap for a live i).
 *   slot_ids, lens   device int32[n_questions];  active  device uint8[n_questions] */
kev_status kev_decode_attn(const void* q_new, const void* k_new, const void* v_new,
                           void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap,
                           const int32_t* slot_ids, const int32_t* lens, const uint8_t* active,
                           int32_t n_questions, void* out, const kev_attn_shape* shape,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           kev_stream_t stream);

/* Size of the scratch area compiled into the library for kev_decode_attn_static (16 MiB). */
#define KEV_STATIC_SCRATCH_BYTES (16u << 20)

/* kev_decode_attn without a caller-provided workspace.  The pages have no counterpart: this is
 * a library-level convenience for callers that cannot allocate device memory (a plugin inside a
 * framework that owns the whole device-memory budget and hands out no allocator, or a
 * latency-critical path where cudaMalloc/cudaFree and their device synchronisation are not
 * allowed).  Same arguments, results and errors as kev_decode_attn, minus the workspace.
 * Scratch: a fixed device array of KEV_STATIC_SCRATCH_BYTES inside the library, held by every
 * GPU that loads it until the process exits.  The host checks of kev_decode_attn come first
 * (same codes, same order); then a call needing more scratch than the array holds
 * (kev_decode_workspace_size(...) > KEV_STATIC_SCRATCH_BYTES) returns KEV_ERR_UNSUPPORTED and
 * launches nothing.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress), so make that first call before any stream capture.  Every call
 * clears, in stream order and before its kernels, the part of the array that must start at
 * zero (scheduling words and arrival counters, a few KB): a call that ended in
 * KEV_ERR_TIMEOUT leaves nothing behind for the next one, unlike a caller workspace, which
 * must then be zeroed again.  Every call shares the array: calls that overlap on the GPU race
 * on it and give wrong results.  Allocates nothing (no cudaMalloc/cudaFree, no allocating
 * library routine). */
kev_status kev_decode_attn_static(const void* q_new, const void* k_new, const void* v_new,
                                  void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap,
                                  const int32_t* slot_ids, const int32_t* lens, const uint8_t* active,
                                  int32_t n_questions, void* out, const kev_attn_shape* shape,
                                  int32_t* dev_status, kev_stream_t stream);

/* lens[i] += (active[i] != 0) for i < n, on the device (no host synchronisation), so a
 * decode loop can be captured in a CUDA graph. */
kev_status kev_decode_advance(int32_t* lens, const uint8_t* active, int32_t n, kev_stream_t stream);

/* One decode step followed by the lens advance: kev_decode_attn, then lens[i] += 1 for every
 * live i once the step is complete (and only if the call is valid: on a device error lens is
 * left as it was).  Same arguments, results and errors as kev_decode_attn; `lens` is read and
 * then advanced.  On the tensor-core path (bf16, d_h = 128) the advance is folded into the
 * kernel that merges split pieces, so a step is two launches instead of three; this is the
 * form to capture in a CUDA graph for a decode loop. */
kev_status kev_decode_step(const void* q_new, const void* k_new, const void* v_new,
                           void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap,
                           const int32_t* slot_ids, int32_t* lens, const uint8_t* active,
                           int32_t n_questions, void* out, const kev_attn_shape* shape,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Per-question temperature sampling
 *
 * Kev architecture article (icman.com.cn), §4.1: each question brings its own temperature,
 * applied to the softmax of its logits at every decode step.  For a live question i with
 * T_i > 0 the token is the smallest k whose cumulative probability under softmax(logits_i /
 * T_i) exceeds u_i (inverse CDF; the uniforms u_i in [0, 1) are inputs, so a step can be
 * replayed); T_i = 0 takes the argmax, ties to the lowest index.  fp32 arithmetic: near a
 * boundary of the cumulative distribution (within its rounding) either neighbour can result.
 * ------------------------------------------------------------------------------------- */

/* logits: device [n_questions, vocab] of `dtype` (kev_dtype; vocab a multiple of 8 for bf16,
 * 4 for fp32, so rows stay 16-byte aligned); temperature, uniforms: device float[n]; active:
 * device uint8[n]; tokens: device int32[n], written for live questions only.  An invalid
 * live temperature or uniform sets KEV_ERR_SAMPLING and no token is written.  One kernel. */
kev_status kev_sample(const void* logits, int32_t n_questions, int32_t vocab, int32_t dtype, const float* temperature,
                      const float* uniforms, const uint8_t* active, int32_t* tokens, int32_t* dev_status,
                      kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Token-grouped LoRA
 *
 * Kev architecture article (icman.com.cn), §3.2: the base layer stays fixed and every token
 * takes the low-rank delta of its own question's adapter, computed per adapter group rather
 * than for every adapter over the whole sequence; §3.3: the scale is the adapter's alpha / rank.
 *   y[t] += scales[a] * lora_b[a] (lora_a[a] x[t])   for t in question i, a = adapter_ids[i] >= 0
 * ------------------------------------------------------------------------------------- */

/* Over the work list kev_build_segments built in `workspace` for the same intervals: x [T,
 * d_in] and y [T, d_out] bf16 (y updated in place; rows of questions without an adapter, id -1,
 * and of tokens in no question are not touched); lora_a [n_adapters, rank, d_in], lora_b
 * [n_adapters, d_out, rank] bf16; scales float[n_adapters]; adapter_ids int32[n_questions]; all
 * device.  rank 16, 32 or 64, d_in a multiple of 64, d_out a multiple of 32 (else
 * KEV_ERR_UNSUPPORTED).  An adapter id outside [-1, n_adapters) sets KEV_ERR_ADAPTER and nothing
 * is written.  bf16 products on the tensor cores, fp32 accumulation, y rounded to nearest even.
 * One kernel. */
kev_status kev_lora_apply(const void* x, void* y, int32_t total_tokens, int32_t d_in, int32_t d_out,
                          const kev_interval* intervals, int32_t n_questions, const int32_t* adapter_ids,
                          const void* lora_a, const void* lora_b, const float* scales, int32_t n_adapters,
                          int32_t rank, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Chunked prefill into slots
 *
 * Inference-engine notes (sakurs2.com), §2.6: a long input is prefilled in pieces that share
 * rounds with decode steps, each later piece using the K/V of the pieces before it.  Question
 * i's chunk is packed tokens [begin_i, end_i): its positions P_i .. P_i + L_i - 1 after the
 * P_i = prefix_lens[i] positions already in slot slot_ids[i].  The chunk's K/V rows go into the
 * slot first, then token begin_i + j attends to positions 0 .. P_i + j of its slot (the cached
 * prefix, and its own chunk causally):
 *   out[begin_i + j, h] = softmax_u(scale q . pool_k[slot_i, g, u]) pool_v[slot_i, g, u],  u <= P_i + j
 * ------------------------------------------------------------------------------------- */

/* Chunked prefill: segment build, slot write, attention.  bf16 only, slot_cap a multiple of 128
 * (else KEV_ERR_UNSUPPORTED); prefix_lens: device int32[n_questions], each a multiple of 128
 * (chunks start on a 128-row tile; else KEV_ERR_PREFIX) with P_i + L_i <= slot_cap (else
 * KEV_ERR_SLOT_OVERFLOW); slots as for kev_prefill_attn (required here).  Besides positions
 * P_i .. P_i + L_i - 1, the slot rows from P_i + L_i up to the next multiple of 128 are set to
 * zero (they hold no position yet; the attention's last key tile reads them).  Rows of tokens in
 * no interval are written as zeros.  A decode step is the one-token chunk at P_i = lens_i
 * without the alignment; use kev_decode_attn for it. */
kev_status kev_prefill_chunk(const void* q, const void* k, const void* v, int32_t total_tokens,
                             const kev_interval* intervals, int32_t n_questions, const int32_t* prefix_lens,
                             const int32_t* slot_ids, void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap,
                             void* out, const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Paged slot pool
 *
 * Inference-engine notes (sakurs2.com), §2.5: K/V are kept in fixed-size blocks taken on
 * demand, a block table records where each block lies, and attention reads K/V through the
 * table.  pool_{k,v}: [n_blocks, H_kv, KEV_PAGE, d_h]; block_table: device int32
 * [n_questions, max_blocks]; position p of question i lives in block
 * block_table[i * max_blocks + p / KEV_PAGE], row p % KEV_PAGE.  Entries past a question's
 * pages are never read.  n_questions * max_blocks <= KEV_MAX_PAGED_ENTRIES, else
 * KEV_ERR_UNSUPPORTED.  A block used by two questions (or twice by one) is KEV_ERR_SLOT --
 * the shared-state bug of the KV-cache isolation article (hnwysp.cn), §2.3 -- and a table
 * row with fewer blocks than the question's pages KEV_ERR_SLOT_OVERFLOW; both are found
 * before anything is written.
 * ------------------------------------------------------------------------------------- */
#define KEV_PAGE 128
#define KEV_MAX_PAGED_ENTRIES 16384

/* Prefill with a paged pool: kev_build_segments (no slot checks), a check of the block tables
 * of the questions' lengths (ceil(L_i / KEV_PAGE) blocks each), the attention, then the bit
 * copy of every question's K/V rows into its blocks.  Other pool rows are not touched. */
kev_status kev_prefill_attn_paged(const void* q, const void* k, const void* v, int32_t total_tokens,
                                  const kev_interval* intervals, int32_t n_questions, const int32_t* block_table,
                                  int32_t max_blocks, void* pool_k, void* pool_v, int32_t n_blocks, void* out,
                                  const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kev_stream_t stream);

/* The paged write alone: kev_build_segments, the table check, the copy of K/V rows into the
 * blocks (prefill workspace). */
kev_status kev_kv_write_paged(const void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                              int32_t n_questions, const int32_t* block_table, int32_t max_blocks, void* pool_k,
                              void* pool_v, int32_t n_blocks, const kev_attn_shape* shape, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, kev_stream_t stream);

/* One decode step over a paged pool (bf16, d_h = 128; else KEV_ERR_UNSUPPORTED): as
 * kev_decode_attn, the new row going to position lens_i, i.e. block
 * block_table[i][lens_i / KEV_PAGE], row lens_i % KEV_PAGE.  A live question needs blocks for
 * pages 0 .. lens_i / KEV_PAGE (else KEV_ERR_SLOT_OVERFLOW), in [0, n_blocks) and distinct
 * among live questions (else KEV_ERR_SLOT).  Workspace: kev_decode_workspace_size(n,
 * max_blocks * KEV_PAGE, shape), zero-filled once as for kev_decode_attn. */
kev_status kev_decode_attn_paged(const void* q_new, const void* k_new, const void* v_new, void* pool_k,
                                 void* pool_v, int32_t n_blocks, const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* lens, const uint8_t* active, int32_t n_questions, void* out,
                                 const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, kev_stream_t stream);

/* Host helper (no CUDA call): block tables for questions needing need[i] blocks, taken from
 * free_map (host uint8[n_blocks], 1 = free) in question order.  Contiguous first (Kev pipeline
 * article, gsyq.cn, §4.3: a batch's questions on neighbouring addresses): a question takes the
 * lowest run of need[i] consecutive free blocks, or, without one (or with contiguous_first =
 * 0), its lowest free blocks one by one.  Writes table (host int32[n * max_blocks], -1 past
 * each row's blocks) and clears the taken blocks in free_map.  Returns 0, or -1 with nothing
 * changed when the free blocks do not suffice or a need[i] exceeds max_blocks. */
int32_t kev_assign_blocks(const int32_t* need, int32_t n, uint8_t* free_map, int32_t n_blocks, int32_t* table,
                          int32_t max_blocks, int32_t contiguous_first);

/* ---------------------------------------------------------------------------------------
 * Rotary position encoding with positions counted per question
 *
 * KV-cache isolation article (hnwysp.cn, news 130224), §7.2: the rotation multiplies Q and
 * K, the cache holds K after its rotation, and a new token's position is the cache length
 * counted from 0.  Packed with isolation, every question counts from 0 as it would alone:
 * token t of question i has position t - begin_i, the decode token of question i position
 * lens_i.  Form: rotate-half -- element j < d_h/2 of a head pairs with element j + d_h/2 and
 * the pair (a, b) turns by p * w_j, w_j = theta^(-2j/d_h): (a cos - b sin, b cos + a sin).
 * Arithmetic in fp32 with the table's cos/sin, results rounded to the storage type (bf16:
 * to nearest even).  Tokens in no question are not rotated.
 * ------------------------------------------------------------------------------------- */

/* Bytes of the cos/sin table for positions [0, max_pos) and head size d_h: max_pos * d_h/2
 * pairs of floats.  0 for max_pos <= 0 or an odd d_h. */
size_t kev_rope_table_size(int32_t max_pos, int32_t d_h);

/* table[p * d_h/2 + j] = {cos(p w_j), sin(p w_j)} for p < max_pos, j < d_h/2: angles and
 * cos/sin in double precision, then rounded to float (one kernel).  `table`: device,
 * 16-byte aligned, kev_rope_table_size bytes, caller-owned.  Build once per (theta, d_h,
 * max_pos) and reuse.  theta > 1. */
kev_status kev_rope_table(void* table, int32_t max_pos, int32_t d_h, double theta, kev_stream_t stream);

/* Prefill-side RoPE over the work list kev_build_segments built in `workspace` for the same
 * intervals and slots: q [T,H_q,d] and k [T,H_kv,d] are rotated IN PLACE at their
 * per-question positions.  With slot_ids != NULL the rotated K rows and the V rows also go
 * into the slots (the slot write, fused: call kev_prefill_from_segments afterwards with
 * slot_ids = NULL).  A question longer than max_pos sets KEV_ERR_POSITION and the call,
 * like the calls after it on the same workspace, writes nothing.  One kernel. */
kev_status kev_rope_prefill(void* q, void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                            int32_t n_questions, const int32_t* slot_ids, void* pool_k, void* pool_v,
                            int32_t n_slots, int32_t slot_cap, const kev_attn_shape* shape, const void* rope_table,
                            int32_t max_pos, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            kev_stream_t stream);

/* Full prefill with RoPE: kev_build_segments, kev_rope_prefill (with the slot write), then
 * kev_prefill_from_segments without a slot write.  q and k are rotated in place. */
kev_status kev_prefill_attn_rope(void* q, void* k, const void* v, int32_t total_tokens,
                                 const kev_interval* intervals, int32_t n_questions, const int32_t* slot_ids,
                                 void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap, void* out,
                                 const kev_attn_shape* shape, const void* rope_table, int32_t max_pos,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kev_stream_t stream);

/* Decode-side RoPE: q_new [N,H_q,d] and k_new [N,H_kv,d] of every live question rotated IN
 * PLACE at position lens_i (the cache length before the step); rows of dropped questions
 * are untouched.  A live lens_i >= max_pos sets KEV_ERR_POSITION and nothing is written.
 * One kernel. */
kev_status kev_rope_decode(void* q_new, void* k_new, const int32_t* lens, const uint8_t* active,
                           int32_t n_questions, const kev_attn_shape* shape, const void* rope_table,
                           int32_t max_pos, int32_t* dev_status, kev_stream_t stream);

/* kev_rope_decode followed by kev_decode_attn: the pool receives the rotated new K row. */
kev_status kev_decode_attn_rope(void* q_new, void* k_new, const void* v_new, void* pool_k, void* pool_v,
                                int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids, const int32_t* lens,
                                const uint8_t* active, int32_t n_questions, void* out,
                                const kev_attn_shape* shape, const void* rope_table, int32_t max_pos,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                kev_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Status
 * ------------------------------------------------------------------------------------- */

/* Synchronises `stream`, reads the device status word and returns it (KEV_OK if no
 * device-side error), or KEV_ERR_CUDA if the stream itself reports an error. */
kev_status kev_read_status(const int32_t* dev_status, kev_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* kev_status_string(kev_status status);

/* Number of kernel launches the most recent successful call of each entry point enqueues
 * (for launch accounting): 0 = prefill_attn, 1 = prefill_from_segments, 2 = build_segments,
 * 3 = kv_write, 4 = decode_attn (2 when the last call ran on the tensor cores: bf16 with
 * d_h = 128, decode and merge kernels; 1 otherwise and before any call), 5 = decode_advance,
 * 6 = rope_table, 7 = rope_prefill, 8 = rope_decode (1 each), 9 = prefill_attn_paged (4:
 * segments, table check, attention, paged write), 10 = kv_write_paged (3), 11 =
 * decode_attn_paged (2), 12 = prefill_chunk (3: segments, slot write, attention), 13 =
 * sample (1), 14 = lora_apply (1), 15 = decode_step (2: decode + merge on the tensor cores,
 * decode + advance otherwise).  -1 for an unknown id. */
int32_t kev_launch_count(int32_t entry_point);

#ifdef __cplusplus
}
#endif

#endif /* KEV_H */
