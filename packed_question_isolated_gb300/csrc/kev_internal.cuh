// Internal declarations shared by the translation units of libkev (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/kev.h"

namespace kev {

// Query rows (and key rows) per prefill tile.  Tiles are laid out per question starting at
// the question's first token, so every key tile of a query tile lies inside its question.
constexpr int kTileM = 128;
// Upper bound on questions per call (the segment builder keeps them in shared memory).
constexpr int kMaxQuestions = 4096;
// Cost bins of the longest-first ordering: tile m (m+1 key tiles) goes to bin min(m, 63).
constexpr int kCostBins = 64;
// Positions per decode work item (split-K chunk).
constexpr int kDecodeChunk = 128;
// Largest q-head group (h_q / h_kv) the tensor-core decode covers with one MMA.
constexpr int kDecodeTcMaxGroup = 16;

// Device status codes: same values as kev_status.
enum : int32_t {
  ST_OK = 0,
  ST_INTERVALS = KEV_ERR_INTERVALS,
  ST_SLOT = KEV_ERR_SLOT,
  ST_OVERFLOW = KEV_ERR_SLOT_OVERFLOW,
  ST_TIMEOUT = KEV_ERR_TIMEOUT,
  ST_POSITION = KEV_ERR_POSITION,
  ST_PREFIX = KEV_ERR_PREFIX,
  ST_SAMPLING = KEV_ERR_SAMPLING,
  ST_ADAPTER = KEV_ERR_ADAPTER,
};

// ---------------------------------------------------------------------------------------
// prefill workspace
// ---------------------------------------------------------------------------------------
struct PrefillHeader {
  int32_t status;       // result of validation (and of bounded waits, if any gave up)
  int32_t n_items;      // work items emitted: {question, row_begin, rows, first_head | n_heads << 16}
  int32_t n_tiles;      // query tiles emitted
  int32_t n_gaps;       // ranges of tokens that belong to no question
  int32_t sched;        // dynamic-scheduling counter (reset by the segment builder)
  int32_t n_questions;
  int32_t total_tokens;
  int32_t h_q;
  int32_t format;       // 0: items (one int4 each); 1: units of the CTA-pair kernel (two int4 each)
};

struct PrefillLayout {
  size_t cu_seqlens;  // int32[N+1]
  size_t tiles;       // int2[max_tiles]  {question, m}
  size_t items;       // int4[max_items]  {question, row_begin, rows, first_head | n_heads << 16}
  size_t gaps;        // int2[N+1]        [begin, end)
  size_t total;
  int64_t max_tiles;
  int64_t max_items;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Cycle budget of one bounded wait inside a kernel: about two seconds at the top SM clock, or
// the value of the environment variable KEV_TEST_WAIT_LIMIT (cycles), read at every launch, so
// that a test can shorten it.
inline long long wait_budget_cycles() {
  const char* s = getenv("KEV_TEST_WAIT_LIMIT");
  if (s && *s) {
    const long long v = atoll(s);
    if (v > 0) return v;
  }
  return 4000000000ll;
}

// Test hook of the timeout path: with KEV_TEST_STALL=1 in the environment at launch, CTA 0 of
// the prefill and decode attention kernels first waits on an mbarrier that nothing ever
// arrives on.  The wait runs out after the budget above, and the kernel takes its real abort
// path (status KEV_ERR_TIMEOUT, abort flag, drain of its own copies and MMAs, TMEM freed, exit).
// Nothing faults, traps or hangs.  Off (0) unless the variable is set.
inline int test_stall_requested() {
  const char* s = getenv("KEV_TEST_STALL");
  return (s && *s == '1') ? 1 : 0;
}

inline PrefillLayout prefill_layout(int32_t n, int32_t T, int32_t h_q) {
  PrefillLayout L;
  size_t off = align_up(sizeof(PrefillHeader), 256);
  L.max_tiles = ((int64_t)T + kTileM - 1) / kTileM + n;  // 64-bit: T may be up to INT32_MAX
  // int4 records: items need at most max_tiles * h_q; CTA-pair units (two int4 each, one per
  // kv head and pair of pair-tiles) at most h_kv * (max_tiles * ceil(G/2) + n) <= (max_tiles + n) * h_q
  L.max_items = (L.max_tiles + n) * (int64_t)h_q;
  L.cu_seqlens = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(n + 1), 256);
  L.tiles = off;
  off = align_up(off + sizeof(int2) * (size_t)L.max_tiles, 256);
  L.items = off;
  off = align_up(off + sizeof(int4) * (size_t)L.max_items, 256);
  L.gaps = off;
  off = align_up(off + sizeof(int2) * (size_t)(n + 1), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------------------
// decode workspace
// ---------------------------------------------------------------------------------------
struct DecodeLayout {
  size_t sched;     // int32[8]  [2] validation code of the call (both paths); tensor-core decode: [0]
                    // batch-grab counter (left at zero), [1] [3] [4] grab plan
  size_t xi0;       // int2[N * H_kv]  tensor-core decode: {global index of chunk 0, chunk count} of each
                    // (question, kv head) (the merge kernel reads these, not lens)
  size_t counters;  // int32[N * H_kv * n_hblocks]  arrivals per (question, kv head, head block); left at zero
  size_t partials;  // float[N * H_kv * n_hblocks * max_chunks * GT * (d + 2)]
  size_t total;
  int32_t max_chunks;
};

// q-heads of one decode item: the group padded to a power of two, at most 8 (larger groups
// are split into blocks of 8).
inline int decode_head_block_size(int group) {
  const int g = group < 8 ? group : 8;
  return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
}

// `tc`: the tensor-core kernel (bf16, d = 128) takes the whole group (up to 16 q-heads, padded
// to 16) per item; the CUDA-core kernel takes blocks of up to 8.
inline DecodeLayout decode_layout(int32_t n, int32_t cap, int32_t h_q, int32_t h_kv, int32_t d, bool tc) {
  DecodeLayout L;
  L.max_chunks = (int32_t)(((int64_t)cap + kDecodeChunk - 1) / kDecodeChunk);
  const int32_t G = h_q / h_kv;
  const int32_t nhb = tc ? 1 : (G + 7) / 8;
  const int32_t GT = tc ? 16 : decode_head_block_size(G);
  size_t off = 0;
  L.sched = off;
  off = align_up(off + 8 * sizeof(int32_t), 256);
  L.xi0 = off;
  off = align_up(off + (tc ? sizeof(int2) * (size_t)n * h_kv : 0), 256);
  L.counters = off;
  off = align_up(off + sizeof(int32_t) * (size_t)n * h_kv * nhb, 256);
  L.partials = off;
  off = align_up(off + sizeof(float) * (size_t)n * h_kv * nhb * L.max_chunks * GT * (d + 2), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------------------
// launch argument blocks
// ---------------------------------------------------------------------------------------
struct SegmentsArgs {
  const kev_interval* intervals;
  const int32_t* slot_ids;  // may be null
  int32_t n;
  int32_t T;
  int32_t n_slots;
  int32_t cap;
  int32_t h_q;
  int32_t group;           // h_q / h_kv
  int32_t heads_per_item;  // consecutive q-heads of one kv group per work item (1 or 2)
  char* ws;
  PrefillLayout layout;
  int32_t* dev_status;  // may be null
  const int32_t* prefix_lens = nullptr;  // chunked prefill: cached positions before each chunk
  int32_t units2 = 0;  // 1: emit the work units of the CTA-pair kernel instead of items
};

// Work unit of the CTA-pair prefill kernel (two int4): {question, kv head g, nkv_A | nkv_B << 16,
// 0}, {s0, s1, s2, s3}.  A "half" s = (m << 8) | h is query tile m (rows m*128.. of the question)
// of q-head g*G + h, or -1 (empty).  The 256-row MMA tile A is halves s0 (even CTA) and s1 (odd
// CTA), tile B halves s2 and s3; nkv_t is the key tiles tile t runs (the larger of its halves'
// m + 1; 0 for an absent tile).
constexpr int kUnitHeadBits = 8;

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const kev_interval* intervals;
  int32_t T;
  int32_t n;
  int32_t h_q;
  int32_t h_kv;
  int32_t group;  // h_q / h_kv
  float scale;
  const char* ws;
  PrefillLayout layout;
  int32_t* dev_status;
  // chunked prefill: keys and values come from the slots [n_slots, H_kv, cap, d], where the
  // chunk's rows were written first; question i's queries sit at positions prefix_lens[i] + j
  const int32_t* prefix_lens = nullptr;
  const int32_t* slot_ids = nullptr;
  const void* pool_k = nullptr;
  const void* pool_v = nullptr;
  int32_t n_slots = 0;
  int32_t cap = 0;
  // CTA-pair kernel: also store every whole 128-row K/V tile of each question into its slot
  // (pools, slot_ids and cap above), from the shared-memory copies the attention loads anyway
  bool store_tiles = false;
};

struct AuxArgs {  // slot write + zero rows of tokens in no question
  const void* k;
  const void* v;
  void* out;  // may be null (slot write only)
  const kev_interval* intervals;
  const int32_t* slot_ids;  // may be null (gap zeroing only)
  void* pool_k;
  void* pool_v;
  int32_t n;
  int32_t T;
  int32_t h_q;
  int32_t h_kv;
  int32_t cap;
  int32_t n_slots;
  const int32_t* block_table = nullptr;  // paged pool (null: contiguous slots): see DecodeArgs
  int32_t max_blocks = 0;
  const int32_t* prefix_lens = nullptr;  // chunked prefill: chunk row j goes to slot position P_i + j,
                                         // and the slot rows up to the next multiple of 128 are zeroed
  int32_t row_bytes;  // d * element size
  const char* ws;
  PrefillLayout layout;
  // launched right after an attention kernel that waited for the segment builder before letting
  // this grid start: run alongside its tail, wait for it at the end
  bool after_attention = false;
  // the attention kernel stored every whole 128-row tile of each question: copy only the rows of
  // each question's last, partial tile
  bool tails_only = false;
};

struct DecodeArgs {
  const void* q_new;
  const void* k_new;
  const void* v_new;
  void* pool_k;
  void* pool_v;
  const int32_t* slot_ids;
  const int32_t* lens;
  const uint8_t* active;
  void* out;
  int32_t n;
  int32_t n_slots;
  int32_t cap;
  int32_t h_q;
  int32_t h_kv;
  int32_t group;
  float scale;
  char* ws;
  DecodeLayout layout;
  int32_t* dev_status;
  // paged pool (null: the contiguous [n_slots, H_kv, cap, d] pool): pool [n_blocks, H_kv, kPage, d],
  // position p of question i in block block_table[i * max_blocks + p / kPage]; cap = max_blocks * kPage
  const int32_t* block_table = nullptr;
  int32_t max_blocks = 0;
  int32_t n_blocks = 0;
  // bounded waits: cycles per wait, and the timeout test hook (both set by the launchers)
  long long wait_budget = 4000000000ll;
  int32_t test_stall = 0;
  // kev_decode_step: lens itself, advanced (lens[i] += 1 for live i) once the step is complete
  int32_t* advance_lens = nullptr;
};

// Host-side launchers (each returns the launch's cudaError_t).
cudaError_t launch_segments(const SegmentsArgs& a, cudaStream_t s);
cudaError_t launch_prefill_simt(const PrefillArgs& a, int d, int num_sms, cudaStream_t s);  // fp32
cudaError_t launch_prefill_tc(const PrefillArgs& a, int d, int num_sms, cudaStream_t s);    // bf16
cudaError_t launch_prefill_pair(const PrefillArgs& a, int num_sms, cudaStream_t s);         // bf16, d = 128
cudaError_t launch_aux(const AuxArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------------------
// paged slot pool (kev_paged.cu)
// ---------------------------------------------------------------------------------------
constexpr int kPage = 128;                  // positions per block (= a decode chunk, a prefill tile)
constexpr int kMaxPagedEntries = 16384;     // n_questions * max_blocks: the validation's hash capacity
static_assert(kPage == KEV_PAGE && kMaxPagedEntries == KEV_MAX_PAGED_ENTRIES && kMaxQuestions == KEV_MAX_QUESTIONS,
              "kev.h and the kernels agree");
struct PagedCheckArgs {                     // prefill side: the block tables of the questions' lengths
  const kev_interval* intervals;
  const int32_t* block_table;
  int32_t n, max_blocks, n_blocks;
  char* ws;  // prefill workspace: the header's status word is set on an error
  int32_t* dev_status;
};
cudaError_t launch_paged_check(const PagedCheckArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------------------
// per-question temperature sampling (kev_sample.cu)
// ---------------------------------------------------------------------------------------
struct SampleArgs {
  const void* logits;  // [n, vocab]
  int32_t n, vocab;
  int32_t elem;  // 2: bf16, 4: fp32
  const float* temperature;
  const float* uniforms;
  const uint8_t* active;
  int32_t* tokens;
  int32_t* dev_status;
};
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------------------
// token-grouped LoRA (kev_lora.cu)
// ---------------------------------------------------------------------------------------
struct LoraArgs {
  const void* x;  // [T, d_in] bf16
  void* y;        // [T, d_out] bf16, updated in place
  int32_t T, d_in, d_out, n, n_adapters, rank;
  const kev_interval* intervals;
  const int32_t* adapter_ids;  // [n], -1: no adapter
  const void* lora_a;          // [n_adapters, rank, d_in]
  const void* lora_b;          // [n_adapters, d_out, rank]
  const float* scales;         // [n_adapters]
  const char* ws;              // prefill workspace of kev_build_segments for the same intervals
  PrefillLayout layout;
  int32_t* dev_status;
};
cudaError_t launch_lora(const LoraArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------------------
// rotary position encoding (kev_rope.cu)
// ---------------------------------------------------------------------------------------
struct RopePrefillArgs {
  void* q;  // [T, H_q, d], rotated in place
  void* k;  // [T, H_kv, d], rotated in place
  const void* v;
  const kev_interval* intervals;
  const int32_t* slot_ids;  // null: no slot write
  void* pool_k;
  void* pool_v;
  int32_t n, T, h_q, h_kv, d, n_slots, cap, max_pos;
  int32_t elem;  // bytes per element: 2 (bf16) or 4 (fp32)
  const float2* table;
  const char* ws;
  PrefillLayout layout;
  int32_t* dev_status;
};
struct RopeDecodeArgs {
  void* q_new;  // [N, H_q, d]
  void* k_new;  // [N, H_kv, d]
  const int32_t* lens;
  const uint8_t* active;
  int32_t n, h_q, h_kv, d, max_pos;
  int32_t elem;
  const float2* table;
  int32_t* dev_status;
};
cudaError_t launch_rope_table(float2* table, int32_t max_pos, int32_t d, double theta, cudaStream_t s);
cudaError_t launch_rope_prefill(const RopePrefillArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_rope_decode(const RopeDecodeArgs& a, cudaStream_t s);
// kev_api.cu: the host checks of kev_decode_attn other than the workspace, and its workspace layout
kev_status decode_check_args(const void* q_new, const void* k_new, const void* v_new, const void* pool_k,
                             const void* pool_v, int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids,
                             const int32_t* lens, const uint8_t* active, int32_t n_questions, const void* out,
                             const kev_attn_shape* shape, const int32_t* dev_status);
DecodeLayout decode_layout_of(int32_t n_questions, int32_t slot_cap, const kev_attn_shape* shape);
cudaError_t launch_decode(const DecodeArgs& a, int d, kev_dtype dt, int num_sms, cudaStream_t s);     // CUDA cores
cudaError_t launch_decode_tc(const DecodeArgs& a, int num_sms, cudaStream_t s);                       // bf16, d = 128
// lens[i] += 1 for active i; with `code` (a device word), only if *code is ST_OK
cudaError_t launch_advance(int32_t* lens, const uint8_t* active, int32_t n, cudaStream_t s,
                           const int32_t* code = nullptr);

// ---------------------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Programmatic dependent launch: a kernel launched with launch_pdl may be scheduled while the
// kernel before it in the stream finishes; it calls pdl_wait() before it reads anything (the
// wait returns once that kernel has completed and its writes are visible), and pdl_trigger()
// lets the kernel after it be scheduled the same way.  Both are no-ops without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// First error wins; later kernels of the call read the word and write nothing.
__device__ __forceinline__ void set_status(int32_t* word, int32_t code) {
  if (word) atomicCAS(word, 0, code);
}

}  // namespace kev
