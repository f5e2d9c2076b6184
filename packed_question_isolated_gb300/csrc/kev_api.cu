// Host side of the C ABI declared in include/kev.h: argument checks and launches.
// No entry point allocates memory or synchronises, except kev_read_status / kev_read_work_list.
#include <math.h>
#include <string.h>

#include <atomic>

#include "kev_internal.cuh"

using namespace kev;

namespace {

// kernel launches of the most recent successful kev_decode_attn (2 on the tensor-core path)
std::atomic<int32_t> g_decode_launches{1};
// ... and of the most recent successful kev_decode_step (2: decode + merge, or decode + advance)
std::atomic<int32_t> g_step_launches{2};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int num_sms_of_current_device() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

kev_status check_shape(const kev_attn_shape* s) {
  if (!s) return KEV_ERR_INVALID_ARG;
  if (s->h_q <= 0 || s->h_kv <= 0) return KEV_ERR_INVALID_ARG;
  if (s->h_q % s->h_kv) return KEV_ERR_UNSUPPORTED;
  if (s->h_q / s->h_kv > 16) return KEV_ERR_UNSUPPORTED;
  if (s->dtype != KEV_BF16 && s->dtype != KEV_FP32) return KEV_ERR_UNSUPPORTED;
  // bf16: 64 or 128 (tensor cores); fp32 (CUDA cores): any multiple of 16 up to 256
  if (s->dtype == KEV_BF16 ? (s->d_h != 64 && s->d_h != 128) : (s->d_h < 16 || s->d_h > 256 || s->d_h % 16))
    return KEV_ERR_UNSUPPORTED;
  if (!(s->scale >= 0.f) || isinf(s->scale)) return KEV_ERR_INVALID_ARG;
  return KEV_OK;
}

// The RoPE kernels pair 16-byte chunks of a head's two halves: head dims 64 and 128.
bool rope_head_dim(const kev_attn_shape* s) { return s->d_h == 64 || s->d_h == 128; }

float effective_scale(const kev_attn_shape* s) {
  return s->scale == 0.f ? 1.0f / sqrtf((float)s->d_h) : s->scale;
}

int elem_size(const kev_attn_shape* s) { return s->dtype == KEV_BF16 ? 2 : 4; }

// bf16 prefill with d = 128 runs on CTA pairs (2-SM MMAs, unit work list); bf16 with d = 64 and the
// chunked prefill on single CTAs (item work list).
bool prefill_on_pairs(const kev_attn_shape* s) { return s->dtype == KEV_BF16 && s->d_h == 128; }

cudaError_t launch_prefill(const PrefillArgs& p, const kev_attn_shape* shape, int sms, cudaStream_t s) {
  if (shape->dtype != KEV_BF16) return launch_prefill_simt(p, shape->d_h, sms, s);
  return prefill_on_pairs(shape) ? launch_prefill_pair(p, sms, s) : launch_prefill_tc(p, shape->d_h, sms, s);
}

// bf16 with d = 128 decodes on the tensor cores; fp32 (no TF32) and d = 64 on the CUDA cores.
bool decode_on_tensor_cores(const kev_attn_shape* s) {
  return s->dtype == KEV_BF16 && s->d_h == 128 && s->h_q / s->h_kv <= kDecodeTcMaxGroup;
}

kev_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KEV_OK : KEV_ERR_CUDA; }

kev_status check_prefill_common(int32_t T, const kev_interval* intervals, int32_t n, const kev_attn_shape* shape,
                                void* ws, size_t ws_bytes) {
  kev_status st = check_shape(shape);
  if (st != KEV_OK) return st;
  if (T < 0 || n < 0) return KEV_ERR_INVALID_ARG;
  if (n > kMaxQuestions) return KEV_ERR_UNSUPPORTED;
  if (n > 0 && (!intervals || ((uintptr_t)intervals & 7u))) return KEV_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & 255u)) return KEV_ERR_INVALID_ARG;
  if (ws_bytes < prefill_layout(n, T, shape->h_q).total) return KEV_ERR_INVALID_ARG;
  return KEV_OK;
}

kev_status check_slots(const int32_t* slot_ids, void* pool_k, void* pool_v, int32_t n_slots, int32_t cap, int32_t n) {
  if (!slot_ids) return KEV_OK;
  if (((uintptr_t)slot_ids & 3u) || !pool_k || !pool_v || !aligned16(pool_k) || !aligned16(pool_v))
    return KEV_ERR_INVALID_ARG;
  if (n_slots <= 0 || cap <= 0) return KEV_ERR_INVALID_ARG;
  (void)n;
  return KEV_OK;
}

SegmentsArgs segments_args(const kev_interval* intervals, int32_t n, int32_t T, const int32_t* slot_ids,
                           int32_t n_slots, int32_t cap, const kev_attn_shape* shape, void* ws,
                           int32_t* dev_status) {
  SegmentsArgs a;
  a.intervals = intervals;
  a.slot_ids = slot_ids;
  a.n = n;
  a.T = T;
  a.n_slots = n_slots;
  a.cap = cap;
  a.h_q = shape->h_q;
  a.group = shape->h_q / shape->h_kv;
  // the tensor-core kernel takes two q-heads of a kv group per item, the fp32 kernel one
  a.heads_per_item = shape->dtype == KEV_BF16 ? 2 : 1;
  a.units2 = prefill_on_pairs(shape) ? 1 : 0;
  a.ws = static_cast<char*>(ws);
  a.layout = prefill_layout(n, T, shape->h_q);
  a.dev_status = dev_status;
  return a;
}

}  // namespace

// Host checks of kev_decode_attn's arguments other than the workspace, in its order.
kev_status kev::decode_check_args(const void* q_new, const void* k_new, const void* v_new, const void* pool_k,
                                  const void* pool_v, int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids,
                                  const int32_t* lens, const uint8_t* active, int32_t n_questions, const void* out,
                                  const kev_attn_shape* shape, const int32_t* dev_status) {
  kev_status st = check_shape(shape);
  if (st != KEV_OK) return st;
  if (n_questions < 0 || n_slots <= 0 || slot_cap <= 0) return KEV_ERR_INVALID_ARG;
  if (n_questions > kMaxQuestions) return KEV_ERR_UNSUPPORTED;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  if (n_questions == 0) return KEV_OK;
  if (!q_new || !k_new || !v_new || !pool_k || !pool_v || !out || !slot_ids || !lens || !active)
    return KEV_ERR_INVALID_ARG;
  if (!aligned16(q_new) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(pool_k) || !aligned16(pool_v) ||
      !aligned16(out) || ((uintptr_t)slot_ids & 3u) || ((uintptr_t)lens & 3u))
    return KEV_ERR_INVALID_ARG;
  return KEV_OK;
}

// The decode workspace layout of a call with these sizes (valid shape assumed).
DecodeLayout kev::decode_layout_of(int32_t n_questions, int32_t slot_cap, const kev_attn_shape* shape) {
  return decode_layout(n_questions, slot_cap, shape->h_q, shape->h_kv, shape->d_h, decode_on_tensor_cores(shape));
}

extern "C" {

size_t kev_prefill_workspace_size(int32_t n_questions, int32_t total_tokens, const kev_attn_shape* shape) {
  if (check_shape(shape) != KEV_OK || n_questions < 0 || total_tokens < 0 || n_questions > kMaxQuestions) return 0;
  return prefill_layout(n_questions, total_tokens, shape->h_q).total;
}

kev_status kev_build_segments(const kev_interval* intervals, int32_t n_questions, int32_t total_tokens,
                              const int32_t* slot_ids, int32_t n_slots, int32_t slot_cap,
                              const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (slot_ids && (((uintptr_t)slot_ids & 3u) || n_slots <= 0 || slot_cap <= 0)) return KEV_ERR_INVALID_ARG;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  SegmentsArgs a = segments_args(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape,
                                 workspace, dev_status);
  return from_cuda(launch_segments(a, (cudaStream_t)stream));
}

int32_t kev_read_work_list(const void* workspace, size_t workspace_bytes, int32_t* items_out, int32_t max_items,
                           kev_stream_t stream) {
  if (!workspace || workspace_bytes < sizeof(PrefillHeader) || max_items < 0) return -1;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return -1;
  PrefillHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (h.status != ST_OK || h.format != 0) return -1;
  const PrefillLayout L = prefill_layout(h.n_questions, h.total_tokens, h.h_q);
  if (workspace_bytes < L.total) return -1;
  const int32_t cnt = h.n_items < max_items ? h.n_items : max_items;
  if (cnt > 0 && items_out) {
    if (cudaMemcpy(items_out, static_cast<const char*>(workspace) + L.items, sizeof(int4) * (size_t)cnt,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      return -1;
  }
  return h.n_items;
}

int32_t kev_read_work_units(const void* workspace, size_t workspace_bytes, int32_t* units_out, int32_t max_units,
                            kev_stream_t stream) {
  if (!workspace || workspace_bytes < sizeof(PrefillHeader) || max_units < 0) return -1;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return -1;
  PrefillHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (h.status != ST_OK || h.format != 1) return -1;
  const PrefillLayout L = prefill_layout(h.n_questions, h.total_tokens, h.h_q);
  if (workspace_bytes < L.total) return -1;
  const int32_t cnt = h.n_items < max_units ? h.n_items : max_units;
  if (cnt > 0 && units_out) {
    if (cudaMemcpy(units_out, static_cast<const char*>(workspace) + L.items, 2 * sizeof(int4) * (size_t)cnt,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      return -1;
  }
  return h.n_items;
}

kev_status kev_prefill_from_segments(const void* q, const void* k, const void* v, int32_t total_tokens,
                                     const kev_interval* intervals, int32_t n_questions, const int32_t* slot_ids,
                                     void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap, void* out,
                                     const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (total_tokens > 0 && (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
    return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  const PrefillLayout layout = prefill_layout(n_questions, total_tokens, shape->h_q);

  PrefillArgs p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.intervals = intervals;
  p.T = total_tokens;
  p.n = n_questions;
  p.h_q = shape->h_q;
  p.h_kv = shape->h_kv;
  p.group = shape->h_q / shape->h_kv;
  p.scale = effective_scale(shape);
  p.ws = static_cast<const char*>(workspace);
  p.layout = layout;
  p.dev_status = dev_status;
  // the CTA-pair kernel stores the whole K/V tiles into the slots itself; the slot write below
  // then copies only each question's last, partial tile
  p.store_tiles = slot_ids != nullptr && total_tokens > 0 && prefill_on_pairs(shape) &&
                  (int64_t)n_slots * shape->h_kv * slot_cap < ((int64_t)1 << 31);  // TMA row coordinates
  if (p.store_tiles) {
    p.slot_ids = slot_ids;
    p.pool_k = pool_k;
    p.pool_v = pool_v;
    p.n_slots = n_slots;
    p.cap = slot_cap;
  }
  cudaError_t e = launch_prefill(p, shape, sms, s);
  if (e != cudaSuccess) return KEV_ERR_CUDA;

  AuxArgs x;
  x.k = k;
  x.v = v;
  x.out = out;
  x.intervals = intervals;
  x.slot_ids = slot_ids;
  x.pool_k = pool_k;
  x.pool_v = pool_v;
  x.n = n_questions;
  x.T = total_tokens;
  x.h_q = shape->h_q;
  x.h_kv = shape->h_kv;
  x.cap = slot_cap;
  x.n_slots = n_slots;
  x.row_bytes = shape->d_h * elem_size(shape);
  x.ws = static_cast<const char*>(workspace);
  x.layout = layout;
  x.after_attention = total_tokens > 0;  // the attention kernel was launched just before
  x.tails_only = p.store_tiles;
  return from_cuda(launch_aux(x, sms, s));
}

kev_status kev_prefill_attn(const void* q, const void* k, const void* v, int32_t total_tokens,
                            const kev_interval* intervals, int32_t n_questions, const int32_t* slot_ids,
                            void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap, void* out,
                            const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, kev_stream_t stream) {
  // full argument check before the first launch, so an invalid call enqueues nothing
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (total_tokens > 0 && (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
    return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  st = kev_build_segments(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape, workspace,
                          workspace_bytes, dev_status, stream);
  if (st != KEV_OK) return st;
  return kev_prefill_from_segments(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots,
                                   slot_cap, out, shape, workspace, workspace_bytes, dev_status, stream);
}

kev_status kev_kv_write(const void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                        int32_t n_questions, const int32_t* slot_ids, void* pool_k, void* pool_v, int32_t n_slots,
                        int32_t slot_cap, const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (!slot_ids) return KEV_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  st = kev_build_segments(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape, workspace,
                          workspace_bytes, dev_status, stream);
  if (st != KEV_OK) return st;
  AuxArgs x;
  x.k = k;
  x.v = v;
  x.out = nullptr;
  x.intervals = intervals;
  x.slot_ids = slot_ids;
  x.pool_k = pool_k;
  x.pool_v = pool_v;
  x.n = n_questions;
  x.T = total_tokens;
  x.h_q = shape->h_q;
  x.h_kv = shape->h_kv;
  x.cap = slot_cap;
  x.n_slots = n_slots;
  x.row_bytes = shape->d_h * elem_size(shape);
  x.ws = static_cast<const char*>(workspace);
  x.layout = prefill_layout(n_questions, total_tokens, shape->h_q);
  x.after_attention = false;
  return from_cuda(launch_aux(x, sms, (cudaStream_t)stream));
}

namespace {

kev_status check_paged(const int32_t* block_table, int32_t max_blocks, void* pool_k, void* pool_v, int32_t n_blocks,
                       int32_t n) {
  if (!block_table || ((uintptr_t)block_table & 3u) || max_blocks <= 0 || n_blocks <= 0) return KEV_ERR_INVALID_ARG;
  if (!pool_k || !pool_v || !aligned16(pool_k) || !aligned16(pool_v)) return KEV_ERR_INVALID_ARG;
  if ((int64_t)n * max_blocks > kMaxPagedEntries || (int64_t)max_blocks * kPage > (1 << 30)) return KEV_ERR_UNSUPPORTED;
  return KEV_OK;
}

// table check and paged write of a prefill whose work list kev_build_segments just built
kev_status paged_prefill_tail(const void* q, const void* k, const void* v, int32_t T, const kev_interval* intervals,
                              int32_t n, const int32_t* block_table, int32_t max_blocks, void* pool_k, void* pool_v,
                              int32_t n_blocks, void* out, const kev_attn_shape* shape, void* ws, int32_t* dev_status,
                              cudaStream_t s) {
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  const PrefillLayout layout = prefill_layout(n, T, shape->h_q);
  PagedCheckArgs c;
  c.intervals = intervals;
  c.block_table = block_table;
  c.n = n;
  c.max_blocks = max_blocks;
  c.n_blocks = n_blocks;
  c.ws = static_cast<char*>(ws);
  c.dev_status = dev_status;
  if (launch_paged_check(c, s) != cudaSuccess) return KEV_ERR_CUDA;
  bool attention = false;
  if (out) {
    PrefillArgs p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.intervals = intervals;
    p.T = T;
    p.n = n;
    p.h_q = shape->h_q;
    p.h_kv = shape->h_kv;
    p.group = shape->h_q / shape->h_kv;
    p.scale = effective_scale(shape);
    p.ws = static_cast<const char*>(ws);
    p.layout = layout;
    p.dev_status = dev_status;
    const cudaError_t e = launch_prefill(p, shape, sms, s);
    if (e != cudaSuccess) return KEV_ERR_CUDA;
    attention = T > 0;
  }
  AuxArgs x;
  x.k = k;
  x.v = v;
  x.out = out;
  x.intervals = intervals;
  x.slot_ids = nullptr;
  x.pool_k = pool_k;
  x.pool_v = pool_v;
  x.n = n;
  x.T = T;
  x.h_q = shape->h_q;
  x.h_kv = shape->h_kv;
  x.cap = max_blocks * kPage;
  x.n_slots = n_blocks;
  x.block_table = block_table;
  x.max_blocks = max_blocks;
  x.row_bytes = shape->d_h * elem_size(shape);
  x.ws = static_cast<const char*>(ws);
  x.layout = layout;
  x.after_attention = attention;
  return from_cuda(launch_aux(x, sms, s));
}

}  // namespace

kev_status kev_lora_apply(const void* x, void* y, int32_t total_tokens, int32_t d_in, int32_t d_out,
                          const kev_interval* intervals, int32_t n_questions, const int32_t* adapter_ids,
                          const void* lora_a, const void* lora_b, const float* scales, int32_t n_adapters,
                          int32_t rank, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          kev_stream_t stream) {
  if (total_tokens < 0 || n_questions < 0 || n_adapters < 0 || d_in <= 0 || d_out <= 0) return KEV_ERR_INVALID_ARG;
  if (n_questions > kMaxQuestions || d_in % 64 || d_out % 32 || (rank != 16 && rank != 32 && rank != 64))
    return KEV_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u)) return KEV_ERR_INVALID_ARG;
  // the work list is that of any shape with one q-head: only cu_seqlens and the status are read
  if (workspace_bytes < prefill_layout(n_questions, total_tokens, 1).cu_seqlens + sizeof(int32_t) * (n_questions + 1))
    return KEV_ERR_INVALID_ARG;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  if (total_tokens == 0 || n_questions == 0) return KEV_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y) || !intervals || ((uintptr_t)intervals & 7u) || !adapter_ids ||
      ((uintptr_t)adapter_ids & 3u))
    return KEV_ERR_INVALID_ARG;
  if (n_adapters > 0 && (!lora_a || !lora_b || !scales || !aligned16(lora_a) || !aligned16(lora_b) ||
                         ((uintptr_t)scales & 3u)))
    return KEV_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  LoraArgs a;
  a.x = x;
  a.y = y;
  a.T = total_tokens;
  a.d_in = d_in;
  a.d_out = d_out;
  a.n = n_questions;
  a.n_adapters = n_adapters;
  a.rank = rank;
  a.intervals = intervals;
  a.adapter_ids = adapter_ids;
  a.lora_a = lora_a;
  a.lora_b = lora_b;
  a.scales = scales;
  a.ws = static_cast<const char*>(workspace);
  a.layout = prefill_layout(n_questions, total_tokens, 1);
  a.dev_status = dev_status;
  return from_cuda(launch_lora(a, sms, (cudaStream_t)stream));
}

kev_status kev_sample(const void* logits, int32_t n_questions, int32_t vocab, int32_t dtype, const float* temperature,
                      const float* uniforms, const uint8_t* active, int32_t* tokens, int32_t* dev_status,
                      kev_stream_t stream) {
  if (n_questions < 0 || vocab <= 0) return KEV_ERR_INVALID_ARG;
  if (dtype != KEV_BF16 && dtype != KEV_FP32) return KEV_ERR_UNSUPPORTED;
  // every CTA checks every live question's temperature and uniform (so an invalid call writes
  // no token): n^2 small reads, bounded by the library's question limit
  if (n_questions > kMaxQuestions) return KEV_ERR_UNSUPPORTED;
  if (vocab % (dtype == KEV_BF16 ? 8 : 4)) return KEV_ERR_UNSUPPORTED;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  if (n_questions == 0) return KEV_OK;
  if (!logits || !aligned16(logits) || !temperature || !uniforms || !active || !tokens || ((uintptr_t)temperature & 3u) ||
      ((uintptr_t)uniforms & 3u) || ((uintptr_t)tokens & 3u))
    return KEV_ERR_INVALID_ARG;
  SampleArgs a;
  a.logits = logits;
  a.n = n_questions;
  a.vocab = vocab;
  a.elem = dtype == KEV_BF16 ? 2 : 4;
  a.temperature = temperature;
  a.uniforms = uniforms;
  a.active = active;
  a.tokens = tokens;
  a.dev_status = dev_status;
  return from_cuda(launch_sample(a, (cudaStream_t)stream));
}

kev_status kev_prefill_chunk(const void* q, const void* k, const void* v, int32_t total_tokens,
                             const kev_interval* intervals, int32_t n_questions, const int32_t* prefix_lens,
                             const int32_t* slot_ids, void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap,
                             void* out, const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (shape->dtype != KEV_BF16 || slot_cap % kTileM != 0) return KEV_ERR_UNSUPPORTED;
  if (total_tokens > 0 && (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
    return KEV_ERR_INVALID_ARG;
  if (!slot_ids || (n_questions > 0 && (!prefix_lens || ((uintptr_t)prefix_lens & 3u)))) return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  // 1. segments, with the prefixes (validation, costs)
  SegmentsArgs sa = segments_args(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape, workspace,
                                  dev_status);
  sa.prefix_lens = prefix_lens;
  sa.units2 = 0;  // the chunked prefill runs on single CTAs over the item list
  if (launch_segments(sa, s) != cudaSuccess) return KEV_ERR_CUDA;
  const PrefillLayout layout = prefill_layout(n_questions, total_tokens, shape->h_q);
  // 2. the chunk's K/V rows into the slots (the attention reads them there), gap rows of out
  AuxArgs x;
  x.k = k;
  x.v = v;
  x.out = out;
  x.intervals = intervals;
  x.slot_ids = slot_ids;
  x.pool_k = pool_k;
  x.pool_v = pool_v;
  x.n = n_questions;
  x.T = total_tokens;
  x.h_q = shape->h_q;
  x.h_kv = shape->h_kv;
  x.cap = slot_cap;
  x.n_slots = n_slots;
  x.prefix_lens = prefix_lens;
  x.row_bytes = shape->d_h * elem_size(shape);
  x.ws = static_cast<const char*>(workspace);
  x.layout = layout;
  x.after_attention = false;
  if (launch_aux(x, sms, s) != cudaSuccess) return KEV_ERR_CUDA;
  // 3. attention over each slot's prefix and the chunk
  PrefillArgs p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.intervals = intervals;
  p.T = total_tokens;
  p.n = n_questions;
  p.h_q = shape->h_q;
  p.h_kv = shape->h_kv;
  p.group = shape->h_q / shape->h_kv;
  p.scale = effective_scale(shape);
  p.ws = static_cast<const char*>(workspace);
  p.layout = layout;
  p.dev_status = dev_status;
  p.prefix_lens = prefix_lens;
  p.slot_ids = slot_ids;
  p.pool_k = pool_k;
  p.pool_v = pool_v;
  p.n_slots = n_slots;
  p.cap = slot_cap;
  return from_cuda(launch_prefill_tc(p, shape->d_h, sms, s));
}

kev_status kev_prefill_attn_paged(const void* q, const void* k, const void* v, int32_t total_tokens,
                                  const kev_interval* intervals, int32_t n_questions, const int32_t* block_table,
                                  int32_t max_blocks, void* pool_k, void* pool_v, int32_t n_blocks, void* out,
                                  const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (total_tokens > 0 && (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
    return KEV_ERR_INVALID_ARG;
  st = check_paged(block_table, max_blocks, pool_k, pool_v, n_blocks, n_questions);
  if (st != KEV_OK) return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  st = kev_build_segments(intervals, n_questions, total_tokens, nullptr, 0, 0, shape, workspace, workspace_bytes,
                          dev_status, stream);
  if (st != KEV_OK) return st;
  return paged_prefill_tail(q, k, v, total_tokens, intervals, n_questions, block_table, max_blocks, pool_k, pool_v,
                            n_blocks, out, shape, workspace, dev_status, (cudaStream_t)stream);
}

kev_status kev_kv_write_paged(const void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                              int32_t n_questions, const int32_t* block_table, int32_t max_blocks, void* pool_k,
                              void* pool_v, int32_t n_blocks, const kev_attn_shape* shape, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (total_tokens > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return KEV_ERR_INVALID_ARG;
  st = check_paged(block_table, max_blocks, pool_k, pool_v, n_blocks, n_questions);
  if (st != KEV_OK) return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  st = kev_build_segments(intervals, n_questions, total_tokens, nullptr, 0, 0, shape, workspace, workspace_bytes,
                          dev_status, stream);
  if (st != KEV_OK) return st;
  return paged_prefill_tail(nullptr, k, v, total_tokens, intervals, n_questions, block_table, max_blocks, pool_k,
                            pool_v, n_blocks, nullptr, shape, workspace, dev_status, (cudaStream_t)stream);
}

kev_status kev_decode_attn_paged(const void* q_new, const void* k_new, const void* v_new, void* pool_k,
                                 void* pool_v, int32_t n_blocks, const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* lens, const uint8_t* active, int32_t n_questions, void* out,
                                 const kev_attn_shape* shape, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_shape(shape);
  if (st != KEV_OK) return st;
  if (!decode_on_tensor_cores(shape)) return KEV_ERR_UNSUPPORTED;
  if (n_questions < 0) return KEV_ERR_INVALID_ARG;
  if (n_questions > kMaxQuestions) return KEV_ERR_UNSUPPORTED;
  st = check_paged(block_table, max_blocks, pool_k, pool_v, n_blocks, n_questions);
  if (st != KEV_OK) return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  if (n_questions == 0) {
    if (dev_status) return from_cuda(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), (cudaStream_t)stream));
    return KEV_OK;
  }
  if (!q_new || !k_new || !v_new || !out || !lens || !active) return KEV_ERR_INVALID_ARG;
  if (!aligned16(q_new) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) || ((uintptr_t)lens & 3u))
    return KEV_ERR_INVALID_ARG;
  const int32_t cap = max_blocks * kPage;
  const DecodeLayout layout = decode_layout(n_questions, cap, shape->h_q, shape->h_kv, shape->d_h, true);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < layout.total) return KEV_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  DecodeArgs a;
  a.q_new = q_new;
  a.k_new = k_new;
  a.v_new = v_new;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.slot_ids = nullptr;
  a.lens = lens;
  a.active = active;
  a.out = out;
  a.n = n_questions;
  a.n_slots = 0;
  a.cap = cap;
  a.h_q = shape->h_q;
  a.h_kv = shape->h_kv;
  a.group = shape->h_q / shape->h_kv;
  a.scale = effective_scale(shape);
  a.ws = static_cast<char*>(workspace);
  a.layout = layout;
  a.dev_status = dev_status;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.n_blocks = n_blocks;
  return from_cuda(launch_decode_tc(a, sms, (cudaStream_t)stream));
}

int32_t kev_assign_blocks(const int32_t* need, int32_t n, uint8_t* free_map, int32_t n_blocks, int32_t* table,
                          int32_t max_blocks, int32_t contiguous_first) {
  if (n < 0 || n_blocks < 0 || max_blocks <= 0 || (n > 0 && (!need || !table)) || (n_blocks > 0 && !free_map))
    return -1;
  int64_t total = 0, avail = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (need[i] < 0 || need[i] > max_blocks) return -1;
    total += need[i];
  }
  for (int32_t b = 0; b < n_blocks; ++b) avail += free_map[b] != 0;
  if (total > avail) return -1;  // every question can take its blocks one by one: no partial change
  for (int32_t i = 0; i < n; ++i) {
    int32_t* row = table + (int64_t)i * max_blocks;
    for (int32_t c = 0; c < max_blocks; ++c) row[c] = -1;
    const int32_t m = need[i];
    if (m == 0) continue;
    int32_t start = -1;
    if (contiguous_first) {
      int32_t run = 0;
      for (int32_t b = 0; b < n_blocks; ++b) {
        run = free_map[b] ? run + 1 : 0;
        if (run == m) {
          start = b - m + 1;
          break;
        }
      }
    }
    if (start >= 0) {
      for (int32_t c = 0; c < m; ++c) {
        row[c] = start + c;
        free_map[start + c] = 0;
      }
    } else {
      int32_t c = 0;
      for (int32_t b = 0; b < n_blocks && c < m; ++b)
        if (free_map[b]) {
          row[c++] = b;
          free_map[b] = 0;
        }
    }
  }
  return 0;
}

size_t kev_rope_table_size(int32_t max_pos, int32_t d_h) {
  if (max_pos <= 0 || d_h <= 0 || (d_h & 1)) return 0;
  return sizeof(float2) * (size_t)max_pos * (size_t)(d_h / 2);
}

kev_status kev_rope_table(void* table, int32_t max_pos, int32_t d_h, double theta, kev_stream_t stream) {
  if (!table || !aligned16(table) || max_pos <= 0 || max_pos > (1 << 24)) return KEV_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return KEV_ERR_UNSUPPORTED;
  if (!(theta > 1.0) || isinf(theta)) return KEV_ERR_INVALID_ARG;
  return from_cuda(launch_rope_table(static_cast<float2*>(table), max_pos, d_h, theta, (cudaStream_t)stream));
}

kev_status kev_rope_prefill(void* q, void* k, const void* v, int32_t total_tokens, const kev_interval* intervals,
                            int32_t n_questions, const int32_t* slot_ids, void* pool_k, void* pool_v,
                            int32_t n_slots, int32_t slot_cap, const kev_attn_shape* shape, const void* rope_table,
                            int32_t max_pos, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            kev_stream_t stream) {
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (!rope_head_dim(shape)) return KEV_ERR_UNSUPPORTED;
  if (total_tokens > 0 && (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)))
    return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  if (!rope_table || !aligned16(rope_table) || max_pos <= 0) return KEV_ERR_INVALID_ARG;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  RopePrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.intervals = intervals;
  a.slot_ids = slot_ids;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.n = n_questions;
  a.T = total_tokens;
  a.h_q = shape->h_q;
  a.h_kv = shape->h_kv;
  a.d = shape->d_h;
  a.n_slots = slot_ids ? n_slots : 0;
  a.cap = slot_ids ? slot_cap : 0;
  a.max_pos = max_pos;
  a.elem = elem_size(shape);
  a.table = static_cast<const float2*>(rope_table);
  a.ws = static_cast<const char*>(workspace);
  a.layout = prefill_layout(n_questions, total_tokens, shape->h_q);
  a.dev_status = dev_status;
  return from_cuda(launch_rope_prefill(a, sms, (cudaStream_t)stream));
}

kev_status kev_prefill_attn_rope(void* q, void* k, const void* v, int32_t total_tokens,
                                 const kev_interval* intervals, int32_t n_questions, const int32_t* slot_ids,
                                 void* pool_k, void* pool_v, int32_t n_slots, int32_t slot_cap, void* out,
                                 const kev_attn_shape* shape, const void* rope_table, int32_t max_pos,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 kev_stream_t stream) {
  // full argument check before the first launch, so an invalid call enqueues nothing
  kev_status st = check_prefill_common(total_tokens, intervals, n_questions, shape, workspace, workspace_bytes);
  if (st != KEV_OK) return st;
  if (!rope_head_dim(shape)) return KEV_ERR_UNSUPPORTED;
  if (total_tokens > 0 && (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)))
    return KEV_ERR_INVALID_ARG;
  st = check_slots(slot_ids, pool_k, pool_v, n_slots, slot_cap, n_questions);
  if (st != KEV_OK) return st;
  if (!rope_table || !aligned16(rope_table) || max_pos <= 0) return KEV_ERR_INVALID_ARG;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  st = kev_build_segments(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape, workspace,
                          workspace_bytes, dev_status, stream);
  if (st != KEV_OK) return st;
  st = kev_rope_prefill(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots, slot_cap,
                        shape, rope_table, max_pos, workspace, workspace_bytes, dev_status, stream);
  if (st != KEV_OK) return st;
  return kev_prefill_from_segments(q, k, v, total_tokens, intervals, n_questions, nullptr, nullptr, nullptr, 0, 0,
                                   out, shape, workspace, workspace_bytes, dev_status, stream);
}

kev_status kev_rope_decode(void* q_new, void* k_new, const int32_t* lens, const uint8_t* active,
                           int32_t n_questions, const kev_attn_shape* shape, const void* rope_table,
                           int32_t max_pos, int32_t* dev_status, kev_stream_t stream) {
  kev_status st = check_shape(shape);
  if (st != KEV_OK) return st;
  if (!rope_head_dim(shape)) return KEV_ERR_UNSUPPORTED;
  if (n_questions < 0) return KEV_ERR_INVALID_ARG;
  if (n_questions > kMaxQuestions) return KEV_ERR_UNSUPPORTED;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return KEV_ERR_INVALID_ARG;
  if (n_questions == 0) return KEV_OK;
  if (!q_new || !k_new || !lens || !active || !aligned16(q_new) || !aligned16(k_new) || ((uintptr_t)lens & 3u))
    return KEV_ERR_INVALID_ARG;
  if (!rope_table || !aligned16(rope_table) || max_pos <= 0) return KEV_ERR_INVALID_ARG;
  RopeDecodeArgs a;
  a.q_new = q_new;
  a.k_new = k_new;
  a.lens = lens;
  a.active = active;
  a.n = n_questions;
  a.h_q = shape->h_q;
  a.h_kv = shape->h_kv;
  a.d = shape->d_h;
  a.max_pos = max_pos;
  a.elem = elem_size(shape);
  a.table = static_cast<const float2*>(rope_table);
  a.dev_status = dev_status;
  return from_cuda(launch_rope_decode(a, (cudaStream_t)stream));
}

kev_status kev_decode_attn_rope(void* q_new, void* k_new, const void* v_new, void* pool_k, void* pool_v,
                                int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids, const int32_t* lens,
                                const uint8_t* active, int32_t n_questions, void* out,
                                const kev_attn_shape* shape, const void* rope_table, int32_t max_pos,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                kev_stream_t stream) {
  // a table that covers the slot: a lens past the table is also past the slot, which the
  // decode rejects on its own, so neither call writes anything for such a step
  if (max_pos < slot_cap) return KEV_ERR_INVALID_ARG;
  kev_status st = check_shape(shape);
  if (st != KEV_OK) return st;
  if (n_questions < 0 || n_slots <= 0 || slot_cap <= 0) return KEV_ERR_INVALID_ARG;
  if (n_questions > 0 && (!v_new || !pool_k || !pool_v || !out || !slot_ids)) return KEV_ERR_INVALID_ARG;
  const DecodeLayout layout =
      decode_layout(n_questions, slot_cap, shape->h_q, shape->h_kv, shape->d_h, decode_on_tensor_cores(shape));
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < layout.total) return KEV_ERR_INVALID_ARG;
  st = kev_rope_decode(q_new, k_new, lens, active, n_questions, shape, rope_table, max_pos, dev_status, stream);
  if (st != KEV_OK) return st;
  return kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active, n_questions,
                         out, shape, workspace, workspace_bytes, dev_status, stream);
}

size_t kev_decode_workspace_size(int32_t n_questions, int32_t slot_cap, const kev_attn_shape* shape) {
  if (check_shape(shape) != KEV_OK || n_questions < 0 || slot_cap <= 0 || n_questions > kMaxQuestions) return 0;
  return decode_layout(n_questions, slot_cap, shape->h_q, shape->h_kv, shape->d_h, decode_on_tensor_cores(shape)).total;
}

}  // extern "C"

namespace {
// kev_decode_attn, and with `advance` (kev_decode_step) lens[i] += 1 for live i once the step is
// complete: in the merge kernel on the tensor-core path, by the advance kernel otherwise.
// `entry` is the launch-count slot of the calling entry point.
kev_status decode_call(const void* q_new, const void* k_new, const void* v_new, void* pool_k, void* pool_v,
                       int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids, const int32_t* lens,
                       const uint8_t* active, int32_t n_questions, void* out, const kev_attn_shape* shape,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, kev_stream_t stream,
                       int32_t* advance, int entry) {
  kev_status st = kev::decode_check_args(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens,
                                         active, n_questions, out, shape, dev_status);
  if (st != KEV_OK) return st;
  if (n_questions == 0) {
    if (dev_status) return from_cuda(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), (cudaStream_t)stream));
    return KEV_OK;
  }
  const DecodeLayout layout =
      decode_layout(n_questions, slot_cap, shape->h_q, shape->h_kv, shape->d_h, decode_on_tensor_cores(shape));
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < layout.total) return KEV_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return KEV_ERR_CUDA;
  DecodeArgs a;
  a.q_new = q_new;
  a.k_new = k_new;
  a.v_new = v_new;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.slot_ids = slot_ids;
  a.lens = lens;
  a.active = active;
  a.out = out;
  a.n = n_questions;
  a.n_slots = n_slots;
  a.cap = slot_cap;
  a.h_q = shape->h_q;
  a.h_kv = shape->h_kv;
  a.group = shape->h_q / shape->h_kv;
  a.scale = effective_scale(shape);
  a.ws = static_cast<char*>(workspace);
  a.layout = layout;
  a.dev_status = dev_status;
  std::atomic<int32_t>& launches = entry == 4 ? g_decode_launches : g_step_launches;
  if (decode_on_tensor_cores(shape)) {  // decode kernel + merge kernel (which also advances lens)
    a.advance_lens = advance;
    st = from_cuda(launch_decode_tc(a, sms, (cudaStream_t)stream));
    if (st == KEV_OK) launches.store(2);
    return st;
  }
  st = from_cuda(launch_decode(a, shape->d_h, (kev_dtype)shape->dtype, sms, (cudaStream_t)stream));
  if (st == KEV_OK && advance)  // only if the step was valid: the decode kernels store their code in sched[2]
    st = from_cuda(launch_advance(advance, active, n_questions, (cudaStream_t)stream,
                                  reinterpret_cast<const int32_t*>(static_cast<char*>(workspace) + layout.sched) + 2));
  if (st == KEV_OK) launches.store(advance ? 2 : 1);
  return st;
}
}  // namespace

extern "C" {


kev_status kev_decode_attn(const void* q_new, const void* k_new, const void* v_new, void* pool_k, void* pool_v,
                           int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids, const int32_t* lens,
                           const uint8_t* active, int32_t n_questions, void* out, const kev_attn_shape* shape,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status, kev_stream_t stream) {
  return decode_call(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active, n_questions, out,
                     shape, workspace, workspace_bytes, dev_status, stream, nullptr, 4);
}

kev_status kev_decode_step(const void* q_new, const void* k_new, const void* v_new, void* pool_k, void* pool_v,
                           int32_t n_slots, int32_t slot_cap, const int32_t* slot_ids, int32_t* lens,
                           const uint8_t* active, int32_t n_questions, void* out, const kev_attn_shape* shape,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status, kev_stream_t stream) {
  return decode_call(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active, n_questions, out,
                     shape, workspace, workspace_bytes, dev_status, stream, lens, 15);
}

kev_status kev_decode_advance(int32_t* lens, const uint8_t* active, int32_t n, kev_stream_t stream) {
  if (n < 0) return KEV_ERR_INVALID_ARG;
  if (n == 0) return KEV_OK;
  if (!lens || !active || ((uintptr_t)lens & 3u)) return KEV_ERR_INVALID_ARG;
  return from_cuda(launch_advance(lens, active, n, (cudaStream_t)stream));
}

kev_status kev_read_status(const int32_t* dev_status, kev_stream_t stream) {
  if (!dev_status) return KEV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KEV_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return KEV_ERR_CUDA;
  if (h < KEV_OK || h > KEV_ERR_ADAPTER) return KEV_ERR_CUDA;
  return (kev_status)h;
}

const char* kev_status_string(kev_status s) {
  switch (s) {
    case KEV_OK: return "ok";
    case KEV_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, bad size or workspace too small)";
    case KEV_ERR_UNSUPPORTED: return "unsupported dtype, head dim or group size";
    case KEV_ERR_INTERVALS: return "intervals reversed, outside [0,T] or overlapping";
    case KEV_ERR_SLOT: return "slot id out of range or shared by two live questions";
    case KEV_ERR_SLOT_OVERFLOW: return "question longer than slot capacity or no room for the decode row";
    case KEV_ERR_TIMEOUT: return "a bounded device wait gave up";
    case KEV_ERR_CUDA: return "CUDA runtime error";
    case KEV_ERR_POSITION: return "a position at or past the RoPE table's max_pos";
    case KEV_ERR_PREFIX: return "a cached prefix length negative or not a multiple of 128";
    case KEV_ERR_SAMPLING: return "a live temperature negative or not finite, or a uniform outside [0, 1)";
    case KEV_ERR_ADAPTER: return "a LoRA adapter id outside [-1, n_adapters)";
  }
  return "unknown status";
}

int32_t kev_launch_count(int32_t entry_point) {
  switch (entry_point) {
    case 0: return 3;  // segments, attention, slot write / gap zero
    case 1: return 2;  // attention, slot write / gap zero
    case 2: return 1;
    case 3: return 2;  // segments, slot write
    case 4: return g_decode_launches.load();
    case 5: return 1;
    case 6: return 1;
    case 7: return 1;
    case 8: return 1;
    case 9: return 4;
    case 10: return 3;
    case 11: return 2;
    case 12: return 3;
    case 13: return 1;
    case 14: return 1;
    case 15: return g_step_launches.load();
  }
  return -1;
}

}  // extern "C"
