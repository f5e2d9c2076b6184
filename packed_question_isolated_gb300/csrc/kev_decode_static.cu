// kev_decode_attn_static: the decode step of kev_decode_attn without a caller workspace.
//
// Some callers cannot allocate device memory at all: a plugin running inside a host
// framework that owns the whole device-memory budget and gives it no allocator, or code on a
// latency-critical path where cudaMalloc / cudaFree (which may synchronise the device) are not
// allowed.  Such callers still own their inputs and outputs, but have nowhere to put the
// decode step's scratch (split-K partial results and per-(question, kv-head) arrival
// counters).  This entry point uses a fixed scratch area compiled into the library instead.
//
// The scratch is one file-scope device array of KEV_STATIC_SCRATCH_BYTES.  Every GPU that
// loads the library holds it until the process exits.  Host code never passes the array's
// name to a kernel (on the host that name is only a stand-in, not a device address): the
// device address is looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device; make that first call before any stream
// capture.  Every call first clears, in stream order, the part of the array that must start at
// zero (the scheduling words and the per-(question, kv head) arrival counters, a few KB), so a
// call that ended in KEV_ERR_TIMEOUT -- which can leave counters behind -- does not disturb the
// next one.  All calls share the array: calls that overlap on the GPU (different streams, or
// different host threads without ordering between them) race on it.
#include <mutex>

#include "kev_internal.cuh"

namespace {

__device__ __align__(256) unsigned char kev_static_scratch[KEV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use.
kev_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KEV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, kev_static_scratch) != cudaSuccess || !ptr) return KEV_ERR_CUDA;
    g_scratch[dev] = ptr;
  }
  *out = g_scratch[dev];
  return KEV_OK;
}

}  // namespace

extern "C" kev_status kev_decode_attn_static(const void* q_new, const void* k_new, const void* v_new, void* pool_k,
                                             void* pool_v, int32_t n_slots, int32_t slot_cap,
                                             const int32_t* slot_ids, const int32_t* lens, const uint8_t* active,
                                             int32_t n_questions, void* out, const kev_attn_shape* shape,
                                             int32_t* dev_status, kev_stream_t stream) {
  // the same host checks as kev_decode_attn, in the same order, before the size limit
  const kev_status chk = kev::decode_check_args(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids,
                                                lens, active, n_questions, out, shape, dev_status);
  if (chk != KEV_OK) return chk;
  if (n_questions == 0)  // nothing to do: kev_decode_attn only clears the status word
    return kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                           n_questions, out, shape, nullptr, 0, dev_status, stream);
  const kev::DecodeLayout layout = kev::decode_layout_of(n_questions, slot_cap, shape);
  if (layout.total > (size_t)KEV_STATIC_SCRATCH_BYTES) return KEV_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = nullptr;
  const kev_status st = scratch_for_current_device(&scratch);
  if (st != KEV_OK) return st;
  // scheduling words and arrival counters start at zero on every call (partials need no clearing)
  if (cudaMemsetAsync(scratch, 0, layout.partials, (cudaStream_t)stream) != cudaSuccess) return KEV_ERR_CUDA;
  return kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                         n_questions, out, shape, scratch, (size_t)KEV_STATIC_SCRATCH_BYTES, dev_status, stream);
}
