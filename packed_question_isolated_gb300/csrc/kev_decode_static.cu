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
// current, on the first call made on that device.  That first call also clears the arrival
// counters (every later call leaves them at zero again), so make it before any stream capture.
// All calls share the array: calls that overlap on the GPU (different streams, or different
// host threads without ordering between them) race on it.
#include <mutex>

#include "kev_internal.cuh"

namespace {

__device__ __align__(256) unsigned char kev_static_scratch[KEV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device, set up on first use.
kev_status scratch_for_current_device(void** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KEV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, kev_static_scratch) != cudaSuccess || !ptr) return KEV_ERR_CUDA;
    // counters must start at zero; clear the whole area once, in stream order
    if (cudaMemsetAsync(ptr, 0, KEV_STATIC_SCRATCH_BYTES, stream) != cudaSuccess) return KEV_ERR_CUDA;
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
  const size_t need = kev_decode_workspace_size(n_questions, slot_cap, shape);
  if (need > (size_t)KEV_STATIC_SCRATCH_BYTES) return KEV_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (need == 0 || n_questions == 0) {
    // bad arguments (or nothing to do): kev_decode_attn answers before it launches anything
    return kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                           n_questions, out, shape, nullptr, 0, dev_status, stream);
  }
  void* scratch = nullptr;
  const kev_status st = scratch_for_current_device(&scratch, (cudaStream_t)stream);
  if (st != KEV_OK) return st;
  return kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                         n_questions, out, shape, scratch, (size_t)KEV_STATIC_SCRATCH_BYTES, dev_status, stream);
}
