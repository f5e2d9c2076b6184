// Packed prefill attention on the CUDA cores (the float32 path: true fp32 FMA, no TF32).
//
// Exact attention, Z = softmax(QK^T / sqrt(d_h) + M) V (inference-engine notes,
// sakurs2.com, §2.1), with M the causal AND block-diagonal mask of the Kev articles
// (icman.com.cn §2.3, gsyq.cn §2.2) applied as a key range: row t of question i reads keys
// [begin_i, t] only.  Keys are taken 32 at a time with the online softmax of the notes'
// §2.4 (running max m, sum l, rescale alpha = exp(m_old - m_new)).
//
// Work: one CTA of 4 warps per item of the segment builder's list (question, 128-row tile,
// q-head); warp w takes rows w, w+4, ...  Inside a 32-key block lane j owns key j for the
// score and dims j, j+32, j+64, ... (< D) for the output accumulator.  D is any multiple of 16
// up to 256, taken at run time; PER = ceil(D / 32) is the accumulator's length.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 256;

template <typename T, int PER>
__global__ void __launch_bounds__(kWarps * 32) prefill_simt_kernel(PrefillArgs a, int D) {
  __shared__ float q_s[kWarps][kMaxD];
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(a.ws);
  if (hdr->status != ST_OK) return;
  if (hdr->format != 0) {  // the work list was built for another kernel (another shape)
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(a.dev_status, KEV_ERR_INVALID_ARG);
    return;
  }
  const int n_items = hdr->n_items;
  const int4* items = reinterpret_cast<const int4*>(a.ws + a.layout.items);
  const T* __restrict__ Q = static_cast<const T*>(a.q);
  const T* __restrict__ K = static_cast<const T*>(a.k);
  const T* __restrict__ V = static_cast<const T*>(a.v);
  T* __restrict__ O = static_cast<T*>(a.out);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t q_row = (int64_t)a.h_q * D, kv_row = (int64_t)a.h_kv * D;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 item = items[it];
    const int seg_begin = a.intervals[item.x].begin;
    const int h = item.w & 0xffff, g = h / a.group;  // one head per item on this path
    for (int r = warp; r < item.z; r += kWarps) {
      const int t = item.y + r;
      __syncwarp();
      for (int c = lane; c < D; c += 32) q_s[warp][c] = to_f32(Q[(int64_t)t * q_row + (int64_t)h * D + c]);
      __syncwarp();
      float m = -INFINITY, l = 0.f;
      float acc[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = 0.f;
      for (int kb = seg_begin; kb <= t; kb += 32) {
        const int key = kb + lane;
        float s = -INFINITY;
        if (key <= t) {
          const T* kr = K + (int64_t)key * kv_row + (int64_t)g * D;
          float dot = 0.f;
#pragma unroll 8
          for (int c = 0; c < D; ++c) dot = fmaf(q_s[warp][c], to_f32(kr[c]), dot);
          s = dot * a.scale;
        }
        const float m_new = fmaxf(m, warp_max(s));
        const float alpha = expf(m - m_new);  // m = -inf on the first block gives 0
        const float p = (key <= t) ? expf(s - m_new) : 0.f;
        l = l * alpha + warp_sum(p);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] *= alpha;
        const int nk = min(32, t - kb + 1);
        for (int j = 0; j < nk; ++j) {
          const float pj = __shfl_sync(0xffffffffu, p, j);
          const T* vr = V + (int64_t)(kb + j) * kv_row + (int64_t)g * D + lane;
#pragma unroll
          for (int e = 0; e < PER; ++e)
            if (lane + 32 * e < D) acc[e] = fmaf(pj, to_f32(vr[32 * e]), acc[e]);
        }
        m = m_new;
      }
      const float inv = 1.f / l;
      T* orow = O + (int64_t)t * q_row + (int64_t)h * D + lane;
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if (lane + 32 * e < D) orow[32 * e] = from_f32<T>(acc[e] * inv);
    }
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, int d, int num_sms, cudaStream_t s) {
  const int64_t max_items = a.layout.max_items;
  if (max_items == 0) return cudaSuccess;
  if (d < 16 || d > kMaxD || d % 16) return cudaErrorInvalidValue;
  const int grid = (int)(max_items < (int64_t)num_sms * 16 ? max_items : (int64_t)num_sms * 16);
  if (d <= 64) prefill_simt_kernel<float, 2><<<grid, kWarps * 32, 0, s>>>(a, d);
  else if (d <= 128) prefill_simt_kernel<float, 4><<<grid, kWarps * 32, 0, s>>>(a, d);
  else prefill_simt_kernel<float, 8><<<grid, kWarps * 32, 0, s>>>(a, d);
  return cudaGetLastError();
}

}  // namespace kev
