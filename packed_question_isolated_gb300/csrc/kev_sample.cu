// Per-question temperature sampling.
//
// Kev architecture article (icman.com.cn), §4.1: every question brings its own temperature,
// applied to the softmax of its logits at each decode step.  Question i with T_i > 0 takes
// token k, the smallest index whose cumulative probability under softmax(logits_i / T_i)
// exceeds its uniform u_i in [0, 1) (inverse CDF: the random number is an input, so a step is
// reproducible); T_i = 0 is the greedy argmax, ties to the lowest index.
//
// sample_kernel: one CTA of 1024 threads per question.  Pass A: online max and sum of
// exp(z - max), z = logit / T, over the row.  Pass B: the row again in tiles of 1024 x 8
// elements in index order (8 consecutive elements per thread); a block scan of the threads'
// sums places the tile's prefix, and the tile in which the running sum passes u * S is searched
// by the one thread whose elements hold the crossing.  Every block first checks every live
// question's temperature and uniform, so an invalid call writes no token.
#include <climits>

#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kSampleThreads = 1024;
constexpr int kPer = 8;  // consecutive elements per thread in a tile of pass B

template <typename E>
__device__ __forceinline__ float to_f(E x);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}

// (max, sum) pairs: the sum rescaled to the larger max
__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mm = fmaxf(m, m2);
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// inclusive scan of v over the block; returns the thread's inclusive prefix, *total the sum
__device__ float block_scan(float v, float* warp_tot, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const float r = x + (warp > 0 ? warp_tot[warp - 1] : 0.f);
  *total = warp_tot[31];
  __syncthreads();  // warp_tot is reused by the next call
  return r;
}

template <typename E>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(SampleArgs a) {
  __shared__ float s_m[32], s_s[32], s_scan[32];
  __shared__ float s_incl[kSampleThreads];  // a tile's inclusive prefixes, thread by thread
  __shared__ int s_i[32];
  __shared__ int s_token;
  pdl_wait();  // the logits, temperatures and uniforms are complete
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  bool bad = false;
  for (int j = tid; j < a.n; j += blockDim.x) {
    if (!a.active[j]) continue;
    const float t = a.temperature[j], u = a.uniforms[j];
    bad |= !(t >= 0.f) || isinf(t) || !(u >= 0.f) || !(u < 1.f);
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) set_status(a.dev_status, ST_SAMPLING);
    return;
  }
  const int i = blockIdx.x;
  if (!a.active[i]) return;
  const int V = a.vocab;
  const E* row = static_cast<const E*>(a.logits) + (int64_t)i * V;
  const float T = a.temperature[i];

  if (T == 0.f) {  // greedy: the first maximum
    float best = -INFINITY;
    int bi = V;
    for (int k = tid; k < V; k += blockDim.x) {
      const float x = to_f(row[k]);
      if (x > best) {  // k increases per thread: the first maximum of this thread
        best = x;
        bi = k;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float b2 = __shfl_down_sync(0xffffffffu, best, o);
      const int i2 = __shfl_down_sync(0xffffffffu, bi, o);
      if (b2 > best || (b2 == best && i2 < bi)) {
        best = b2;
        bi = i2;
      }
    }
    if (lane == 0) {
      s_m[warp] = best;
      s_i[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float b = s_m[0];
      int bk = s_i[0];
      for (int w = 1; w < 32; ++w)
        if (s_m[w] > b || (s_m[w] == b && s_i[w] < bk)) {
          b = s_m[w];
          bk = s_i[w];
        }
      a.tokens[i] = bk < V ? bk : 0;
    }
    return;
  }

  const float inv_t = 1.0f / T;
  // pass A: online max and sum
  float m = -INFINITY, s = 0.f;
  for (int k = tid; k < V; k += blockDim.x) {
    const float z = to_f(row[k]) * inv_t;
    if (z > m) {
      s = (m == -INFINITY ? 0.f : s * expf(m - z)) + 1.f;
      m = z;
    } else {
      s += expf(z - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ms_combine(m, s, __shfl_down_sync(0xffffffffu, m, o), __shfl_down_sync(0xffffffffu, s, o));
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = s;
  }
  __syncthreads();
  if (tid == 0) {
    float mm = s_m[0], ss = s_s[0];
    for (int w = 1; w < 32; ++w) ms_combine(mm, ss, s_m[w], s_s[w]);
    s_m[0] = mm;
    s_s[0] = ss;
    s_token = INT_MAX;
  }
  __syncthreads();
  const float mx = s_m[0];
  const float target = a.uniforms[i] * s_s[0];

  // pass B: tiles in index order; the running sum crosses the target in exactly one place
  float running = 0.f;
  int last_pos = -1;  // this thread's last element with a nonzero weight (rounding fallback)
  for (int base = 0; base < V; base += kSampleThreads * kPer) {
    const int k0 = base + tid * kPer;
    float w[kPer];
    float local = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      w[e] = k0 + e < V ? expf(to_f(row[k0 + e]) * inv_t - mx) : 0.f;
      local += w[e];
      if (w[e] > 0.f) last_pos = k0 + e;
    }
    float tile;
    // this thread's elements cover [running + excl, running + incl): excl is the previous
    // thread's inclusive prefix itself, so consecutive intervals meet exactly
    s_incl[tid] = block_scan(local, s_scan, &tile);
    __syncthreads();
    const float incl = s_incl[tid];
    const float excl = tid > 0 ? s_incl[tid - 1] : 0.f;
    tile = s_incl[kSampleThreads - 1];
    const float before = running + excl;
    if (running + tile > target) {
      if (before <= target && target < running + incl) {  // the crossing is in this thread's elements
        float c = before;
        int tok = k0 + kPer - 1;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          c += w[e];
          if (c > target) {
            tok = k0 + e;
            break;
          }
        }
        atomicMin(&s_token, tok);  // the intervals partition the tile: one thread, in any rounding
      }
      __syncthreads();
      break;
    }
    running += tile;
    __syncthreads();  // s_incl is rewritten by the next tile
  }
  __syncthreads();
  if (s_token == INT_MAX) {  // rounding left the target at or above the sum: the last nonzero weight
    __shared__ int s_last;
    if (tid == 0) s_last = -1;
    __syncthreads();
    atomicMax(&s_last, last_pos);
    __syncthreads();
    if (tid == 0) a.tokens[i] = s_last >= 0 ? s_last : 0;
    return;
  }
  if (tid == 0) a.tokens[i] = s_token;
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s) {
  auto kern = a.elem == 2 ? sample_kernel<__nv_bfloat16> : sample_kernel<float>;
  return launch_pdl(kern, dim3(a.n), dim3(kSampleThreads), 0, s, a);
}

}  // namespace kev
