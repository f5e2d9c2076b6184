// Per-question temperature sampling.
//
// Kev architecture article (icman.com.cn), §4.1: every question brings its own temperature,
// applied to the softmax of its logits at each decode step.  Question i with T_i > 0 takes
// token k, the smallest index whose cumulative probability under softmax(logits_i / T_i)
// exceeds its uniform u_i in [0, 1) (inverse CDF: the random number is an input, so a step is
// reproducible); T_i = 0 is the greedy argmax, ties to the lowest index.
//
// sample_kernel: one CTA of 1024 threads per question; thread t owns the t-th contiguous range
// of the row.  Each thread keeps an online max and sum of exp(z - max), z = logit / T, over its
// range; after a block reduction of the max, its range's weight is its sum rescaled to the row
// max, and one block scan of those weights gives every thread its interval of the cumulative
// weight.  The one thread whose interval holds u * total walks its range to the crossing.  Every
// block first checks every live question's temperature and uniform, so an invalid call writes
// no token.
#include <climits>

#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kSampleThreads = 1024;

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

// 8 consecutive logits from k0 (a multiple of 8), as floats; positions at or past k_hi give -inf
template <typename E>
__device__ __forceinline__ void load8(const E* row, int k0, int k_hi, float* f);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* row, int k0, int k_hi, float* f) {
  if (k0 + 8 <= k_hi) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k0));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = k0 + e < k_hi ? __bfloat162float(row[k0 + e]) : -INFINITY;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* row, int k0, int k_hi, float* f) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = k0 + 4 * h;
    if (b + 4 <= k_hi) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + b));
      f[4 * h] = v.x;
      f[4 * h + 1] = v.y;
      f[4 * h + 2] = v.z;
      f[4 * h + 3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) f[4 * h + e] = b + e < k_hi ? row[b + e] : -INFINITY;
    }
  }
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
  __shared__ float s_incl[kSampleThreads];  // inclusive prefixes of the ranges' weights
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
  // every thread owns one contiguous range of the row, in index order, of a multiple of 8
  // elements (16-byte aligned: rows are, the vocabulary being a multiple of 8 or 4)
  const int per = ((V + kSampleThreads - 1) / kSampleThreads + 7) / 8 * 8;
  const int k_lo = min(V, tid * per), k_hi = min(V, k_lo + per);
  // max and sum of exp(z - max) over the range, 16 logits (two vector loads) at a time
  float m = -INFINITY, s = 0.f;
  for (int k0 = k_lo; k0 < k_hi; k0 += 32) {
    float f[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) load8<E>(row, k0 + 8 * v, k_hi, f + 8 * v);  // four loads in flight
    float bm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      f[e] *= inv_t;
      bm = fmaxf(bm, f[e]);
    }
    if (bm > m) {
      s = m == -INFINITY ? 0.f : s * expf(m - bm);
      m = bm;
    }
    float add = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) add += expf(f[e] - m);  // exp(-inf) = 0 past the range
    s += add;
  }
  float bm = m, bs = s;  // block max (and sum, unused beyond the max)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ms_combine(bm, bs, __shfl_down_sync(0xffffffffu, bm, o), __shfl_down_sync(0xffffffffu, bs, o));
  if (lane == 0) {
    s_m[warp] = bm;
    s_s[warp] = bs;
  }
  __syncthreads();
  if (tid == 0) {
    float mm = s_m[0], ss = s_s[0];
    for (int w = 1; w < 32; ++w) ms_combine(mm, ss, s_m[w], s_s[w]);
    s_m[0] = mm;
    s_token = INT_MAX;
  }
  __syncthreads();
  const float mx = s_m[0];
  // the range's weight relative to the row max, then one scan: thread t covers
  // [excl_t, incl_t) of the cumulative weight, excl_t being thread t-1's incl itself
  const float local = m == -INFINITY ? 0.f : s * expf(m - mx);
  float total;
  s_incl[tid] = block_scan(local, s_scan, &total);
  __syncthreads();
  total = s_incl[kSampleThreads - 1];
  const float incl = s_incl[tid];
  const float excl = tid > 0 ? s_incl[tid - 1] : 0.f;
  const float target = a.uniforms[i] * total;
  // the crossing is in one thread's range: that thread's warp walks the range together, one
  // vector of 8 per lane in a pass (per / 8 <= 32 for a vocabulary up to 262,144), then a warp
  // scan finds the lane and the element
  const bool mine = excl <= target && target < incl;
  const unsigned who = __ballot_sync(0xffffffffu, mine);
  if (who) {
    const int src = __ffs(who) - 1;  // the claiming lane (one, in any rounding: the first)
    const int r_lo = __shfl_sync(0xffffffffu, k_lo, src), r_hi = __shfl_sync(0xffffffffu, k_hi, src);
    const float base = __shfl_sync(0xffffffffu, excl, src);
    int tok = r_hi - 1;
    float c0 = base;  // cumulative weight before this pass
    for (int p0 = r_lo; p0 < r_hi; p0 += 256) {
      const int k0 = p0 + 8 * lane;
      float f[8];
      load8<E>(row, k0, r_hi, f);
      float w[8], lsum = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        w[e] = expf(f[e] * inv_t - mx);
        lsum += w[e];
      }
      float x = lsum;  // inclusive scan over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float before = c0 + (x - lsum);
      const bool cross = before + lsum > target && k0 < r_hi;
      const unsigned hits = __ballot_sync(0xffffffffu, cross);
      if (hits) {
        const int hl = __ffs(hits) - 1;
        if (lane == hl) {
          float c = before;
          int t = min(k0 + 7, r_hi - 1);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            c += w[e];
            if (c > target) {
              t = k0 + e;
              break;
            }
          }
          tok = t;
        }
        tok = __shfl_sync(0xffffffffu, tok, hl);
        break;
      }
      c0 += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) atomicMin(&s_token, tok);
  }
  __syncthreads();
  if (s_token == INT_MAX) {  // rounding left the target at or above the total: the last element with weight
    __shared__ int s_last;
    if (tid == 0) s_last = 0;
    __syncthreads();
    for (int k = k_hi - 1; k >= k_lo; --k)
      if (expf(to_f(row[k]) * inv_t - mx) > 0.f) {
        atomicMax(&s_last, k);
        break;
      }
    __syncthreads();
    if (tid == 0) a.tokens[i] = s_last;
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
