// Per-question temperature sampling.
//
// Kev architecture article (icman.com.cn), §4.1: every question brings its own temperature,
// applied to the softmax of its logits at each decode step.  Question i with T_i > 0 takes
// token k, the smallest index whose cumulative probability under softmax(logits_i / T_i)
// exceeds its uniform u_i in [0, 1) (inverse CDF: the random number is an input, so a step is
// reproducible); T_i = 0 is the greedy argmax, ties to the lowest index.
//
// sample_kernel: one thread-block cluster of S <= 8 CTAs per question (S grows with the
// vocabulary), CTA r of the cluster owning the r-th contiguous segment of the row, and thread t
// of a CTA the t-th contiguous range of its segment.  Each thread keeps an online max and sum of
// exp(z - max), z = logit / T, over its range; a block reduction gives the segment's (max, sum),
// which the CTAs exchange through distributed shared memory.  Every CTA of the cluster then
// derives the same row max, segment weights and cumulative intervals, so exactly one CTA, the one
// whose segment's interval holds u * total, goes on: one block scan of its threads' weights, and
// the one thread whose interval holds the rest of the target walks its range to the crossing.
// Greedy rows exchange each segment's first maximum the same way.  Every block first checks
// every live question's temperature and uniform, so an invalid call writes no token.
#include <algorithm>
#include <climits>

#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kSampleThreads = 512;
constexpr int kMaxCluster = 8;  // the portable cluster size

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; shared-memory writes before it are visible to the
// whole cluster after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the 32-bit word at the same shared-memory offset as `p` in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t ld_peer_u32(const void* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}


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
    float w = lane < kSampleThreads / 32 ? warp_tot[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const float r = x + (warp > 0 ? warp_tot[warp - 1] : 0.f);
  *total = warp_tot[kSampleThreads / 32 - 1];
  __syncthreads();  // warp_tot is reused by the next call
  return r;
}

template <typename E>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(SampleArgs a, int seg) {
  constexpr int kWarps = kSampleThreads / 32;
  __shared__ float s_m[kWarps], s_s[kWarps], s_scan[32];
  __shared__ float s_incl[kSampleThreads];  // inclusive prefixes of the ranges' weights
  __shared__ int s_i[kWarps];
  __shared__ uint32_t s_part[2];            // this segment's (max, sum) or (first max, its index), for the peers
  __shared__ float s_row[4];                // row max, this segment's interval, total
  __shared__ int s_fb;                      // last segment with weight (or 0)
  __shared__ int s_token, s_last;
  pdl_wait();  // the logits, temperatures and uniforms are complete
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t S = cluster_size(), rank = cluster_rank();
  const int i = blockIdx.x / S;
  const int V = a.vocab;
  const E* row = static_cast<const E*>(a.logits) + (int64_t)i * V;
  const int q_lo = min(V, (int)rank * seg), q_hi = min(V, q_lo + seg);  // this CTA's segment
  // every thread owns one contiguous range of the segment, in index order, of a multiple of 8
  // elements (16-byte aligned: rows are, the vocabulary being a multiple of 8 or 4, and so is
  // the segment size)
  const int per = ((seg + kSampleThreads - 1) / kSampleThreads + 7) / 8 * 8;
  const int k_lo = min(q_hi, q_lo + tid * per), k_hi = min(q_hi, k_lo + per);
  // the range's first kFirst logits (five vector loads: the whole range of a 151,936-token
  // vocabulary over 8 CTAs) go out before the checks: reads inside the row, used only when the
  // call is valid and the question live; longer ranges continue 32 at a time
  constexpr int kFirst = 40;
  float f0[kFirst];
#pragma unroll
  for (int v = 0; v < kFirst / 8; ++v) load8<E>(row, k_lo + 8 * v, k_hi, f0 + 8 * v);
  bool bad = false;
  for (int j = tid; j < a.n; j += blockDim.x) {
    if (!a.active[j]) continue;
    const float t = a.temperature[j], u = a.uniforms[j];
    bad |= !(t >= 0.f) || isinf(t) || !(u >= 0.f) || !(u < 1.f);
  }
  // the same answer in every CTA: whole clusters leave together
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) set_status(a.dev_status, ST_SAMPLING);
    return;
  }
  if (!a.active[i]) return;  // the whole cluster
  const float T = a.temperature[i];

  if (T == 0.f) {  // greedy: the first maximum
    float best = -INFINITY;
    int bi = V;
    auto scan = [&](const auto& f, int k0) {
      constexpr int N = sizeof(f) / sizeof(float);
#pragma unroll
      for (int e = 0; e < N; ++e)
        if (f[e] > best) {  // k increases per thread: the first maximum of this thread
          best = f[e];
          bi = k0 + e;
        }
    };
    scan(f0, k_lo);
    for (int k0 = k_lo + kFirst; k0 < k_hi; k0 += 32) {
      float f[32];
#pragma unroll
      for (int v = 0; v < 4; ++v) load8<E>(row, k0 + 8 * v, k_hi, f + 8 * v);
      scan(f, k0);
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
      for (int w = 1; w < kWarps; ++w)
        if (s_m[w] > b || (s_m[w] == b && s_i[w] < bk)) {
          b = s_m[w];
          bk = s_i[w];
        }
      s_part[0] = __float_as_uint(b);
      s_part[1] = (uint32_t)bk;
    }
    cluster_sync_all();
    if (rank == 0 && tid == 0) {  // segments in index order: a later one wins only when larger
      float b = -INFINITY;
      int bk = V;
      for (uint32_t r = 0; r < S; ++r) {
        const float br = __uint_as_float(ld_peer_u32(&s_part[0], r));
        const int kr = (int)ld_peer_u32(&s_part[1], r);
        if (br > b || (br == b && kr < bk)) {
          b = br;
          bk = kr;
        }
      }
      a.tokens[i] = bk < V ? bk : 0;
    }
    cluster_sync_all();  // the peers keep their shared memory until rank 0 has read it
    return;
  }

  const float inv_t = 1.0f / T;
  // max and sum of exp(z - max) over the range, 32 logits at a time
  float m = -INFINITY, s = 0.f;
  auto accumulate = [&](auto& f) {
    constexpr int N = sizeof(f) / sizeof(float);
    float bm = -INFINITY;
#pragma unroll
    for (int e = 0; e < N; ++e) {
      f[e] *= inv_t;
      bm = fmaxf(bm, f[e]);
    }
    if (bm > m) {
      s = m == -INFINITY ? 0.f : s * expf(m - bm);
      m = bm;
    }
    float add = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) add += expf(f[e] - m);  // exp(-inf) = 0 past the range
    s += add;
  };
  accumulate(f0);
  for (int k0 = k_lo + kFirst; k0 < k_hi; k0 += 32) {
    float f[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) load8<E>(row, k0 + 8 * v, k_hi, f + 8 * v);  // four loads in flight
    accumulate(f);
  }
  float bm = m, bs = s;  // the segment's max and sum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ms_combine(bm, bs, __shfl_down_sync(0xffffffffu, bm, o), __shfl_down_sync(0xffffffffu, bs, o));
  if (lane == 0) {
    s_m[warp] = bm;
    s_s[warp] = bs;
  }
  __syncthreads();
  if (tid == 0) {
    float mm = s_m[0], ss = s_s[0];
    for (int w = 1; w < kWarps; ++w) ms_combine(mm, ss, s_m[w], s_s[w]);
    s_part[0] = __float_as_uint(mm);
    s_part[1] = __float_as_uint(ss);
    s_token = INT_MAX;
  }
  cluster_sync_all();
  if (warp == 0) {
    // lane r < S: segment r's (max, sum); the row max, the segments' weights relative to it and
    // their inclusive prefix, by the same instructions on the same values in every CTA
    float mr = -INFINITY, sr = 0.f;
    if (lane < (int)S) {
      mr = __uint_as_float(ld_peer_u32(&s_part[0], lane));
      sr = __uint_as_float(ld_peer_u32(&s_part[1], lane));
    }
    float mx = mr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float w = mr == -INFINITY ? 0.f : sr * expf(mr - mx);
    float incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    const unsigned has = __ballot_sync(0xffffffffu, w > 0.f);
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == (int)rank) {
      s_row[1] = rank > 0 ? excl : 0.f;
      s_row[2] = incl;
    }
    if (lane == 0) {
      s_row[0] = mx;
      s_row[3] = total;
      s_fb = has ? 31 - __clz(has) : 0;
    }
  }
  cluster_sync_all();  // every CTA has read its peers' parts: none reads another's shared memory after this
  const float mx = s_row[0], seg_excl = s_row[1], seg_incl = s_row[2], total = s_row[3];
  const float target = a.uniforms[i] * total;
  // the segment whose interval holds the target (one at most, the intervals being contiguous);
  // none when rounding leaves the target at or above the total: then the last segment with weight
  const bool claim = seg_excl <= target && target < seg_incl;
  const bool fallback = !(target < total) && (int)rank == s_fb;
  if (!claim && !fallback) return;
  const float t_in = claim ? target - seg_excl : INFINITY;

  // this segment's ranges relative to the row max, then one scan: thread t covers
  // [excl_t, incl_t) of the segment's cumulative weight, excl_t being thread t-1's incl itself
  const float local = m == -INFINITY ? 0.f : s * expf(m - mx);
  float seg_total;
  s_incl[tid] = block_scan(local, s_scan, &seg_total);
  __syncthreads();
  const float incl = s_incl[tid];
  const float excl = tid > 0 ? s_incl[tid - 1] : 0.f;
  // the crossing is in one thread's range: that thread's warp walks the range together, one
  // vector of 8 per lane in a pass, then a warp scan finds the lane and the element
  const bool mine = excl <= t_in && t_in < incl;
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
      const bool cross = before + lsum > t_in && k0 < r_hi;
      const unsigned hits = __ballot_sync(0xffffffffu, cross);
      if (hits) {
        const int hl = __ffs(hits) - 1;
        if (lane == hl) {
          float c = before;
          int t = min(k0 + 7, r_hi - 1);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            c += w[e];
            if (c > t_in) {
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
  if (s_token == INT_MAX) {  // no crossing in the segment (rounding, or the fallback): its last element with weight
    if (tid == 0) s_last = q_lo;
    __syncthreads();
    for (int k = k_hi - 1; k >= k_lo; --k)
      if (expf(to_f(row[k]) * inv_t - mx) > 0.f) {
        atomicMax(&s_last, k);
        break;
      }
    __syncthreads();
    if (tid == 0) a.tokens[i] = s_last < V ? s_last : 0;
    return;
  }
  if (tid == 0) a.tokens[i] = s_token;
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s) {
  auto kern = a.elem == 2 ? sample_kernel<__nv_bfloat16> : sample_kernel<float>;
  // S CTAs per question, so that a thread has about 32 logits or more; segments of a multiple
  // of 8 logits
  const int S = std::min(kMaxCluster, std::max(1, (a.vocab + kSampleThreads * 32 - 1) / (kSampleThreads * 32)));
  const int seg = ((a.vocab + S - 1) / S + 7) / 8 * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n * S);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, seg);
}

}  // namespace kev
