// Decode step over the KV slot pool: compaction, append, split-K attention, fixed-order merge.
//
// Decode with a cache (inference-engine notes, sakurs2.com, §2.2): only K/V are cached; the
// new row is appended at position n = lens_i and the new query attends to all n + 1
// positions, no mask.  Early stop (Kev pipeline article, gsyq.cn news 368355, §1.2, §2.3):
// a question with active[i] == 0 is removed from the step -- it contributes no work item,
// so its slot is neither read nor written.
//
// One launch.  Every CTA first runs the same prologue over the N questions (validation,
// per-question chunk counts, prefix sum of work items: the compacted list of live
// (question, kv-head, chunk) items), so no second launch or grid-wide wait is needed.
// Items are chunks of kDecodeChunk positions of one (question, kv head); a CTA computes
// the partial (m, l, o) of all G q-heads of the group for its chunk.  When a (question,
// kv head) has several chunks, the CTA that arrives last (atomic counter) merges the
// partials in chunk order, so the result does not depend on timing.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kGMax = 16;

struct DecodeSmem {
  int item_base[kMaxQuestions + 1];  // prefix of work items over questions (dropped: 0 items)
  int hash[2 * kMaxQuestions];       // live slot ids, open addressing
  float q[kGMax][128];               // the group's queries in fp32
  float wm[kWarps][kGMax];
  float wl[kWarps][kGMax];
  float wo[kWarps][kGMax][128];
  int flags;
  int scan_tmp[kWarps + 1];
  int last;
};

__device__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base += tmp[w];
    tot += tmp[w];
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

template <typename T>
__device__ __forceinline__ const T* kv_row_ptr(const DecodeArgs& a, const void* pool, const void* fresh, int slot,
                                               int g, int pos, int n, int i, int D) {
  if (pos == n) return static_cast<const T*>(fresh) + ((int64_t)i * a.h_kv + g) * D;
  return static_cast<const T*>(pool) + (((int64_t)slot * a.h_kv + g) * a.cap + pos) * D;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
  constexpr int PER = D / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DecodeSmem& S = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n, G = a.group;

  // ---- prologue: validation (live questions only) ------------------------------------
  int hs = 1;
  while (hs < 2 * n) hs <<= 1;
  if (tid == 0) S.flags = 0;
  for (int j = tid; j < hs; j += kThreads) S.hash[j] = -1;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    if (!a.active[i]) continue;
    const int slot = a.slot_ids[i];
    const int len = a.lens[i];
    if (slot < 0 || slot >= a.n_slots) { atomicOr(&S.flags, 1); continue; }
    if (len < 0 || len >= a.cap) atomicOr(&S.flags, 2);
    unsigned h = ((unsigned)slot * 2654435761u) & (unsigned)(hs - 1);
    for (int probe = 0; probe < hs; ++probe) {
      const int prev = atomicCAS(&S.hash[h], -1, slot);
      if (prev == -1) break;
      if (prev == slot) { atomicOr(&S.flags, 4); break; }
      h = (h + 1) & (unsigned)(hs - 1);
    }
  }
  __syncthreads();
  const int f = S.flags;
  const int code = (f & 1) ? ST_SLOT : (f & 2) ? ST_OVERFLOW : (f & 4) ? ST_SLOT : ST_OK;
  if (blockIdx.x == 0 && tid == 0 && a.dev_status) *a.dev_status = code;
  if (code != ST_OK) return;

  // ---- compacted work list: items of live questions only -----------------------------
  int running = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + tid;
    int cnt = 0;
    if (i < n && a.active[i]) cnt = a.h_kv * ((a.lens[i] + 1 + kDecodeChunk - 1) / kDecodeChunk);
    int tot;
    const int off = block_exclusive_scan(cnt, S.scan_tmp, &tot);
    if (i < n) S.item_base[i] = running + off;
    running += tot;
  }
  if (tid == 0) S.item_base[n] = running;
  __syncthreads();
  const int total_items = running;

  int* counters = reinterpret_cast<int*>(a.ws + a.layout.counters);
  float* partials = reinterpret_cast<float*>(a.ws + a.layout.partials);
  const int pstride = G * (D + 2);

  for (int it = blockIdx.x; it < total_items; it += gridDim.x) {
    // question owning item `it`: item_base[i] <= it < item_base[i+1]
    int lo = 0, hi = n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (S.item_base[mid] <= it) lo = mid; else hi = mid;
    }
    const int i = lo;
    const int len = a.lens[i];
    const int slot = a.slot_ids[i];
    const int nch = (len + 1 + kDecodeChunk - 1) / kDecodeChunk;
    const int r = it - S.item_base[i];
    const int g = r / nch, c = r % nch;
    const int p0 = c * kDecodeChunk, p1 = min(p0 + kDecodeChunk, len + 1);

    // queries of the group's q-heads, fp32
    const T* qsrc = static_cast<const T*>(a.q_new) + ((int64_t)i * a.h_q + (int64_t)g * G) * D;
    for (int e = tid; e < G * D; e += kThreads) S.q[e / D][e % D] = to_f32(qsrc[e]);
    // append the new row (only the chunk that holds position len does it)
    if (p0 <= len && len < p1) {
      const int64_t dst = (((int64_t)slot * a.h_kv + g) * a.cap + len) * D;
      const int64_t src = ((int64_t)i * a.h_kv + g) * D;
      for (int e = tid; e < D; e += kThreads) {
        static_cast<T*>(a.pool_k)[dst + e] = static_cast<const T*>(a.k_new)[src + e];
        static_cast<T*>(a.pool_v)[dst + e] = static_cast<const T*>(a.v_new)[src + e];
      }
    }
    __syncthreads();

    float m[kGMax], l[kGMax], acc[kGMax][PER];
#pragma unroll
    for (int gg = 0; gg < kGMax; ++gg) {
      m[gg] = -INFINITY;
      l[gg] = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[gg][e] = 0.f;
    }
    for (int b0 = p0 + warp * 32; b0 < p1; b0 += kWarps * 32) {
      const int pos = b0 + lane;
      const bool valid = pos < p1;
      float s[kGMax];
#pragma unroll
      for (int gg = 0; gg < kGMax; ++gg) s[gg] = 0.f;
      if (valid) {
        const T* kr = kv_row_ptr<T>(a, a.pool_k, a.k_new, slot, g, pos, len, i, D);
        for (int cidx = 0; cidx < D; ++cidx) {
          const float kv = to_f32(kr[cidx]);
#pragma unroll
          for (int gg = 0; gg < kGMax; ++gg)
            if (gg < G) s[gg] = fmaf(S.q[gg][cidx], kv, s[gg]);
        }
      }
      float p[kGMax];
#pragma unroll
      for (int gg = 0; gg < kGMax; ++gg) {
        if (gg < G) {
          const float sc = valid ? s[gg] * a.scale : -INFINITY;
          const float m_new = fmaxf(m[gg], warp_max(sc));
          const float alpha = expf(m[gg] - m_new);
          p[gg] = valid ? expf(sc - m_new) : 0.f;
          l[gg] = l[gg] * alpha + warp_sum(p[gg]);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[gg][e] *= alpha;
          m[gg] = m_new;
        }
      }
      const int nk = min(32, p1 - b0);
      for (int j = 0; j < nk; ++j) {
        const T* vr = kv_row_ptr<T>(a, a.pool_v, a.v_new, slot, g, b0 + j, len, i, D) + lane * PER;
        float vv[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) vv[e] = to_f32(vr[e]);
#pragma unroll
        for (int gg = 0; gg < kGMax; ++gg) {
          if (gg < G) {
            const float pj = __shfl_sync(0xffffffffu, p[gg], j);
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[gg][e] = fmaf(pj, vv[e], acc[gg][e]);
          }
        }
      }
    }
    // combine the warps of the CTA
#pragma unroll
    for (int gg = 0; gg < kGMax; ++gg) {
      if (gg < G) {
        if (lane == 0) {
          S.wm[warp][gg] = m[gg];
          S.wl[warp][gg] = l[gg];
        }
#pragma unroll
        for (int e = 0; e < PER; ++e) S.wo[warp][gg][lane * PER + e] = acc[gg][e];
      }
    }
    __syncthreads();
    float* part = partials + (((int64_t)i * a.h_kv + g) * a.layout.max_chunks + c) * pstride;
    for (int e = tid; e < G * D; e += kThreads) {
      const int gg = e / D, dd = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, S.wm[w][gg]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sc = expf(S.wm[w][gg] - M);  // warps that saw no position: exp(-inf) = 0
        L += S.wl[w][gg] * sc;
        O += S.wo[w][gg][dd] * sc;
      }
      if (nch == 1) {
        static_cast<T*>(a.out)[((int64_t)i * a.h_q + (int64_t)g * G + gg) * D + dd] = from_f32<T>(O / L);
      } else {
        part[gg * D + dd] = O;
        if (dd == 0) {
          part[G * D + gg] = M;
          part[G * D + G + gg] = L;
        }
      }
    }
    if (nch > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(&counters[i * a.h_kv + g], 1);
        S.last = (prev == nch - 1);
      }
      __syncthreads();
      if (S.last) {
        __threadfence();
        const float* base = partials + ((int64_t)i * a.h_kv + g) * a.layout.max_chunks * pstride;
        for (int e = tid; e < G * D; e += kThreads) {
          const int gg = e / D, dd = e % D;
          float M = -INFINITY;
          for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(base + cc * pstride + G * D + gg));
          float L = 0.f, O = 0.f;
          for (int cc = 0; cc < nch; ++cc) {
            const float* pc = base + cc * pstride;
            const float sc = expf(__ldcg(pc + G * D + gg) - M);
            L += __ldcg(pc + G * D + G + gg) * sc;
            O += __ldcg(pc + gg * D + dd) * sc;
          }
          static_cast<T*>(a.out)[((int64_t)i * a.h_q + (int64_t)g * G + gg) * D + dd] = from_f32<T>(O / L);
        }
        if (tid == 0) counters[i * a.h_kv + g] = 0;
      }
    }
    __syncthreads();
  }
}

__global__ void advance_kernel(int32_t* lens, const uint8_t* active, int32_t n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && active[i]) lens[i] += 1;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int d, kev_dtype dt, int num_sms, cudaStream_t s) {
  const size_t smem = sizeof(DecodeSmem);
  const int grid = num_sms * 2;
  cudaError_t e = cudaSuccess;
  if (dt == KEV_FP32) {
    if (d == 64) {
      e = cudaFuncSetAttribute(decode_kernel<float, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_kernel<float, 64><<<grid, kThreads, smem, s>>>(a);
    } else {
      e = cudaFuncSetAttribute(decode_kernel<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_kernel<float, 128><<<grid, kThreads, smem, s>>>(a);
    }
  } else {
    if (d == 64) {
      e = cudaFuncSetAttribute(decode_kernel<__nv_bfloat16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_kernel<__nv_bfloat16, 64><<<grid, kThreads, smem, s>>>(a);
    } else {
      e = cudaFuncSetAttribute(decode_kernel<__nv_bfloat16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_kernel<__nv_bfloat16, 128><<<grid, kThreads, smem, s>>>(a);
    }
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_advance(int32_t* lens, const uint8_t* active, int32_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  advance_kernel<<<(n + 255) / 256, 256, 0, s>>>(lens, active, n);
  return cudaGetLastError();
}

}  // namespace kev
