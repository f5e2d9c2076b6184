// Rotary position encoding with positions counted per question.
//
// KV-cache isolation article (hnwysp.cn, news 130224), §7.2: the rotation multiplies Q and K,
// the cache holds K after its rotation, and a new token's position is the cache length counted
// from 0.  Packed with isolation, every question counts its positions from 0 as it would alone:
// token t of question i has position t - begin_i, and the decode token of question i position
// lens_i.  Rotate-half form: element j < d/2 of a head pairs with element j + d/2 and the pair
// (a, b) turns by the angle p * w_j, w_j = theta^(-2j/d): (a cos - b sin, b cos + a sin).
//
// rope_table_kernel     cos/sin of every (position, j) in double precision, stored as floats
//                       (computed once, then read from L2 by the two kernels below).
// rope_prefill_kernel   one thread per 16-byte chunk pair (chunk c of the first half of a head
//                       row with chunk c of the second half) of the q-heads and kv-heads of a
//                       question token, in cu_seqlens order (the question found by binary
//                       search in shared memory), rotated in place; with a slot pool the rotated
//                       K chunks and the V row also go into the question's slot (the slot write,
//                       fused into the same pass).  HBM-bound: q, k and v are read once, q and k
//                       written once, the slot rows written once.
// rope_decode_kernel    the same rotation of q_new / k_new rows of live questions at lens_i.
//
// A position past the table (a question longer than max_pos, a live lens_i >= max_pos) is a
// data error found before anything is written: every block checks every question first.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kRopeThreads = 256;

__device__ __forceinline__ void unpack(uint4 v, float* f, __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unpack(uint4 v, float* f, float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack(const float* f, __nv_bfloat16*) {
  return make_uint4(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3]), bf16x2_rn(f[4], f[5]), bf16x2_rn(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack(const float* f, float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

// The rotation of one chunk pair held in registers (va: first-half chunk, vb: second-half chunk);
// cs = the table's cos/sin of those j at this position.
template <typename E>
__device__ __forceinline__ void rotate_regs(uint4& va, uint4& vb, const float2* __restrict__ cs) {
  constexpr int EV = 16 / sizeof(E);
  float a[EV], b[EV], ra[EV], rb[EV];
  unpack(va, a, static_cast<E*>(nullptr));
  unpack(vb, b, static_cast<E*>(nullptr));
  const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int e = 0; e < EV; e += 2) {
    const float4 t = __ldg(cs4 + e / 2);  // {cos_j, sin_j, cos_j+1, sin_j+1}
    ra[e] = a[e] * t.x - b[e] * t.y;
    rb[e] = b[e] * t.x + a[e] * t.y;
    ra[e + 1] = a[e + 1] * t.z - b[e + 1] * t.w;
    rb[e + 1] = b[e + 1] * t.z + a[e + 1] * t.w;
  }
  va = pack(ra, static_cast<E*>(nullptr));
  vb = pack(rb, static_cast<E*>(nullptr));
}

// Rotates chunk c of one head row in place: elements [c*EV, c*EV + EV) of the first half with
// the same elements of the second half.
template <typename E>
__device__ __forceinline__ void rotate_chunk(E* __restrict__ row, int c, int half, const float2* __restrict__ cs) {
  constexpr int EV = 16 / sizeof(E);
  uint4* pa = reinterpret_cast<uint4*>(row + c * EV);
  uint4* pb = reinterpret_cast<uint4*>(row + half + c * EV);
  uint4 va = *pa, vb = *pb;
  rotate_regs<E>(va, vb, cs + c * EV);
  *pa = va;
  *pb = vb;
}

__device__ __forceinline__ int question_of(const int32_t* cu, int n, int r) {
  int lo = 0, hi = n;  // cu[lo] <= r < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void rope_table_kernel(float2* table, int64_t count, int half, int d, double theta) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= count) return;
  const int p = (int)(idx / half), j = (int)(idx % half);
  const double w = pow(theta, -2.0 * j / d);
  double s, c;
  sincos((double)p * w, &s, &c);
  table[idx] = make_float2((float)c, (float)s);
}

template <typename E>
__global__ void __launch_bounds__(kRopeThreads) rope_prefill_kernel(RopePrefillArgs a) {
  extern __shared__ int32_t s_cu[];                                // [n + 1]
  int2* s_bs = reinterpret_cast<int2*>(s_cu + ((a.n + 2) & ~1));  // [n] {begin, slot}
  __shared__ int s_ok;
  pdl_wait();  // the segment builder's results and the producers of q, k, v are complete
  pdl_trigger();
  PrefillHeader* hdr = reinterpret_cast<PrefillHeader*>(const_cast<char*>(a.ws));
  const int32_t* cu = reinterpret_cast<const int32_t*>(a.ws + a.layout.cu_seqlens);
  if (threadIdx.x == 0) s_ok = hdr->status == ST_OK;
  for (int i = threadIdx.x; i <= a.n; i += blockDim.x) s_cu[i] = cu[i];
  for (int i = threadIdx.x; i < a.n; i += blockDim.x)
    s_bs[i] = make_int2(a.intervals[i].begin, a.slot_ids ? a.slot_ids[i] : -1);
  __syncthreads();
  if (!s_ok) return;
  bool bad = false;  // a question longer than the table: nothing is written by this call
  for (int i = threadIdx.x; i < a.n; i += blockDim.x) bad |= s_cu[i + 1] - s_cu[i] > a.max_pos;
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      atomicCAS(&hdr->status, ST_OK, ST_POSITION);  // the attention and slot-write kernels after this one skip
      set_status(a.dev_status, ST_POSITION);
    }
    return;
  }

  // one task per thread: a chunk pair of one head row of a token (rotation in place; the
  // rotated K chunk also to the slot), or, with a slot pool, one 16-byte vector of the token's
  // V row to the slot.  Consecutive threads take consecutive chunks of one token.
  constexpr int EV = 16 / sizeof(E);
  const int half = a.d / 2;
  const int vh = half / EV;   // chunk pairs per head row
  const int vrow = a.d / EV;  // 16-byte vectors per head row
  const int rot = (a.h_q + a.h_kv) * vh;
  const int per_row = rot + (a.slot_ids ? a.h_kv * vrow : 0);
  const int64_t tasks = (int64_t)s_cu[a.n] * per_row;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < tasks; u += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(u / per_row), w = (int)(u % per_row);
    const int i = question_of(s_cu, a.n, r);
    const int j = r - s_cu[i];  // position inside the question
    const int2 bs = s_bs[i];
    const int64_t t = bs.x + j;  // packed token
    const bool to_slot = bs.y >= 0 && bs.y < a.n_slots && j < a.cap;  // (the segment builder checked them)
    if (w < rot) {
      const int h = w / vh, c = w % vh;
      E* row;
      E* prow = nullptr;
      if (h < a.h_q) {
        row = static_cast<E*>(a.q) + (t * a.h_q + h) * a.d;
      } else {
        const int g = h - a.h_q;
        row = static_cast<E*>(a.k) + (t * a.h_kv + g) * a.d;
        if (to_slot) prow = static_cast<E*>(a.pool_k) + (((int64_t)bs.y * a.h_kv + g) * a.cap + j) * a.d;
      }
      uint4* pa = reinterpret_cast<uint4*>(row + c * EV);
      uint4* pb = reinterpret_cast<uint4*>(row + half + c * EV);
      uint4 va = *pa, vb = *pb;
      rotate_regs<E>(va, vb, a.table + (int64_t)j * half + c * EV);
      *pa = va;
      *pb = vb;
      if (prow) {
        *reinterpret_cast<uint4*>(prow + c * EV) = va;
        *reinterpret_cast<uint4*>(prow + half + c * EV) = vb;
      }
    } else if (to_slot) {
      const int x = w - rot, g = x / vrow, c = x % vrow;
      static_cast<uint4*>(a.pool_v)[(((int64_t)bs.y * a.h_kv + g) * a.cap + j) * vrow + c] =
          __ldg(static_cast<const uint4*>(a.v) + (t * a.h_kv + g) * vrow + c);
    }
  }
}

template <typename E>
__global__ void __launch_bounds__(kRopeThreads) rope_decode_kernel(RopeDecodeArgs a) {
  pdl_wait();  // q_new, k_new, lens and active are as the kernels before this one left them
  pdl_trigger();
  bool bad = false;  // a live position past the table: nothing is written by this call
  for (int i = threadIdx.x; i < a.n; i += blockDim.x) bad |= a.active[i] && (a.lens[i] < 0 || a.lens[i] >= a.max_pos);
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(a.dev_status, ST_POSITION);
    return;
  }
  constexpr int EV = 16 / sizeof(E);
  const int half = a.d / 2;
  const int vh = half / EV;
  const int per_q = (a.h_q + a.h_kv) * vh;
  const int64_t tasks = (int64_t)a.n * per_q;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < tasks; u += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(u / per_q), w = (int)(u % per_q);
    if (!a.active[i]) continue;
    const int h = w / vh, c = w % vh;
    const float2* cs = a.table + (int64_t)a.lens[i] * half;
    E* row = h < a.h_q ? static_cast<E*>(a.q_new) + ((int64_t)i * a.h_q + h) * a.d
                       : static_cast<E*>(a.k_new) + ((int64_t)i * a.h_kv + (h - a.h_q)) * a.d;
    rotate_chunk<E>(row, c, half, cs);
  }
}

}  // namespace

cudaError_t launch_rope_table(float2* table, int32_t max_pos, int32_t d, double theta, cudaStream_t s) {
  const int half = d / 2;
  const int64_t count = (int64_t)max_pos * half;
  const int blocks = (int)((count + kRopeThreads - 1) / kRopeThreads);
  rope_table_kernel<<<blocks, kRopeThreads, 0, s>>>(table, count, half, d, theta);
  return cudaGetLastError();
}

cudaError_t launch_rope_prefill(const RopePrefillArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = sizeof(int32_t) * (size_t)((a.n + 2) & ~1) + sizeof(int2) * (size_t)a.n;
  auto kern = a.elem == 2 ? rope_prefill_kernel<__nv_bfloat16> : rope_prefill_kernel<float>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0;  // one resident wave: every block loops over the tasks
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRopeThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return launch_pdl(kern, dim3(num_sms * per_sm), dim3(kRopeThreads), smem, s, a);
}

cudaError_t launch_rope_decode(const RopeDecodeArgs& a, cudaStream_t s) {
  const int EV = 16 / a.elem;
  const int64_t tasks = (int64_t)a.n * (a.h_q + a.h_kv) * (a.d / 2 / EV);
  int blocks = (int)((tasks + kRopeThreads - 1) / kRopeThreads);
  if (blocks < 1) blocks = 1;
  if (blocks > 1024) blocks = 1024;
  auto kern = a.elem == 2 ? rope_decode_kernel<__nv_bfloat16> : rope_decode_kernel<float>;
  return launch_pdl(kern, dim3(blocks), dim3(kRopeThreads), 0, s, a);
}

}  // namespace kev
