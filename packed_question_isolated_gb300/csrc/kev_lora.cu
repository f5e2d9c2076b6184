// Token-grouped LoRA: the low-rank delta of each question's adapter on that question's tokens.
//
// Kev architecture article (icman.com.cn), §3.2: the base layer stays fixed and each token takes
// the delta of the adapter of the question it belongs to; rather than running every adapter over
// the whole sequence and masking, tokens are processed per adapter group.  §3.3: the scale is the
// adapter's alpha / rank.  For token t of question i with adapter a = adapter_ids[i] >= 0:
//   y[t] += scale_a * B_a (A_a x[t]),   A_a: [r, d_in], B_a: [d_out, r]   (bf16, fp32 accumulation)
// A question's tokens are contiguous in the packed batch, so a tile of its rows is one adapter
// group with no gather or scatter.
//
// lora_kernel: a CTA takes 16 consecutive rows of one question, tiles in cu_seqlens order from the
// segment builder's work list; its 4 warps split d_in for h (partial sums added through shared
// memory) and d_out for y, loading the y and B_a fragments of 8 n-tiles before the MMAs (y is
// read and written in place, so later loads could not move above earlier stores).  With rank 16 the op reads x and reads
// and writes y for ~10 FLOPs per byte, so it is HBM-bound; the two products run on the warp-level
// tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate), fragments straight from global memory:
//   h [16 x r] = x [16 x d_in] . A_a^T      (A_a's rows are the MMA's column-major B operand)
//   y [16 x d_out] += scale h . B_a^T        (h's fp32 accumulator fragments are, pair by pair,
//                                             the bf16 A operand of the second MMA; C = y)
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kLoraWarps = 4;
constexpr int kLoraRows = 16;  // rows per CTA tile: the 4 warps split d_in, then d_out
constexpr int kNBatch = 8;     // n-tiles of y a warp loads before it multiplies and stores

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 f2_of(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ int question_of(const int32_t* cu, int n, int r) {
  int lo = 0, hi = n;  // cu[lo] <= r < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

template <int R>  // rank: a multiple of 16
__global__ void __launch_bounds__(32 * kLoraWarps) lora_kernel(LoraArgs a) {
  extern __shared__ int32_t s_tiles[];  // [n + 1] exclusive prefix of each question's tile count
  __shared__ int s_scan[33];
  __shared__ int s_ok;
  pdl_wait();  // the segment builder's work list, x and y are complete
  pdl_trigger();
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(a.ws);
  const int32_t* cu = reinterpret_cast<const int32_t*>(a.ws + a.layout.cu_seqlens);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_ok = hdr->status == ST_OK;
  // every block checks every adapter id first: an invalid call writes nothing
  bool bad = false;
  for (int i = tid; i < a.n; i += blockDim.x) bad |= a.adapter_ids[i] < -1 || a.adapter_ids[i] >= a.n_adapters;
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) set_status(a.dev_status, ST_ADAPTER);
    return;
  }
  if (!s_ok) return;
  // tiles of questions with an adapter, in question order: s_tiles[i] = first tile of question i
  int running = 0;
  for (int base = 0; base < a.n; base += blockDim.x) {
    const int i = base + tid;
    const int cnt = i < a.n && a.adapter_ids[i] >= 0 ? (cu[i + 1] - cu[i] + kLoraRows - 1) / kLoraRows : 0;
    int x = cnt;  // block scan (4 warps)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    int off = 0;
    for (int w = 0; w < warp; ++w) off += s_scan[w];
    if (i < a.n) s_tiles[i] = running + off + x - cnt;
    int tot = 0;
    for (int w = 0; w < kLoraWarps; ++w) tot += s_scan[w];
    __syncthreads();
    running += tot;
  }
  if (tid == 0) s_tiles[a.n] = running;
  __syncthreads();
  const int n_tiles = s_tiles[a.n];

  __shared__ float s_h[kLoraWarps][16][R + 1];  // partial h of each warp (padded rows)
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.x);
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.y);
  const int g = lane >> 2, c2 = (lane & 3) * 2;  // fragment row / column pair of this lane
  const int k_span = a.d_in / kLoraWarps, n_span = a.d_out / kLoraWarps;  // host: multiples of 16 / 8
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int i = question_of(s_tiles, a.n, t);  // s_tiles is a prefix like cu_seqlens
    const int ad = a.adapter_ids[i];
    const kev_interval iv = a.intervals[i];
    const int r0 = iv.begin + (t - s_tiles[i]) * kLoraRows;
    const int rows = min(kLoraRows, iv.end - r0);
    const bool ok0 = g < rows, ok1 = g + 8 < rows;
    const __nv_bfloat16* x0 = X + (int64_t)(r0 + g) * a.d_in;
    const __nv_bfloat16* x1 = X + (int64_t)(r0 + g + 8) * a.d_in;
    const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(a.lora_a) + (int64_t)ad * R * a.d_in;
    const __nv_bfloat16* B = static_cast<const __nv_bfloat16*>(a.lora_b) + (int64_t)ad * a.d_out * R;

    // partial h = x . A^T over this warp's share of d_in: R / 8 accumulator tiles of 16 x 8
    float h[R / 8][4];
#pragma unroll
    for (int n = 0; n < R / 8; ++n) h[n][0] = h[n][1] = h[n][2] = h[n][3] = 0.f;
    const int k_beg = warp * k_span, k_end = k_beg + k_span;
#pragma unroll 4
    for (int k0 = k_beg; k0 < k_end; k0 += 16) {
      uint32_t af[4];
      af[0] = ok0 ? __ldg(reinterpret_cast<const uint32_t*>(x0 + k0 + c2)) : 0u;
      af[1] = ok1 ? __ldg(reinterpret_cast<const uint32_t*>(x1 + k0 + c2)) : 0u;
      af[2] = ok0 ? __ldg(reinterpret_cast<const uint32_t*>(x0 + k0 + 8 + c2)) : 0u;
      af[3] = ok1 ? __ldg(reinterpret_cast<const uint32_t*>(x1 + k0 + 8 + c2)) : 0u;
#pragma unroll
      for (int n = 0; n < R / 8; ++n) {
        const __nv_bfloat16* arow = A + (int64_t)(n * 8 + g) * a.d_in + k0;  // rank n*8+g
        uint32_t bf[2];
        bf[0] = __ldg(reinterpret_cast<const uint32_t*>(arow + c2));
        bf[1] = __ldg(reinterpret_cast<const uint32_t*>(arow + 8 + c2));
        mma_bf16_16816(h[n], af, bf);
      }
    }
#pragma unroll
    for (int n = 0; n < R / 8; ++n) {
      s_h[warp][g][n * 8 + c2] = h[n][0];
      s_h[warp][g][n * 8 + c2 + 1] = h[n][1];
      s_h[warp][g + 8][n * 8 + c2] = h[n][2];
      s_h[warp][g + 8][n * 8 + c2 + 1] = h[n][3];
    }
    __syncthreads();
#pragma unroll
    for (int n = 0; n < R / 8; ++n) {  // every warp: the whole h, summed in a fixed order
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kLoraWarps; ++w) {
        v[0] += s_h[w][g][n * 8 + c2];
        v[1] += s_h[w][g][n * 8 + c2 + 1];
        v[2] += s_h[w][g + 8][n * 8 + c2];
        v[3] += s_h[w][g + 8][n * 8 + c2 + 1];
      }
      h[n][0] = v[0];
      h[n][1] = v[1];
      h[n][2] = v[2];
      h[n][3] = v[3];
    }
    __syncthreads();  // s_h is rewritten by the next tile
    // h (scaled) as the bf16 A operand of y += h . B^T: k-step j takes accumulator tiles 2j, 2j+1
    const float sc = a.scales[ad];
    uint32_t hf[R / 16][4];
#pragma unroll
    for (int j = 0; j < R / 16; ++j) {
      hf[j][0] = bf16x2_of(sc * h[2 * j][0], sc * h[2 * j][1]);
      hf[j][1] = bf16x2_of(sc * h[2 * j][2], sc * h[2 * j][3]);
      hf[j][2] = bf16x2_of(sc * h[2 * j + 1][0], sc * h[2 * j + 1][1]);
      hf[j][3] = bf16x2_of(sc * h[2 * j + 1][2], sc * h[2 * j + 1][3]);
    }
    __nv_bfloat16* y0 = Y + (int64_t)(r0 + g) * a.d_out;
    __nv_bfloat16* y1 = Y + (int64_t)(r0 + g + 8) * a.d_out;
    const int n_beg = warp * n_span, n_end = n_beg + n_span;
    for (int nb = n_beg; nb < n_end; nb += 8 * kNBatch) {
      uint32_t yv[kNBatch][2], bv[kNBatch][R / 16][2];
#pragma unroll
      for (int q = 0; q < kNBatch; ++q) {  // every load of the batch first
        const int n0 = nb + 8 * q;
        if (n0 < n_end) {
          yv[q][0] = ok0 ? *reinterpret_cast<const uint32_t*>(y0 + n0 + c2) : 0u;
          yv[q][1] = ok1 ? *reinterpret_cast<const uint32_t*>(y1 + n0 + c2) : 0u;
          const __nv_bfloat16* brow = B + (int64_t)(n0 + g) * R;  // output column n0+g
#pragma unroll
          for (int j = 0; j < R / 16; ++j) {
            bv[q][j][0] = __ldg(reinterpret_cast<const uint32_t*>(brow + 16 * j + c2));
            bv[q][j][1] = __ldg(reinterpret_cast<const uint32_t*>(brow + 16 * j + 8 + c2));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kNBatch; ++q) {
        const int n0 = nb + 8 * q;
        if (n0 >= n_end) break;
        const float2 u0 = f2_of(yv[q][0]), u1 = f2_of(yv[q][1]);
        float acc[4] = {u0.x, u0.y, u1.x, u1.y};
#pragma unroll
        for (int j = 0; j < R / 16; ++j) mma_bf16_16816(acc, hf[j], bv[q][j]);
        if (ok0) *reinterpret_cast<uint32_t*>(y0 + n0 + c2) = bf16x2_of(acc[0], acc[1]);
        if (ok1) *reinterpret_cast<uint32_t*>(y1 + n0 + c2) = bf16x2_of(acc[2], acc[3]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_lora(const LoraArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = sizeof(int32_t) * (size_t)(a.n + 1);
  auto kern = a.rank == 16 ? lora_kernel<16> : a.rank == 32 ? lora_kernel<32> : lora_kernel<64>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3(num_sms * 8), dim3(32 * kLoraWarps), smem, s, a);
}

}  // namespace kev
