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
// segment builder's work list.  With rank 16 the op reads x and reads and writes y for ~10 FLOPs
// per byte, so it is HBM-bound, and what sets its speed is the bytes in flight.  So the tile's
// operands go through shared memory as a pipeline of asynchronous 16-byte copies
// (cp.async, 3 to 6 stages by rank, waits in hardware only): first chunks of x's columns with the same
// columns of A_a, then chunks of y's columns with the rows of B_a for them.  The 4 warps split
// each chunk's 32-wide k-steps (n-blocks); the two products run on the warp-level tensor-core
// MMA (m16n8k16, bf16 in, fp32 accumulate) with fragments read from shared memory:
//   h [16 x r] = x [16 x d_in] . A_a^T      (A_a's rows are the MMA's column-major B operand;
//                                             per-warp partials summed in a fixed order)
//   y [16 x d_out] += scale h . B_a^T        (h's fp32 accumulator fragments are, pair by pair,
//                                             the bf16 A operand of the second MMA; C = y)
// The new y goes back into the stage and leaves it in 16-byte stores.  For h, lane (g, c) reads
// x and A_a at k0 + 8c .. k0 + 8c + 7 in one 16-byte load: words 0, 1 are the A / B fragment pairs
// of one MMA, words 2, 3 those of another, i.e. the MMA's k slots map to other columns than its
// fragment layout names, the same mapping for both operands of a sum over k.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kLoraWarps = 4;

// A CTA tile is kRows rows, kMT m16 MMA tiles (measured on the Qwen2.5-7B batch through a 3584 x
// 3584 rank-16 projection: 16-row tiles 55 us, 32-row tiles 65 us; half as many CTAs, each with
// twice the work per chunk, lose more than the larger share of x and y in a stage gains).
// Shared-memory stage of one chunk of 128 columns: x (or y) rows, then A_a rows (or B_a rows,
// one per output column of the chunk).  Rows of x, A_a and y are padded by 64 bytes, so the two rows
// a quarter warp reads in a 16-byte fragment load fall on different banks; B_a rows by 16 bytes,
// and placed so that the 8 a fragment load reads are consecutive (b_pos), on 8 bank groups.
template <int R>
struct LoraCfg {
  static constexpr int kRows = 16;
  static constexpr int kMT = kRows / 16;
  static constexpr int kC = 128;  // columns of x / y per chunk
  static constexpr int kStages = R == 16 ? 6 : R == 32 ? 4 : 3;
  static constexpr int kRowB = kC * 2 + 64;
  static constexpr int kBRowB = R * 2 + 16;
  static constexpr int kP1 = (kRows + R) * kRowB;
  static constexpr int kP2 = kRows * kRowB + kC * kBRowB;
  static constexpr int kStage = ((kP1 > kP2 ? kP1 : kP2) + 127) / 128 * 128;
};
// staged row of output column j of a chunk: bits 3-4 of j move to bits 1-2 and bits 1-2 to 3-4
__device__ __forceinline__ int b_pos(int j) {
  return (j & ~31) | (j & 1) | (((j >> 3) & 3) << 1) | (((j >> 1) & 3) << 3);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  // 16 bytes, or 16 zero bytes when !valid (src is not read then)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}

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
  using Cfg = LoraCfg<R>;
  constexpr int KC = Cfg::kC, NS = Cfg::kStages, ROWS = Cfg::kRows, MT = Cfg::kMT;
  extern __shared__ __align__(128) unsigned char lora_smem[];
  int32_t* s_tiles = reinterpret_cast<int32_t*>(lora_smem);  // [n + 1] first tile of each question
  const uint32_t stages = static_cast<uint32_t>(__cvta_generic_to_shared(lora_smem)) +
                          (uint32_t)(((a.n + 1) * 4 + 127) / 128 * 128);
  __shared__ int s_scan[33];
  __shared__ int s_ok;
  __shared__ float s_h[kLoraWarps][ROWS][R + 1];  // partial h of each warp (padded rows)
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
    const int cnt = i < a.n && a.adapter_ids[i] >= 0 ? (cu[i + 1] - cu[i] + ROWS - 1) / ROWS : 0;
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

  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.x);
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.y);
  const int g = lane >> 2, c = lane & 3, c2 = c * 2;  // fragment row, column quad of this lane
  const int p1 = (a.d_in + KC - 1) / KC, n_chunks = p1 + (a.d_out + KC - 1) / KC;
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int i = question_of(s_tiles, a.n, t);  // s_tiles is a prefix like cu_seqlens
    const int ad = a.adapter_ids[i];
    const kev_interval iv = a.intervals[i];
    const int r0 = iv.begin + (t - s_tiles[i]) * ROWS;
    const int rows = min(ROWS, iv.end - r0);
    const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(a.lora_a) + (int64_t)ad * R * a.d_in;
    const __nv_bfloat16* B = static_cast<const __nv_bfloat16*>(a.lora_b) + (int64_t)ad * a.d_out * R;

    // copies of chunk ci into stage ci % NS (every thread a share of its 16-byte pieces), then
    // one commit group per chunk, empty past the last one so the group count stays uniform;
    // rows past the tile's end are filled with zeros, not read
    // Thread tid copies the 16-byte column pcol of rows prow + 8u of a stage (a chunk is 128
    // columns, 16 pieces a row); its source rows are fixed for the tile, so their addresses are
    // formed once here.  Rows past the tile's end are filled with zeros, not read; columns past
    // d_in (d_out) in the last chunk are neither copied nor read.
    static_assert(KC == 128 && 32 * kLoraWarps == 128, "16 pieces a row, 8 rows a pass of the block");
    constexpr int U1 = (ROWS + R) / 8, U2 = ROWS / 8;
    const int prow = tid >> 4, pcol = (tid & 15) * 8;
    const __nv_bfloat16* src1[U1];  // x rows, then A_a rows (column pcol of chunk 0)
#pragma unroll
    for (int u = 0; u < U1; ++u) {
      const int row = prow + 8 * u;
      src1[u] = row < ROWS ? X + (int64_t)(r0 + (row < rows ? row : 0)) * a.d_in + pcol
                           : A + (int64_t)(row - ROWS) * a.d_in + pcol;
    }
    __nv_bfloat16* ysrc[U2];  // y rows (column pcol of chunk 0): copied in, and written back
#pragma unroll
    for (int u = 0; u < U2; ++u) ysrc[u] = Y + (int64_t)(r0 + (prow + 8 * u < rows ? prow + 8 * u : 0)) * a.d_out + pcol;
    auto issue = [&](int ci) {
      if (ci < n_chunks) {
        const uint32_t st = stages + (uint32_t)(ci % NS) * Cfg::kStage + prow * Cfg::kRowB + pcol * 2;
        if (ci < p1) {
          const int c0 = ci * KC;
          if (c0 + pcol < a.d_in) {
#pragma unroll
            for (int u = 0; u < U1; ++u)
              cp_async16(st + 8 * u * Cfg::kRowB, src1[u] + c0, prow + 8 * u >= ROWS || prow + 8 * u < rows);
          }
        } else {
          const int n0 = (ci - p1) * KC, nc = min(KC, a.d_out - n0);
          if (n0 + pcol < a.d_out) {
#pragma unroll
            for (int u = 0; u < U2; ++u) cp_async16(st + 8 * u * Cfg::kRowB, ysrc[u] + n0, prow + 8 * u < rows);
          }
          const uint32_t bst = stages + (uint32_t)(ci % NS) * Cfg::kStage + ROWS * Cfg::kRowB;
          for (int e = tid; e < nc * (R / 8); e += 32 * kLoraWarps) {
            const int j = e / (R / 8), part = e % (R / 8);
            cp_async16(bst + b_pos(j) * Cfg::kBRowB + part * 16, B + (int64_t)(n0 + j) * R + part * 8, true);
          }
        }
      }
      cp_async_commit();
    };

    for (int ci = 0; ci < NS - 1; ++ci) issue(ci);
    float h[MT][R / 8][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int n = 0; n < R / 8; ++n) h[m][n][0] = h[m][n][1] = h[m][n][2] = h[m][n][3] = 0.f;
    uint32_t hf[MT][R / 16][4];
    for (int ci = 0; ci < n_chunks; ++ci) {
      cp_async_wait<NS - 2>();  // this thread's copies of chunk ci have landed
      __syncthreads();          // everyone's have, and chunk ci - 1's stage is no longer read
      issue(ci + NS - 1);
      const uint32_t st = stages + (uint32_t)(ci % NS) * Cfg::kStage;
      if (ci < p1) {
        // partial h over this warp's k-steps of the chunk
        const int ksteps = min(KC, a.d_in - ci * KC) / 32;
        for (int s = warp; s < ksteps; s += kLoraWarps) {
          const uint32_t colb = (uint32_t)(32 * s + 8 * c) * 2;
          uint4 aw[R / 8];
#pragma unroll
          for (int n = 0; n < R / 8; ++n) aw[n] = lds128(st + (ROWS + n * 8 + g) * Cfg::kRowB + colb);  // rank n*8+g
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 xa = lds128(st + (16 * m + g) * Cfg::kRowB + colb);
            const uint4 xb = lds128(st + (16 * m + g + 8) * Cfg::kRowB + colb);
            const uint32_t af0[4] = {xa.x, xb.x, xa.y, xb.y};
            const uint32_t af1[4] = {xa.z, xb.z, xa.w, xb.w};
#pragma unroll
            for (int n = 0; n < R / 8; ++n) {
              const uint32_t bf0[2] = {aw[n].x, aw[n].y};
              const uint32_t bf1[2] = {aw[n].z, aw[n].w};
              mma_bf16_16816(h[m][n], af0, bf0);
              mma_bf16_16816(h[m][n], af1, bf1);
            }
          }
        }
        continue;
      }
      if (ci == p1) {  // the whole h, the warps' partials summed in a fixed order
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int n = 0; n < R / 8; ++n) {
            s_h[warp][16 * m + g][n * 8 + c2] = h[m][n][0];
            s_h[warp][16 * m + g][n * 8 + c2 + 1] = h[m][n][1];
            s_h[warp][16 * m + g + 8][n * 8 + c2] = h[m][n][2];
            s_h[warp][16 * m + g + 8][n * 8 + c2 + 1] = h[m][n][3];
          }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int n = 0; n < R / 8; ++n) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kLoraWarps; ++w) {
              v[0] += s_h[w][16 * m + g][n * 8 + c2];
              v[1] += s_h[w][16 * m + g][n * 8 + c2 + 1];
              v[2] += s_h[w][16 * m + g + 8][n * 8 + c2];
              v[3] += s_h[w][16 * m + g + 8][n * 8 + c2 + 1];
            }
            h[m][n][0] = v[0];
            h[m][n][1] = v[1];
            h[m][n][2] = v[2];
            h[m][n][3] = v[3];
          }
        __syncthreads();  // s_h is rewritten by the next tile
        // h (scaled) as the bf16 A operand of y += h . B^T: k-step j takes accumulator tiles 2j, 2j+1
        const float sc = a.scales[ad];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int j = 0; j < R / 16; ++j) {
            hf[m][j][0] = bf16x2_of(sc * h[m][2 * j][0], sc * h[m][2 * j][1]);
            hf[m][j][1] = bf16x2_of(sc * h[m][2 * j][2], sc * h[m][2 * j][3]);
            hf[m][j][2] = bf16x2_of(sc * h[m][2 * j + 1][0], sc * h[m][2 * j + 1][1]);
            hf[m][j][3] = bf16x2_of(sc * h[m][2 * j + 1][2], sc * h[m][2 * j + 1][3]);
          }
      }
      // y += h . B^T on this warp's n-blocks of the chunk, in place in the stage.  In the block at
      // n0, lane (g, c) holds y columns n0 + 8c .. n0 + 8c + 7 of rows g and g + 8 of each m-tile
      // (one 16-byte load each); MMA q (0..3) takes the pair n0 + 8c + 2q, +1 as its C slots 2c,
      // 2c + 1, so its n-slot j is column n0 + 8 (j / 2) + 2q + j % 2, staged at b_pos = n0 + j + 8q
      const int n0 = (ci - p1) * KC, nc = min(KC, a.d_out - n0);
      const uint32_t bst = st + ROWS * Cfg::kRowB;
      for (int nb = warp; nb < nc / 32; nb += kLoraWarps) {
        uint32_t wa[MT][4], wb[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint32_t y0 = st + (16 * m + g) * Cfg::kRowB + (uint32_t)(32 * nb + 8 * c) * 2;
          const uint4 ya = lds128(y0), yb = lds128(y0 + 8 * Cfg::kRowB);
          wa[m][0] = ya.x; wa[m][1] = ya.y; wa[m][2] = ya.z; wa[m][3] = ya.w;
          wb[m][0] = yb.x; wb[m][1] = yb.y; wb[m][2] = yb.z; wb[m][3] = yb.w;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t brow = bst + (uint32_t)(32 * nb + 8 * q + g) * Cfg::kBRowB;
          uint32_t bf[R / 16][2];
#pragma unroll
          for (int j = 0; j < R / 16; ++j) {
            bf[j][0] = lds32(brow + (16 * j + c2) * 2);
            bf[j][1] = lds32(brow + (16 * j + 8 + c2) * 2);
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float2 u0 = f2_of(wa[m][q]), u1 = f2_of(wb[m][q]);
            float acc[4] = {u0.x, u0.y, u1.x, u1.y};
#pragma unroll
            for (int j = 0; j < R / 16; ++j) mma_bf16_16816(acc, hf[m][j], bf[j]);
            wa[m][q] = bf16x2_of(acc[0], acc[1]);
            wb[m][q] = bf16x2_of(acc[2], acc[3]);
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint32_t y0 = st + (16 * m + g) * Cfg::kRowB + (uint32_t)(32 * nb + 8 * c) * 2;
          sts128(y0, wa[m]);
          sts128(y0 + 8 * Cfg::kRowB, wb[m]);
        }
      }
      __syncthreads();
      // the chunk's new rows back to y, the pieces this thread copied in
      if (n0 + pcol < a.d_out) {
#pragma unroll
        for (int u = 0; u < U2; ++u)
          if (prow + 8 * u < rows)
            *reinterpret_cast<uint4*>(ysrc[u] + n0) = lds128(st + (prow + 8 * u) * Cfg::kRowB + pcol * 2);
      }
    }
    cp_async_wait<0>();  // only empty groups are left
    __syncthreads();     // the next tile's copies may overwrite every stage
  }
}

template <int R>
cudaError_t launch_rank(const LoraArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = (size_t)(((a.n + 1) * 4 + 127) / 128 * 128) + (size_t)LoraCfg<R>::kStages * LoraCfg<R>::kStage;
  cudaError_t e = cudaFuncSetAttribute(lora_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lora_kernel<R>, 32 * kLoraWarps, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  return launch_pdl(lora_kernel<R>, dim3(num_sms * per_sm), dim3(32 * kLoraWarps), smem, s, a);
}

}  // namespace

cudaError_t launch_lora(const LoraArgs& a, int num_sms, cudaStream_t s) {
  if (a.rank == 16) return launch_rank<16>(a, num_sms, s);
  if (a.rank == 32) return launch_rank<32>(a, num_sms, s);
  return launch_rank<64>(a, num_sms, s);
}

}  // namespace kev
