// Packed prefill attention on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// Computes, for every work item (question i, 128-row query tile m, q-head h) of the segment
// builder's list, the exact attention of the inference-engine notes (sakurs2.com, §2.1,
// Z = softmax(QK^T / sqrt(d_h) + M) V) restricted by the causal AND block-diagonal mask of
// the Kev articles (icman.com.cn §2.3, gsyq.cn §2.2): the tile's rows read key tiles
// 0..m of their own question only, and only the diagonal tile m needs the element mask
// (key <= row).  Tiles are FlashAttention-style (notes §2.4): the T x T score matrix never
// leaves the chip, and the softmax is the online form with a running max m, sum l and a
// rescale of the accumulator when the max moves.
//
// GB300 mapping (one persistent CTA per SM, 192 threads):
//   warp 0     TMA producer: Q tile (128 x d) once per item, then K/V tiles (128 x d) into a
//              2-stage ring; 128-byte swizzled boxes, completion counted on mbarriers.
//   warp 1     MMA issuer: S = Q K^T into one of two TMEM buffers (128 x 128 fp32), then
//              O += P V into a TMEM accumulator (128 x d fp32) with tcgen05.mma, and
//              tcgen05.commit to release stages and signal the softmax warps.
//   warps 2-5  softmax: each thread owns one query row (its TMEM lane), reads its S row
//              with tcgen05.ld, applies the diagonal mask, updates m and l, writes P as
//              bf16 into a swizzled shared-memory tile for the PV MMA, and rescales its O
//              row in TMEM only when its running max grew by more than 2^8 (exact: O and l
//              always share the same reference max).  The epilogue divides by l and
//              stores bf16 rows; rows past the question's end are not stored.
// Every wait is bounded; a wait that gives up sets KEV_ERR_TIMEOUT and raises the CTA's
// abort flag, and the CTA drains its own copies and MMAs before freeing TMEM and exiting.
#include <cuda.h>
#include <stdlib.h>

#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;

constexpr int kBM = 128;            // query rows per tile
constexpr int kBN = 128;            // keys per tile
constexpr int kStages = 2;          // K/V ring depth
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;      // log2 units: rescale O when the max grows by > 2^8
constexpr long long kDrainBudget = 4000000000ll;  // cycles to wait for in-flight work on abort
constexpr int kPSub = kBM * 128;               // bytes of one 64-key column block of P

struct TcParams {
  char* ws;
  PrefillLayout layout;
  const kev_interval* intervals;
  void* out;
  int32_t h_q;
  int32_t group;
  float scale_log2;  // scale * log2(e)
  int32_t* dev_status;
  long long wait_budget;  // cycles per bounded wait
};

template <int D>
struct Smem {
  static constexpr int kSub = D / 64;             // 64-column (128-byte) sub-tiles per row
  static constexpr int kSubBytes = kBM * 128;     // one 128-row x 128-byte sub-tile
  static constexpr int kTileBytes = kBM * D * 2;  // one Q/K/V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kBar = kP + kBM * kBN * 2;
  static constexpr int kBytes = kBar + 1024;
  static constexpr int kLaunchBytes = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done, o_free, drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: abort flag for waits that must not give up early
};

__device__ __forceinline__ void raise_timeout(const TcParams& p, Bars* b) {
  PrefillHeader* hdr = reinterpret_cast<PrefillHeader*>(p.ws);
  atomicCAS(&hdr->status, 0, ST_TIMEOUT);
  set_status(p.dev_status, ST_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b->abort) = 1;
}

// All lanes wait; the warp agrees on the outcome so warp-collective tcgen05 ops stay uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using L = Smem<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(p.ws);
  if (hdr->status != ST_OK) return;
  const int n_items = hdr->n_items;
  if ((int)blockIdx.x >= n_items) return;
  const int4* items = reinterpret_cast<const int4*>(p.ws + p.layout.items);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tm_o = tmem + 2u * kBN;
  volatile int* abort_flag = &bars->abort;
  const volatile int* never = &bars->never;
  const long long budget = p.wait_budget;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_iter = 0, n = 0, q_loads = 0;
      uint32_t kv_loads[kStages] = {0, 0};
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
        const int4 item = items[it];
        const int seg_begin = p.intervals[item.x].begin;
        const int nkv = (item.y - seg_begin) / kBM + 1;
        const int g = item.w / p.group;
        if (n > 0 && !mbar_wait(&bars->q_empty, (n - 1) & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full, L::kTileBytes);
        for (int c = 0; c < L::kSub; ++c)
          tma_load_2d(smem + L::kQ + c * L::kSubBytes, &tm_q, item.w * D + c * 64, item.y, &bars->q_full);
        ++q_loads;
        for (int j = 0; j < nkv; ++j, ++kv_iter) {
          const int s = kv_iter % kStages;
          const uint32_t round = kv_iter / kStages;
          if (round > 0 && !mbar_wait(&bars->kv_empty[s], (round - 1) & 1, abort_flag, budget)) {
            ok = false;
            break;
          }
          const int key0 = seg_begin + j * kBN;
          mbar_arrive_expect_tx(&bars->k_full[s], L::kTileBytes);
          for (int c = 0; c < L::kSub; ++c)
            tma_load_2d(smem + L::kK + s * L::kTileBytes + c * L::kSubBytes, &tm_k, g * D + c * 64, key0,
                        &bars->k_full[s]);
          mbar_arrive_expect_tx(&bars->v_full[s], L::kTileBytes);
          for (int c = 0; c < L::kSub; ++c)
            tma_load_2d(smem + L::kV + s * L::kTileBytes + c * L::kSubBytes, &tm_v, g * D + c * 64, key0,
                        &bars->v_full[s]);
          ++kv_loads[s];
        }
      }
      if (!ok) raise_timeout(p, bars);
      if (*abort_flag) {
        // every copy issued by this thread lands before the CTA leaves
        if (q_loads) mbar_wait(&bars->q_full, (q_loads - 1) & 1, never, kDrainBudget);
        for (int s = 0; s < kStages; ++s) {
          if (kv_loads[s]) {
            mbar_wait(&bars->k_full[s], (kv_loads[s] - 1) & 1, never, kDrainBudget);
            mbar_wait(&bars->v_full[s], (kv_loads[s] - 1) & 1, never, kDrainBudget);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      const uint32_t p_addr = smem_u32(smem + L::kP);
      uint32_t kv_iter = 0, s_iter = 0, p_iter = 0, n = 0;
      bool ok = true;

      auto issue_s = [&](uint32_t kvi) -> bool {
        const int s = kvi % kStages;
        const uint32_t round = kvi / kStages;
        if (!mbar_wait(&bars->k_full[s], round & 1, abort_flag, budget)) return false;
        const int sb = s_iter & 1;
        const uint32_t sround = s_iter >> 1;
        if (sround > 0 && !mbar_wait(&bars->s_free[sb], (sround - 1) & 1, abort_flag, budget)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + L::kK + s * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kSubBytes + (kk & 3) * 32;
          umma_bf16(tmem + sb * kBN, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                    idesc_s, kk > 0);
        }
        umma_commit(&bars->s_full[sb]);
        ++s_iter;
        return true;
      };

      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
        const int4 item = items[it];
        const int seg_begin = p.intervals[item.x].begin;
        const int nkv = (item.y - seg_begin) / kBM + 1;
        if (!mbar_wait(&bars->q_full, n & 1, abort_flag, budget) || !issue_s(kv_iter)) {
          ok = false;
          break;
        }
        if (nkv == 1) umma_commit(&bars->q_empty);
        for (int j = 0; j < nkv; ++j) {
          if (j + 1 < nkv) {
            if (!issue_s(kv_iter + j + 1)) {
              ok = false;
              break;
            }
            if (j + 1 == nkv - 1) umma_commit(&bars->q_empty);  // last use of this Q tile issued
          }
          const int s = (kv_iter + j) % kStages;
          const uint32_t round = (kv_iter + j) / kStages;
          if (!mbar_wait(&bars->p_full, p_iter & 1, abort_flag, budget) ||
              !mbar_wait(&bars->v_full[s], round & 1, abort_flag, budget) ||
              (j == 0 && n > 0 && !mbar_wait(&bars->o_free, (n - 1) & 1, abort_flag, budget))) {
            ok = false;
            break;
          }
          ++p_iter;
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + L::kV + s * L::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t a = sdesc_sw128(p_addr + (kk >> 2) * kPSub + (kk & 3) * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(v_addr + kk * 16 * 128, L::kSubBytes, 1024);
            umma_bf16(tm_o, a, b, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars->kv_empty[s]);
          umma_commit(&bars->o_done);
        }
        kv_iter += nkv;
      }
      if (!ok) raise_timeout(p, bars);
      // every MMA this thread issued is complete before TMEM is freed
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, never, kDrainBudget);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;  // a warp may only touch TMEM lanes [32*(warp%4), +32)
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t p_addr = smem_u32(smem + L::kP);
    const float sl2 = p.scale_log2;
    uint32_t s_iter = 0, o_iter = 0;
    bool ok = true;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);

    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 item = items[it];
      const int seg_begin = p.intervals[item.x].begin;
      const int nkv = (item.y - seg_begin) / kBM + 1;
      float m_run = -INFINITY, l_run = 0.f;

      for (int j = 0; j < nkv; ++j) {
        const int sb = s_iter & 1;
        const uint32_t sround = s_iter >> 1;
        if (!warp_wait(&bars->s_full[sb], sround & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float t[kBN];
        {
          uint32_t sr[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tmem + sb * kBN + lane_off + c * 32, sr[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) t[c * 32 + e] = __uint_as_float(sr[c][e]) * sl2;
        }
        tc_fence_before();
        mbar_arrive(&bars->s_free[sb]);
        ++s_iter;

        if (j == nkv - 1) {  // diagonal tile: key x is visible to row r iff x <= r
#pragma unroll
          for (int x = 0; x < kBN; ++x)
            if (x > r) t[x] = -INFINITY;
        }
        float mt = t[0];
#pragma unroll
        for (int x = 1; x < kBN; ++x) mt = fmaxf(mt, t[x]);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_run = mt;
        } else if (mt > m_run + kRescaleThreshold) {
          alpha = ex2_approx(m_run - mt);
          m_run = mt;
          l_run *= alpha;
          rescale = true;
        }
        uint32_t pk[kBN / 2];
        float rs = 0.f;
#pragma unroll
        for (int x = 0; x < kBN; x += 2) {
          const float a = ex2_approx(t[x] - m_run);
          const float b = ex2_approx(t[x + 1] - m_run);
          rs += a + b;
          pk[x >> 1] = pack_bf16x2(a, b);
        }
        l_run += rs;

        if (j > 0) {  // PV of the previous tile must be done: it reads P and accumulates O
          if (!warp_wait(&bars->o_done, o_iter & 1, abort_flag, budget)) {
            ok = false;
            break;
          }
          ++o_iter;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + lane_off + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tm_o + lane_off + c * 32, o);
          }
          tmem_st_wait();
        }
#pragma unroll
        for (int ch = 0; ch < kBN / 8; ++ch) {
          const uint32_t addr = p_addr + (ch >> 3) * kPSub + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
          st_shared_v4(addr, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full);
      }
      if (!ok) break;

      // epilogue: O / l -> bf16 rows of this item
      if (!warp_wait(&bars->o_done, o_iter & 1, abort_flag, budget)) {
        ok = false;
        break;
      }
      ++o_iter;
      tc_fence_after();
      const float inv = 1.f / l_run;
      const bool valid = r < item.z;
      __nv_bfloat16* orow = out + ((int64_t)(item.y + r) * p.h_q + item.w) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tm_o + lane_off + c * 32, o);
        tmem_ld_wait(o);
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
    }
    if (!ok && lane == 0) raise_timeout(p, bars);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 view [rows, cols] (cols contiguous), boxes of 64 columns x 128 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

long long wait_budget_cycles() {
  const char* s = getenv("KEV_TEST_WAIT_LIMIT");
  if (s && *s) {
    const long long v = atoll(s);
    if (v > 0) return v;
  }
  return 4000000000ll;  // about two seconds at the top SM clock
}

template <int D>
cudaError_t launch_tc(const PrefillArgs& a, int num_sms, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, (uint64_t)a.h_q * D, (uint64_t)a.T) ||
      !make_map(&mk, a.k, (uint64_t)a.h_kv * D, (uint64_t)a.T) ||
      !make_map(&mv, a.v, (uint64_t)a.h_kv * D, (uint64_t)a.T))
    return cudaErrorInvalidValue;
  TcParams p;
  p.ws = const_cast<char*>(a.ws);
  p.layout = a.layout;
  p.intervals = a.intervals;
  p.out = a.out;
  p.h_q = a.h_q;
  p.group = a.group;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.dev_status = a.dev_status;
  p.wait_budget = wait_budget_cycles();
  const int smem = Smem<D>::kLaunchBytes;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t max_items = a.layout.max_items;
  const int grid = (int)(max_items < num_sms ? max_items : num_sms);
  prefill_tc_kernel<D><<<grid, kThreads, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, int d, int num_sms, cudaStream_t s) {
  if (a.T <= 0 || a.layout.max_items == 0) return cudaSuccess;
  return d == 64 ? launch_tc<64>(a, num_sms, s) : launch_tc<128>(a, num_sms, s);
}

}  // namespace kev
