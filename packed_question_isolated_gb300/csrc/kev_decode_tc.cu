// Decode step over the KV slot pool on the 5th-generation tensor cores (bf16, d = 128).
//
// Decode with a cache (inference-engine notes, sakurs2.com, §2.2): only K/V are cached; the
// new K/V row is appended at position n = lens_i and the new query attends to all n + 1
// positions, no mask.  Early-stopped questions (Kev pipeline article, gsyq.cn §2.3) have no
// work chunk and are neither read nor written.
//
// Work: the same compacted chunk list and per-CTA contiguous ranges as the CUDA-core decode
// kernel (one persistent CTA per SM).  A chunk is 128 positions of one (question, kv head);
// the G q-heads of the group (padded to 16) are the N dimension of two small MMAs:
//   S^T [128 keys x 16 heads] = K_chunk [128 x d] . Q^T      (A = K tile, K-major, from SMEM)
//   O^T [d x 16 heads]       += V_chunk^T [d x 128] . P^T    (A = V tile read MN-major)
// so the CUDA cores only run the softmax over 128 x 16 scores per chunk and the kernel is a
// TMA stream of K/V tiles: decode is HBM-bound, and this keeps its instruction count tiny.
//
// Roles (192 threads): warp 0 issues the TMA loads (K, V tiles of 128 rows, the 16 query rows)
// into a ring of stages; warp 1 issues the MMAs without blocking on either kind (a stage is
// released as soon as its PV is issued and done); warps 2-5 (one thread per key row for S^T,
// one thread per head dimension for O^T): per-head column max and sum over the chunk with
// warp shuffles and a 4-warp exchange, the online rescale of O^T in TMEM, P^T into shared
// memory, the new K/V row and the zeroing of V rows past the question's length (fix-ups of
// the chunk that holds position n), and the output / split-K partials.  Consecutive chunks of
// one (question, kv head) in a CTA accumulate in TMEM; the pieces of one (question, kv head)
// that different CTAs produce are merged in a fixed order by the CTA that finishes last.
#include <cuda.h>
#include <stdlib.h>

#include "kev_decode_common.cuh"
#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;
using dec::ItemInfo;
using dec::range_owner;
using dec::range_start;

constexpr int kD = 128;
constexpr int kN = 16;             // q-heads per item (MMA N)
constexpr int kC = dec::kChunk;    // 128 keys per chunk
constexpr int kThreads = 192;
constexpr int kSoftmax = 128;      // threads of warps 2-5
constexpr long long kDrainBudget = 4000000000ll;
constexpr uint32_t kTmemCols = 64; // S^T x2 (16 cols each) + O^T (16 cols)

struct DTcParams {
  DecodeArgs a;
  long long wait_budget;
};

template <int NS>
struct TSmem {
  static constexpr int kKBytes = kC * kD * 2;        // 32 KB, 2 sub-tiles of 128 rows x 128 B
  static constexpr int kQBytes = kN * kD * 2;        // 4 KB, 2 sub-tiles of 16 rows x 128 B
  static constexpr int kStageBytes = 2 * kKBytes + kQBytes;
  static constexpr int kStage = 0;
  static constexpr int kPBytes = kN * kC * 2;          // P^T: 2 sub-tiles of 16 rows x 128 B
  static constexpr int kP = kStage + NS * kStageBytes;  // two P^T buffers (chunk parity)
  static constexpr int kRed = kP + 2 * kPBytes;         // float red_m[4][16], red_l[2][4][16]
  static constexpr int kBar = kRed + 3 * 4 * kN * 4;
  static constexpr int kBase = kBar + 512;              // int item_base[N+1], then int2 meta[N]
  static __host__ __device__ constexpr int meta_off(int n) { return kBase + ((n + 2) / 2) * 8; }
  static __host__ __device__ constexpr int bytes(int n) { return meta_off(n) + n * 8 + 1024; }
};

struct TBars {
  uint64_t full[3], empty[3];
  uint64_t fixed, s_full[2], s_free[2], p_full[2], o_done[2], o_free, drain;
  uint32_t tmem_base;
  int flags, last, abort, never;
  int scan_tmp[8];
};

__device__ __forceinline__ void named_sync_sm() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSoftmax) : "memory");
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void raise_timeout(const DecodeArgs& a, TBars* b) {
  set_status(a.dev_status, ST_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b->abort) = 1;
}

// Reduce 16 per-lane values over the warp (max or sum).  Reduce-scatter: after the steps,
// lane l holds the warp result for head H(l) = 8 b4 + 4 b3 + 2 b2 + b1 (bits of l), and lanes
// l, l ^ 1 hold the same head.
template <bool MAX>
__device__ __forceinline__ float warp_reduce16(float (&v)[kN], int lane) {
  auto op = [](float x, float y) { return MAX ? fmaxf(x, y) : x + y; };
  float a8[8], a4[4], a2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float send = u16 ? v[k] : v[k + 8];
    const float keep = u16 ? v[k + 8] : v[k];
    a8[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = u8 ? a8[k] : a8[k + 4];
    const float keep = u8 ? a8[k + 4] : a8[k];
    a4[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = u4 ? a4[k] : a4[k + 2];
    const float keep = u4 ? a4[k + 2] : a4[k];
    a2[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = u2 ? a2[0] : a2[1];
  const float keep = u2 ? a2[1] : a2[0];
  float r = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(r, __shfl_xor_sync(0xffffffffu, r, 1));
}
__device__ __forceinline__ int reduce16_head(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                               const __grid_constant__ CUtensorMap tm_v,
                                                               const __grid_constant__ CUtensorMap tm_q,
                                                               const DTcParams prm) {
  using L = TSmem<NS>;
  const DecodeArgs& a = prm.a;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TBars* bars = reinterpret_cast<TBars*>(smem + L::kBar);
  int* item_base = reinterpret_cast<int*>(smem + L::kBase);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off(a.n));
  int* hash = reinterpret_cast<int*>(smem + L::kStage);
  float* red_m = reinterpret_cast<float*>(smem + L::kRed);
  float* red_l = red_m + 4 * kN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    bars->abort = 0;
    bars->never = 0;
  }
  const int total = dec::prologue<kThreads>(a, 1, item_base, meta, hash, &bars->flags, bars->scan_tmp);
  if (total < 0) return;
  const int nb = min((int)gridDim.x, total);  // every CTA range non-empty
  if ((int)blockIdx.x >= nb) return;
  const int x_begin = range_start(blockIdx.x, total, nb);
  const int x_end = range_start(blockIdx.x + 1, total, nb);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->fixed, kSoftmax);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], kSoftmax);
    }
    mbar_init(&bars->p_full[0], kSoftmax);
    mbar_init(&bars->p_full[1], kSoftmax);
    mbar_init(&bars->o_done[0], 1);
    mbar_init(&bars->o_done[1], 1);
    mbar_init(&bars->o_free, kSoftmax);
    mbar_init(&bars->drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // the hash is dead from here on: the stages may be written
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tm_o = tmem + 2 * kN;
  volatile int* abort_flag = &bars->abort;
  const volatile int* never = &bars->never;
  const long long budget = prm.wait_budget;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued[3] = {0, 0, 0};
      bool ok = true;
      uint32_t it = 0;
      for (int x = x_begin; x < x_end; ++x, ++it) {
        const ItemInfo fi = dec::decode_item<kN>(a, item_base, meta, x, 1);
        const int s = it % NS;
        const uint32_t round = it / NS;
        if (round > 0 && !mbar_wait(&bars->empty[s], (round - 1) & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        unsigned char* st = smem + L::kStage + s * L::kStageBytes;
        const int row0 = (fi.slot * a.h_kv + fi.g) * a.cap + fi.p0;
        mbar_arrive_expect_tx(&bars->full[s], L::kStageBytes);
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(st + c * (kC * 128), &tm_k, c * 64, row0, &bars->full[s]);
          tma_load_2d(st + L::kKBytes + c * (kC * 128), &tm_v, c * 64, row0, &bars->full[s]);
          tma_load_2d(st + 2 * L::kKBytes + c * (kN * 128), &tm_q, c * 64, fi.i * a.h_q + fi.h0, &bars->full[s]);
        }
        ++issued[s];
      }
      if (!ok) raise_timeout(a, bars);
      for (int s = 0; s < NS; ++s)  // every copy lands before the CTA leaves
        if (issued[s]) mbar_wait(&bars->full[s], (issued[s] - 1) & 1, never, kDrainBudget);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, kN, false, false);  // K (K-major) x Q^T
      constexpr uint32_t idesc_o = idesc_bf16(128, kN, true, false);   // V^T (MN-major) x P^T
      const uint32_t p_addr = smem_u32(smem + L::kP);
      // Non-blocking issue loop: S of the next chunk as soon as its tiles (and fix-ups) are in
      // and an S buffer is free, PV of the next chunk as soon as its P is written.  Neither
      // waits behind the other, so a stage is released right after its PV.
      const int count = x_end - x_begin;
      int ns = 0, np = 0;  // next chunk for S, for PV
      uint32_t fix_cnt = 0, pieces = 0;
      bool ok = true;
      long long t_last = clock64();
      while (np < count) {
        bool progressed = false;
        if (ns < count) {
          const ItemInfo fi = dec::decode_item<kN>(a, item_base, meta, x_begin + ns, 1);
          const int s = ns % NS, sb = ns & 1;
          const bool fix = fi.c == fi.nch - 1;  // the chunk with the new row is fixed up first
          if (mbar_test(&bars->full[s], (ns / NS) & 1) && (!fix || mbar_test(&bars->fixed, fix_cnt & 1)) &&
              (ns < 2 || mbar_test(&bars->s_free[sb], ((ns >> 1) - 1) & 1))) {
            tc_fence_after();
            const uint32_t k_addr = smem_u32(smem + L::kStage + s * L::kStageBytes);
            const uint32_t q_addr = k_addr + 2 * L::kKBytes;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint64_t ak = sdesc_sw128(k_addr + (kk >> 2) * (kC * 128) + (kk & 3) * 32, 16, 1024);
              const uint64_t bq = sdesc_sw128(q_addr + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
              umma_bf16(tmem + sb * kN, ak, bq, idesc_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(&bars->s_full[sb]);
            if (fix) ++fix_cnt;
            ++ns;
            progressed = true;
          }
        }
        if (np < ns) {
          const int x = x_begin + np;
          const ItemInfo fi = dec::decode_item<kN>(a, item_base, meta, x, 1);
          const bool first = (x == x_begin) || fi.c == 0;
          const bool last = (x == x_end - 1) || fi.c == fi.nch - 1;
          if (mbar_test(&bars->p_full[np & 1], (np >> 1) & 1) &&
              (!first || pieces == 0 || mbar_test(&bars->o_free, (pieces - 1) & 1))) {
            tc_fence_after();
            const int s = np % NS;
            const uint32_t v_addr = smem_u32(smem + L::kStage + s * L::kStageBytes + L::kKBytes);
#pragma unroll
            for (int kk = 0; kk < kC / 16; ++kk) {
              const uint64_t av = sdesc_sw128(v_addr + kk * 16 * 128, kC * 128, 1024);
              const uint64_t bp =
                  sdesc_sw128(p_addr + (np & 1) * L::kPBytes + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
              umma_bf16(tm_o, av, bp, idesc_o, (first && kk == 0) ? 0u : 1u);
            }
            umma_commit(&bars->o_done[np & 1]);
            umma_commit(&bars->empty[s]);
            if (last) ++pieces;
            ++np;
            progressed = true;
          }
        }
        if (progressed) {
          t_last = clock64();
        } else {
          if (*abort_flag || clock64() - t_last > budget) {
            ok = false;
            break;
          }
          __nanosleep(32);  // leave the issue slots to the softmax warps
        }
      }
      if (!ok) raise_timeout(a, bars);
      umma_commit(&bars->drain);  // every MMA is complete before TMEM is freed
      mbar_wait(&bars->drain, 0, never, kDrainBudget);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;            // key row (S^T) and head dimension (O^T) of this thread
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int sid = tid - 64;                // 0..127 among the softmax threads
    const float sl2 = a.scale * 1.4426950408889634f;
    int* counters = reinterpret_cast<int*>(a.ws + a.layout.counters);
    float* partials = reinterpret_cast<float*>(a.ws + a.layout.partials);
    constexpr int pstride = kN * (kD + 2);
    unsigned char* pbuf = smem + L::kP;
    float m_run[kN], l_run[kN];
    uint32_t obs[2] = {0, 0};  // phases of o_done[0/1] seen
    bool ok = true;
    uint32_t it = 0;
    for (int x = x_begin; x < x_end; ++x, ++it) {
      const ItemInfo fi = dec::decode_item<kN>(a, item_base, meta, x, 1);
      const int s = it % NS, sb = it & 1;
      const bool first = (x == x_begin) || fi.c == 0;
      const bool last = (x == x_end - 1) || fi.c == fi.nch - 1;
      const int nr = fi.p1 - fi.p0;  // valid rows, the new one included
      unsigned char* kst = smem + L::kStage + s * L::kStageBytes;
      unsigned char* vst = kst + L::kKBytes;

      if (fi.c == fi.nch - 1) {
        // fix-ups of the chunk that holds position n = len: the new K/V row goes into the
        // swizzled tiles (and, once, into the pool); V rows past it are zeroed (their P is 0,
        // but stale pool contents could hold NaN bit patterns)
        if (!warp_wait(&bars->full[s], (it / NS) & 1, abort_flag, budget)) { ok = false; break; }
        const int rn = fi.len - fi.p0;
        const int64_t src = ((int64_t)fi.i * a.h_kv + fi.g) * kD * 2;
        const int64_t dst = (((int64_t)fi.slot * a.h_kv + fi.g) * a.cap + fi.len) * kD * 2;
        if (sid < 32) {
          const int ch = sid & 15;  // 16-byte chunk of the 256-byte row
          const bool isv = sid >= 16;
          const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(isv ? a.v_new : a.k_new) +
                                                          src + ch * 16);
          unsigned char* tile = isv ? vst : kst;
          *reinterpret_cast<uint4*>(tile + (ch >> 3) * (kC * 128) + rn * 128 + (((ch & 7) ^ (rn & 7)) << 4)) = w;
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(isv ? a.pool_v : a.pool_k) + dst + ch * 16) = w;
        }
        for (int e = (nr * 16) + sid; e < kC * 16; e += kSoftmax) {  // rows nr..127, 16 chunks each
          const int row = e >> 4, ch = e & 15;
          *reinterpret_cast<uint4*>(vst + (ch >> 3) * (kC * 128) + row * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->fixed);
      }

      // scores of this thread's key row for the 16 heads
      if (!warp_wait(&bars->s_full[sb], (it >> 1) & 1, abort_flag, budget)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[kN];
      tmem_ld16(tmem + sb * kN + lane_off, sr);
      tmem_ld_wait16(sr);
      tc_fence_before();
      mbar_arrive(&bars->s_free[sb]);
      float t[kN];
      const bool valid = r < nr;
#pragma unroll
      for (int h = 0; h < kN; ++h) t[h] = valid ? __uint_as_float(sr[h]) * sl2 : -INFINITY;

      auto column_max = [&](float (&cm)[kN]) {
        float v[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) v[h] = t[h];
        const float wm = warp_reduce16<true>(v, lane);
        if ((lane & 1) == 0) red_m[q4 * kN + reduce16_head(lane)] = wm;
        named_sync_sm();
#pragma unroll
        for (int h = 0; h < kN; ++h)
          cm[h] = fmaxf(fmaxf(red_m[h], red_m[kN + h]), fmaxf(red_m[2 * kN + h], red_m[3 * kN + h]));
      };
      auto exp_and_sum = [&](float (&p)[kN], float (&cs)[kN]) {
        float v[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) v[h] = p[h] = ex2_approx(t[h] - m_run[h]);
        // exchange buffer by chunk parity: the next chunk writes the other one before any
        // barrier, while slow threads may still read this one
        float* rl = red_l + (it & 1) * 4 * kN;
        const float ws = warp_reduce16<false>(v, lane);
        if ((lane & 1) == 0) rl[q4 * kN + reduce16_head(lane)] = ws;
        named_sync_sm();
#pragma unroll
        for (int h = 0; h < kN; ++h) cs[h] = (rl[h] + rl[kN + h]) + (rl[2 * kN + h] + rl[3 * kN + h]);
      };
      // PV(k) complete?  (o_done[k & 1] completes once per chunk of that parity)
      auto wait_pv = [&](int k) -> bool {
        const int b = k & 1;
        const uint32_t ph = (uint32_t)k >> 1;
        if (obs[b] > ph) return true;
        if (!warp_wait(&bars->o_done[b], ph & 1, abort_flag, budget)) return false;
        obs[b] = ph + 1;
        return true;
      };

      // The reference max of each head is fixed at the first chunk of a piece: it only guards
      // the exponentials against overflow (P is bf16, O and l accumulate in fp32, so their
      // precision is relative).  A later chunk whose sum signals overflow risk (its scores
      // grew by ~2^57 over the reference) takes the exact path: new max, O^T and l rescaled.
      float p[kN], cs[kN];
      if (first) {
        float cm[kN];
        column_max(cm);
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          m_run[h] = cm[h];  // finite: every chunk holds at least one row
          l_run[h] = 0.f;
        }
      }
      exp_and_sum(p, cs);
      bool big = false;
#pragma unroll
      for (int h = 0; h < kN; ++h) big |= !(cs[h] <= 1.8446744e19f);  // identical in all threads
      if (big) {
        float cm[kN], alpha[kN];
        column_max(cm);
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          const float m_new = fmaxf(m_run[h], cm[h]);
          alpha[h] = ex2_approx(m_run[h] - m_new);
          m_run[h] = m_new;
          l_run[h] *= alpha[h];
        }
        if (!first) {  // O^T holds the chunks before this one: rescale it once PV(it-1) is done
          if (!wait_pv((int)it - 1)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(tm_o + lane_off, o);
          tmem_ld_wait16(o);
#pragma unroll
          for (int h = 0; h < kN; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          tmem_st16(tm_o + lane_off, o);
          tmem_st_wait();
        }
        named_sync_sm();  // this chunk's sums are read by every thread before they are rewritten
        exp_and_sum(p, cs);
      }
#pragma unroll
      for (int h = 0; h < kN; ++h) l_run[h] += cs[h];

      // P^T buffer it & 1 was last read by PV(it - 2)
      if (it >= 2 && !wait_pv((int)it - 2)) { ok = false; break; }
      // P^T: row h = head, column = key r, bf16, 128-byte swizzled (K-major B operand)
      {
        unsigned char* pb = pbuf + (it & 1) * L::kPBytes;
        const int sub = r >> 6, kb = (r & 63) * 2;
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          const int off = sub * (kN * 128) + h * 128 + ((((kb >> 4) ^ (h & 7))) << 4) + (kb & 15);
          *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(p[h]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[it & 1]);

      if (!last) continue;
      // ---- end of a piece: this thread holds dimension r of O for the 16 heads ----------
      if (!wait_pv((int)it)) { ok = false; break; }
      tc_fence_after();
      float ov[kN];
      {
        uint32_t o[16];
        tmem_ld16(tm_o + lane_off, o);
        tmem_ld_wait16(o);
#pragma unroll
        for (int h = 0; h < kN; ++h) ov[h] = __uint_as_float(o[h]);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      const int x0 = x - fi.c;
      const int c_start = max(x_begin, x0) - x0;
      const bool whole = (c_start == 0) && (fi.c == fi.nch - 1);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
      if (whole) {
        for (int h = 0; h < fi.nh; ++h)
          out[((int64_t)fi.i * a.h_q + fi.h0 + h) * kD + r] = __float2bfloat16_rn(ov[h] / l_run[h]);
        continue;
      }
      const int cidx = fi.i * a.h_kv + fi.g;
      float* part = partials + ((int64_t)cidx * a.layout.max_chunks + c_start) * pstride;
#pragma unroll
      for (int h = 0; h < kN; ++h) part[h * kD + r] = ov[h];
      if (sid < kN) {
        part[kN * kD + sid] = m_run[sid];
        part[kN * kD + kN + sid] = l_run[sid];
      }
      __threadfence();  // this CTA's partial is visible before its arrival is counted
      named_sync_sm();
      if (sid == 0) {
        const int b_first = range_owner(x0, total, nb), b_last = range_owner(x0 + fi.nch - 1, total, nb);
        bars->last = (atomicAdd(&counters[cidx], 1) == b_last - b_first);
      }
      named_sync_sm();
      if (bars->last) {
        __threadfence();
        const int b_first = range_owner(x0, total, nb), b_last = range_owner(x0 + fi.nch - 1, total, nb);
        const float* base = partials + (int64_t)cidx * a.layout.max_chunks * pstride;
        for (int h = 0; h < fi.nh; ++h) {
          float M = -INFINITY;
          for (int b = b_first; b <= b_last; ++b) {
            const int cs = max(range_start(b, total, nb), x0) - x0;
            M = fmaxf(M, __ldcg(base + cs * pstride + kN * kD + h));
          }
          float Lsum = 0.f, O = 0.f;
          for (int b = b_first; b <= b_last; ++b) {
            const int cs = max(range_start(b, total, nb), x0) - x0;
            const float* pc = base + cs * pstride;
            const float wgt = ex2_approx(__ldcg(pc + kN * kD + h) - M);
            Lsum += __ldcg(pc + kN * kD + kN + h) * wgt;
            O += __ldcg(pc + h * kD + r) * wgt;
          }
          out[((int64_t)fi.i * a.h_q + fi.h0 + h) * kD + r] = __float2bfloat16_rn(O / Lsum);
        }
        if (sid == 0) counters[cidx] = 0;
      }
      named_sync_sm();  // `last` is read by every thread before the next piece may set it
    }
    if (!ok && lane == 0) raise_timeout(a, bars);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

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

// 2-D bf16 view [rows, 128] of a row-major tensor, boxes of 64 columns x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, box_rows};
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
  return 4000000000ll;
}

template <int NS>
cudaError_t launch_ns(const DecodeArgs& a, int num_sms, cudaStream_t st, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mq) {
  const int smem = TSmem<NS>::bytes(a.n);
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  DTcParams p;
  p.a = a;
  p.wait_budget = wait_budget_cycles();
  decode_tc_kernel<NS><<<num_sms, kThreads, smem, st>>>(mk, mv, mq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int num_sms, cudaStream_t st) {
  CUtensorMap mk, mv, mq;
  const uint64_t pool_rows = (uint64_t)a.n_slots * a.h_kv * a.cap;
  if (!make_map(&mk, a.pool_k, pool_rows, kC) || !make_map(&mv, a.pool_v, pool_rows, kC) ||
      !make_map(&mq, a.q_new, (uint64_t)a.n * a.h_q, kN))
    return cudaErrorInvalidValue;
  constexpr int kMaxSmem = 232448;
  if (TSmem<3>::bytes(a.n) <= kMaxSmem) return launch_ns<3>(a, num_sms, st, mk, mv, mq);
  return launch_ns<2>(a, num_sms, st, mk, mv, mq);
}

}  // namespace kev
