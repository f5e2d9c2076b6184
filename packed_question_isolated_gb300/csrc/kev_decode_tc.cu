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
// Roles (384 threads): warp 0 issues the TMA loads (K, V tiles, the 16 query rows, and for the
// chunk that holds position n its new K and V rows) into a ring of stages and records each
// chunk's position in the stage; warp 11 does the fix-ups of that chunk as soon as it lands (the
// new K/V row into the tiles and, once, into the pool; V rows past n zeroed up to the end of
// the last 16-key PV step), so they never wait behind the softmax of the chunk before; warp 1
// issues the S MMAs, warp 6 the PV MMAs (each on its own thread, so neither waits behind the
// other; a stage is released when its PV completes); warps 2-5 (one thread per key row for S^T):
// the softmax over the group's heads only, with a reference max per piece and per-thread sums,
// P^T into shared memory; warps 7-10 (one thread per head dimension of O^T): the output /
// split-K partials.  Consecutive chunks of one (question, kv head) in a CTA accumulate in TMEM;
// the pieces of one (question, kv head) that different CTAs produce are merged in a fixed order
// by a second kernel.
#include <cuda.h>
#include <stdlib.h>

#include <climits>

#include "kev_decode_common.cuh"
#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;
using dec::ItemInfo;

constexpr int kD = 128;
constexpr int kN = 16;             // MMA N: q-heads of one group, padded to 16
constexpr int kC = dec::kChunk;    // 128 keys per chunk
constexpr int kBatch = 4;          // most consecutive chunks per dynamic grab
// A call of at most kSmallPerCta chunks per CTA hands out its last kTailPerCta chunks per CTA in
// grabs of kTailBatch chunks (measured: the 128-step decode of 256 short questions 2.12 -> 1.99 ms;
// on the 32-question Qwen3-8B decode, ~18 chunks per CTA, any such tail was slower)
constexpr int kSmallPerCta = 8;
constexpr int kTailPerCta = 4;
constexpr int kTailBatch = 2;
constexpr int kThreads = 384;
constexpr int kQuad = 128;         // threads of the softmax (warps 2-5) and of the epilogue (warps 7-10)
constexpr long long kDrainBudget = 4000000000ll;
constexpr uint32_t kTmemCols = 64; // S^T x2 (cols 0, 16) + O^T x2 (cols 32, 48), 16 cols each
// A chunk whose scores exceed the piece's reference max by more than this (log2 units) takes
// the exact rescaling path: below it, P < 2^64 and the fp32 sums cannot overflow.
constexpr float kLog2Guard = 64.f;

// Tensor maps of one call: the K/V pools in boxes of 16 << j rows (j < kBoxSizes), the new queries.
constexpr int kBoxSizes = 4;
struct DecodeMaps {
  CUtensorMap k[kBoxSizes], v[kBoxSizes], q;
};

struct DTcParams {
  DecodeArgs a;
  long long wait_budget;
};

// What the producer knows about the chunk in a stage; the consumers read it from here.
struct StageInfo {
  int i, g, c, nch, len;
  int row0;   // pool row (of the [rows, d] view) of the chunk's first position for kv head g
  int xi0;    // global index of chunk 0 of this (question, kv head)
  int flags;  // kFirst / kLast of a piece, kFix: holds position n, kEnd: no more chunks
};
constexpr int kFirst = 1, kLast = 2, kFix = 4, kEnd = 8;

// A finished piece, handed from the softmax to the epilogue warps.
struct PieceInfo {
  int i, g, c_start, nch, n_in, xi0, flags, pad;  // flags: kWhole, kEnd
  float m[kN];                                    // reference max per head (log2 units)
  float l4[4][kN];                                // per-warp partial sums per head
};
constexpr int kWhole = 1;

template <int NS>
struct TSmem {
  static constexpr int kKBytes = kC * kD * 2;        // 32 KB, 2 sub-tiles of 128 rows x 128 B
  static constexpr int kQBytes = kN * kD * 2;        // 4 KB, 2 sub-tiles of 16 rows x 128 B
  static constexpr int kStageBytes = 2 * kKBytes + kQBytes;
  static constexpr int kStage = 0;
  static constexpr int kPBytes = kN * kC * 2;           // P^T: 2 sub-tiles of 16 rows x 128 B
  static constexpr int kP = kStage + NS * kStageBytes;   // two P^T buffers (chunk parity)
  static constexpr int kRed = kP + 2 * kPBytes;          // float red_m[4][16]
  static constexpr int kPiece = kRed + 4 * kN * 4;       // PieceInfo[2]
  static constexpr int kInfo = kPiece + 2 * (int)sizeof(PieceInfo);  // StageInfo[NS]
  static constexpr int kNew = kInfo + NS * (int)sizeof(StageInfo);  // per stage: the new K and V rows
  static constexpr int kBar = kNew + NS * 2 * kD * 2;
  static constexpr int kBase = kBar + 512;               // int item_base[N+1], then int2 meta[N]
  static __host__ __device__ constexpr int meta_off(int n) { return kBase + ((n + 2) / 2) * 8; }
  static __host__ __device__ constexpr int bytes(int n) { return meta_off(n) + n * 8 + 1024; }
};

struct TBars {
  uint64_t full[3], empty[3];
  uint64_t fixed[3], s_full[2], s_free[2], p_full[2], o_done[2];  // fixed: per stage, once per chunk
  uint64_t o_full[2], o_free[2], pc_full[2];  // per piece buffer: O^T complete, O^T + info consumed, info written
  uint64_t drain_s, drain_p;
  uint64_t stall;  // timeout test hook: nothing ever arrives on it
  uint32_t tmem_base;
  int flags, last, abort, never;
  int scan_tmp[11];
};

// named barriers: 1 = softmax warps, 2 = epilogue warps
template <int ID>
__device__ __forceinline__ void named_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(kQuad) : "memory");
}
template <int ID>
__device__ __forceinline__ bool named_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(ID), "n"(kQuad)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void raise_timeout(const DecodeArgs& a, TBars* b) {
  set_status(a.dev_status, ST_TIMEOUT);
  reinterpret_cast<int*>(a.ws + a.layout.sched)[2] = ST_TIMEOUT;  // the merge kernel skips the call
  *reinterpret_cast<volatile int*>(&b->abort) = 1;
}

// Reduce NH per-lane values over the warp (max or sum).  Reduce-scatter halving steps over
// lane bits 16, 8, ... leave each lane with the partial of one head, the remaining butterfly
// steps finish it; lane l then holds the warp result for head reduce_head<NH>(l).
template <int NH, bool MAX>
__device__ __forceinline__ float warp_reduce(const float (&v)[NH], int lane) {
  auto op = [](float x, float y) { return MAX ? fmaxf(x, y) : x + y; };
  float a[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) a[h] = v[h];
#pragma unroll
  for (int half = NH / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool up = lane & bit;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? a[k] : a[k + half];
      const float keep = up ? a[k + half] : a[k];
      a[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
#pragma unroll
  for (int bit = 16 / NH; bit >= 1; bit >>= 1) a[0] = op(a[0], __shfl_xor_sync(0xffffffffu, a[0], bit));
  return a[0];
}
template <int NH>
__device__ __forceinline__ int reduce_head(int lane) {
  int h = 0;
#pragma unroll
  for (int half = NH / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) h += (lane & bit) ? half : 0;
  return h;
}
// one lane per head writes the warp result
template <int NH>
__device__ __forceinline__ bool reduce_writer(int lane) {
  return (lane & (32 / NH - 1)) == 0;
}

// The fixed plan of the dynamic grabs: batches of B = kBatch consecutive chunks over [0, x1),
// then batches of kTailBatch chunks over [x1, total) (on a small call the last kTailPerCta chunks
// per CTA, else what is left of the B-chunk batches).  Batch boundaries depend on the chunk index
// only (not on which CTA grabs what), so the pieces, and hence the results, are the same on every
// run.
struct BatchPlan {
  int B, n1, x1, nbat, total;
  __device__ int start(int b) const { return b < n1 ? b * B : x1 + (b - n1) * kTailBatch; }
  __device__ int end(int b) const { return b < n1 ? (b + 1) * B : min(x1 + (b - n1 + 1) * kTailBatch, total); }
  __device__ int of(int x) const { return x < x1 ? x / B : n1 + (x - x1) / kTailBatch; }
};
__device__ __forceinline__ BatchPlan make_plan(int total, int ctas) {
  const int tail = total <= kSmallPerCta * ctas ? kTailPerCta * ctas : 0;
  BatchPlan p;
  p.B = kBatch;  // measured: fixed 4-chunk batches beat a per-call size on small and large decodes
  p.n1 = total > tail ? (total - tail) / p.B : 0;
  p.x1 = p.n1 * p.B;
  p.nbat = p.n1 + (total - p.x1 + kTailBatch - 1) / kTailBatch;
  p.total = total;
  return p;
}

// Sequential walk over the compacted chunk list: the chunk after (i, g, c) is (i, g, c + 1),
// else (i, g + 1, 0), else chunk 0 of the next live question.
struct Cursor {
  int i, g, c, nch, len, slot;
};
__device__ __forceinline__ Cursor cursor_at(const DecodeArgs& a, const int* item_base, const int2* meta, int x) {
  const ItemInfo f = dec::decode_item<kN>(a, item_base, meta, x, 1);
  return Cursor{f.i, f.g, f.c, f.nch, f.len, f.slot};
}
__device__ __forceinline__ void cursor_next(Cursor& u, const DecodeArgs& a, const int* item_base, const int2* meta) {
  if (++u.c < u.nch) return;
  u.c = 0;
  if (++u.g < a.h_kv) return;
  u.g = 0;
  int j = u.i + 1;
  while (j < a.n && item_base[j + 1] == item_base[j]) ++j;  // dropped questions have no chunk
  u.i = j;
  if (j >= a.n) return;  // past the last chunk: not used
  const int2 m = meta[j];
  u.len = m.x;
  u.slot = m.y;
  u.nch = (u.len + 1 + kC - 1) / kC;
}

template <int NS, int NH>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeMaps maps,
                                                               const DTcParams prm) {
  using L = TSmem<NS>;
  const DecodeArgs& a = prm.a;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TBars* bars = reinterpret_cast<TBars*>(smem + L::kBar);
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + L::kInfo);
  PieceInfo* pinfo = reinterpret_cast<PieceInfo*>(smem + L::kPiece);
  int* item_base = reinterpret_cast<int*>(smem + L::kBase);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off(a.n));
  int* hash = reinterpret_cast<int*>(smem + L::kStage);
  float* red_m = reinterpret_cast<float*>(smem + L::kRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* sched = reinterpret_cast<int*>(a.ws + a.layout.sched);

  // barriers, tensor maps and the TMEM columns depend on nothing the kernels before this one
  // write: set them up while those finish
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) mbar_init(&bars->fixed[s], 32);  // the fix-up warp
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], kQuad);
      mbar_init(&bars->p_full[b], kQuad);
      mbar_init(&bars->o_done[b], 1);
      mbar_init(&bars->o_full[b], 1);
      mbar_init(&bars->o_free[b], kQuad);
      mbar_init(&bars->pc_full[b], kQuad);
    }
    mbar_init(&bars->drain_s, 1);
    mbar_init(&bars->drain_p, 1);
    mbar_init(&bars->stall, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int j = 0; j < kBoxSizes; ++j) {
      tma_prefetch_desc(&maps.k[j]);
      tma_prefetch_desc(&maps.v[j]);
    }
    tma_prefetch_desc(&maps.q);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();  // lens, the pool and the counters are as the kernels before this one left them
  // the first batch grab goes out now; its latency hides behind the validation (the merge
  // kernel that follows resets the counter for the next call)
  int grab = 0;
  if (tid == 0) {
    grab = atomicAdd(&sched[0], 1);
    bars->abort = 0;
    bars->never = 0;
  }
  const int total = dec::prologue<kThreads>(a, 1, item_base, meta, hash, &bars->flags, bars->scan_tmp, &sched[2]);

  if (total >= 0) {
    if (blockIdx.x == 0 && tid == 0) {  // the merge kernel rebuilds the pieces from the plan
      const BatchPlan plan = make_plan(total, gridDim.x);
      sched[1] = plan.x1;
      sched[3] = plan.n1;
      sched[4] = plan.B;
    }
    tc_fence_before();
    __syncthreads();  // the hash is dead from here on: the stages may be written
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;
    const volatile int* never = &bars->never;
    const long long budget = prm.wait_budget;

    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      if (lane == 0) {
        uint32_t issued[3] = {0, 0, 0};
        // timeout test hook: a wait that runs out (nothing arrives), then the abort path
        bool ok = !(a.test_stall && blockIdx.x == 0) || mbar_wait(&bars->stall, 0, abort_flag, budget);
        const BatchPlan plan = make_plan(total, gridDim.x);
        int k = 0;  // position in the stage ring
        // the next grab goes out when a batch starts: its round trip hides behind the batch
        // (two in flight measured slower: a CTA then holds more work when the list runs out)
        int bat = grab;
        while (ok && bat < plan.nbat) {
          const int next = atomicAdd(&sched[0], 1);
          const int x0 = plan.start(bat), x1 = plan.end(bat);
          Cursor u = cursor_at(a, item_base, meta, x0);
          for (int x = x0; x < x1; ++x, ++k) {
            const int s = k % NS;
            const uint32_t round = k / NS;
            if (round > 0 && !mbar_wait(&bars->empty[s], (round - 1) & 1, abort_flag, budget)) {
              ok = false;
              break;
            }
            int flags = 0;
            if (x == x0 || u.c == 0) flags |= kFirst;
            if (x == x1 - 1 || u.c == u.nch - 1) flags |= kLast;
            if (u.c == u.nch - 1) flags |= kFix;
            // contiguous pool: slot row block; paged pool: the chunk is one block (its table entry)
            const int row0 = a.block_table ? (a.block_table[(int64_t)u.i * a.max_blocks + u.c] * a.h_kv + u.g) * kC
                                           : (u.slot * a.h_kv + u.g) * a.cap + u.c * kC;
            info[s] = StageInfo{u.i, u.g, u.c, u.nch, u.len, row0, x - u.c, flags};
            unsigned char* st = smem + L::kStage + s * L::kStageBytes;
            const int qrow = u.i * a.h_q + u.g * a.group;
            // The chunk that holds position n = len reads only its len - 128 c cached rows, in
            // one box per 64-column half of the smallest height that covers them (a TMA copy costs
            // about as much to issue whatever its size); the rows past them are masked, or zeroed
            // for V, by the fix-ups.  Every other chunk is a whole 128-row tile.
            const int rows = (flags & kFix) ? u.len - u.c * kC : kC;
            const int j = rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : 3;
            const int new_bytes = (flags & kFix) ? 2 * kD * 2 : 0;  // the new K and V rows, for the fix-ups
            mbar_arrive_expect_tx(&bars->full[s], (rows > 0 ? (16 << j) * 512 : 0) + L::kQBytes + new_bytes);  // release: info[s]
            if (new_bytes) {
              const int64_t src = ((int64_t)u.i * a.h_kv + u.g) * kD * 2;
              unsigned char* nb = smem + L::kNew + s * 2 * kD * 2;
              bulk_load(nb, static_cast<const unsigned char*>(a.k_new) + src, kD * 2, &bars->full[s]);
              bulk_load(nb + kD * 2, static_cast<const unsigned char*>(a.v_new) + src, kD * 2, &bars->full[s]);
            }
            if (rows > 0)
              for (int c = 0; c < 2; ++c) {
                tma_load_2d(st + c * (kC * 128), &maps.k[j], c * 64, row0, &bars->full[s]);
                tma_load_2d(st + L::kKBytes + c * (kC * 128), &maps.v[j], c * 64, row0, &bars->full[s]);
              }
            for (int c = 0; c < 2; ++c)
              tma_load_2d(st + 2 * L::kKBytes + c * (kN * 128), &maps.q, c * 64, qrow, &bars->full[s]);
            ++issued[s];
            cursor_next(u, a, item_base, meta);
          }
          bat = next;
        }
        // no more work for this CTA: the merge grid may be launched (it waits for this grid)
        pdl_trigger();
        if (ok) {  // end of the stream: a stage whose info says so, completed without copies
          const int s = k % NS;
          const uint32_t round = k / NS;
          if (round > 0 && !mbar_wait(&bars->empty[s], (round - 1) & 1, abort_flag, budget)) {
            ok = false;
          } else {
            info[s].flags = kEnd;
            mbar_arrive(&bars->full[s]);
          }
        }
        if (!ok) {
          raise_timeout(a, bars);
          for (int s = 0; s < NS; ++s)  // every copy lands before the CTA leaves
            if (issued[s]) mbar_wait(&bars->full[s], (issued[s] - 1) & 1, never, kDrainBudget);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- S issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16(128, kN, false, false);  // K (K-major) x Q^T
        bool ok = true;
        for (int k = 0;; ++k) {
          const int s = k % NS, sb = k & 1;
          if (!mbar_wait(&bars->full[s], (k / NS) & 1, abort_flag, budget)) { ok = false; break; }
          const int flags = info[s].flags;
          if (flags & kEnd) break;
          // the new row is written into the tiles first
          if ((flags & kFix) && !mbar_wait(&bars->fixed[s], (k / NS) & 1, abort_flag, budget)) { ok = false; break; }
          if (k >= 2 && !mbar_wait(&bars->s_free[sb], ((k >> 1) - 1) & 1, abort_flag, budget)) { ok = false; break; }
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
        }
        if (!ok) raise_timeout(a, bars);
        umma_commit(&bars->drain_s);  // every MMA of this thread is complete before TMEM is freed
        mbar_wait(&bars->drain_s, 0, never, kDrainBudget);
      }
    } else if (warp == 6) {
      // ---------------------------------------------------------------- PV issuer
      if (lane == 0) {
        constexpr uint32_t idesc_o = idesc_bf16(128, kN, true, false);  // V^T (MN-major) x P^T
        const uint32_t p_addr = smem_u32(smem + L::kP);
        int pc = 0;  // piece index: O^T buffer pc & 1
        bool ok = true;
        for (int k = 0;; ++k) {
          const int s = k % NS;
          // full[s] is long complete (S ran on this stage); waiting on it orders the read of info[s]
          if (!mbar_wait(&bars->full[s], (k / NS) & 1, abort_flag, budget)) { ok = false; break; }
          const int flags = info[s].flags;
          if (flags & kEnd) break;
          const bool first = flags & kFirst;
          // the chunk that holds position n: its keys past n have P = 0, so only the 16-key steps
          // up to n run (the fix-ups zero the V rows between n and the end of the last step)
          const int nk = (flags & kFix) ? (min(kC, info[s].len + 1 - info[s].c * kC) + 15) >> 4 : kC / 16;
          if (!mbar_wait(&bars->p_full[k & 1], (k >> 1) & 1, abort_flag, budget)) { ok = false; break; }
          if (first && pc >= 2 && !mbar_wait(&bars->o_free[pc & 1], ((pc >> 1) - 1) & 1, abort_flag, budget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + L::kStage + s * L::kStageBytes + L::kKBytes);
          const uint32_t d_o = tmem + (2 + (pc & 1)) * kN;
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk) {
            if (kk >= nk) break;
            const uint64_t av = sdesc_sw128(v_addr + kk * 16 * 128, kC * 128, 1024);
            const uint64_t bp =
                sdesc_sw128(p_addr + (k & 1) * L::kPBytes + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16(d_o, av, bp, idesc_o, (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(&bars->o_done[k & 1]);
          umma_commit(&bars->empty[s]);
          if (flags & kLast) {
            umma_commit(&bars->o_full[pc & 1]);
            ++pc;
          }
        }
        if (!ok) raise_timeout(a, bars);
        umma_commit(&bars->drain_p);
        mbar_wait(&bars->drain_p, 0, never, kDrainBudget);
      }
    } else if (warp == 11) {
      // ---------------------------------------------------------------- fix-up warp
      // Per chunk, once its stage has landed: for the chunk that holds position n = len, the new
      // K/V row (it came with the stage) goes into the swizzled tiles and, once, into the pool,
      // and V rows past it, up to the end of the last 16-key PV step, are zeroed (their P is 0,
      // but stale contents could hold NaN bit patterns).  fixed[s] completes once per chunk.
      bool ok = true;
      for (int k = 0;; ++k) {
        const int s = k % NS;
        ok = warp_wait(&bars->full[s], (k / NS) & 1, abort_flag, budget);
        if (!ok) break;
        const StageInfo inf = info[s];
        if (inf.flags & kEnd) break;
        if (inf.flags & kFix) {
          unsigned char* kst = smem + L::kStage + s * L::kStageBytes;
          unsigned char* vst = kst + L::kKBytes;
          const int p0 = inf.c * kC;
          const int nr = min(kC, inf.len + 1 - p0);
          const int rn = inf.len - p0;
          const int64_t dst = ((int64_t)inf.row0 + rn) * kD * 2;  // the new row's pool row
          const int ch = lane & 15;  // 16-byte chunk of the 256-byte row
          const bool isv = lane >= 16;
          const uint4 w = *reinterpret_cast<const uint4*>(smem + L::kNew + s * 2 * kD * 2 + (isv ? kD * 2 : 0) + ch * 16);
          unsigned char* tile = isv ? vst : kst;
          *reinterpret_cast<uint4*>(tile + (ch >> 3) * (kC * 128) + rn * 128 + (((ch & 7) ^ (rn & 7)) << 4)) = w;
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(isv ? a.pool_v : a.pool_k) + dst + ch * 16) = w;
          const int rows_pv = ((nr + 15) >> 4) << 4;  // rows the PV MMAs read
          for (int e = (nr * 16) + lane; e < rows_pv * 16; e += 32) {  // rows nr..rows_pv-1, 16 chunks each
            const int row = e >> 4, c16 = e & 15;
            *reinterpret_cast<uint4*>(vst + (c16 >> 3) * (kC * 128) + row * 128 + (c16 & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars->fixed[s]);
      }
      if (!ok && lane == 0) raise_timeout(a, bars);
    } else if (warp <= 5) {
      // ---------------------------------------------------------------- softmax warps 2-5
      const int q4 = warp & 3;                 // TMEM lane quarter of this warp
      const int r = q4 * 32 + lane;            // key row of S^T owned by this thread
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const int sid = tid - 64;                // 0..127
      const float sl2 = a.scale * 1.4426950408889634f;
      unsigned char* pbuf = smem + L::kP;
      float m_ref[NH], l_thr[NH];  // reference max (identical in all threads), this thread's sums
      uint32_t obs[2] = {0, 0};    // phases of o_done[0/1] seen
      int pc = 0, c_start = 0, n_in = 0;
      // A failed (timed-out) wait makes `ok` false and raises the abort flag, so every other
      // wait fails fast; the warps keep the same barrier sequence and leave together at a vote.
      bool ok = true;
      auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return;
        ok = warp_wait(bar, parity, abort_flag, budget);
        if (!ok) *abort_flag = 1;
      };
      auto column_max = [&](const float (&t)[NH], float (&cm)[NH]) {
        const float wm = warp_reduce<NH, true>(t, lane);
        if (reduce_writer<NH>(lane)) red_m[q4 * kN + reduce_head<NH>(lane)] = wm;
        named_sync<1>();
#pragma unroll
        for (int h = 0; h < NH; ++h)
          cm[h] = fmaxf(fmaxf(red_m[h], red_m[kN + h]), fmaxf(red_m[2 * kN + h], red_m[3 * kN + h]));
      };
      auto wait_pv = [&](int k) {  // PV(k) complete (o_done[k & 1] completes once per chunk of that parity)
        const int b = k & 1;
        const uint32_t ph = (uint32_t)k >> 1;
        if (obs[b] > ph) return;
        wait_ok(&bars->o_done[b], ph & 1);
        obs[b] = ph + 1;
      };
      // piece slot pc & 1 is free once the epilogue consumed piece pc - 2
      auto wait_slot = [&]() {
        if (pc >= 2) wait_ok(&bars->o_free[pc & 1], ((pc >> 1) - 1) & 1);
      };

      int k = 0;
      for (;; ++k) {
        const int s = k % NS, sb = k & 1;
        wait_ok(&bars->full[s], (k / NS) & 1);
        const StageInfo inf = info[s];
        if (named_or<1>(!ok || (inf.flags & kEnd))) break;  // identical in all threads when ok
        const bool first = inf.flags & kFirst, last = inf.flags & kLast;
        const int p0 = inf.c * kC;
        const int nr = min(kC, inf.len + 1 - p0);  // valid rows, the new one included

        // scores of this thread's key row for the group's heads
        wait_ok(&bars->s_full[sb], (k >> 1) & 1);
        tc_fence_after();
        uint32_t sr[NH];
        tmem_ld_cols<NH>(tmem + sb * kN + lane_off, sr);
        tc_fence_before();
        mbar_arrive(&bars->s_free[sb]);
        float t[NH];
        const bool valid = r < nr;
#pragma unroll
        for (int h = 0; h < NH; ++h) t[h] = valid ? __uint_as_float(sr[h]) * sl2 : -INFINITY;

        // The reference max of each head is fixed at the first chunk of a piece; it only
        // guards the exponentials against overflow (P is bf16, O and the sums accumulate in
        // fp32, so their precision is relative).  A later chunk whose scores exceed it by more
        // than the guard takes the exact path: new max, O^T and the sums rescaled.
        if (first) {
          column_max(t, m_ref);  // finite: every chunk holds at least one valid row
#pragma unroll
          for (int h = 0; h < NH; ++h) l_thr[h] = 0.f;
          c_start = inf.c;
          n_in = 0;
        }
        bool big = false;
#pragma unroll
        for (int h = 0; h < NH; ++h) big |= (t[h] - m_ref[h] > kLog2Guard);
        if (named_or<1>(big || !ok)) {
          if (named_or<1>(!ok)) break;  // every softmax thread leaves here together
          float cm[NH], alpha[NH];
          column_max(t, cm);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float m_new = fmaxf(m_ref[h], cm[h]);
            alpha[h] = ex2_approx(m_ref[h] - m_new);
            m_ref[h] = m_new;
            l_thr[h] *= alpha[h];
          }
          if (!first) {  // O^T holds the piece's chunks before this one: rescale once PV(k-1) is done
            wait_pv(k - 1);
            tc_fence_after();
            const uint32_t t_o = tmem + (2 + (pc & 1)) * kN + lane_off;
            uint32_t o[NH];
            tmem_ld_cols<NH>(t_o, o);
#pragma unroll
            for (int h = 0; h < NH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st_cols<NH>(t_o, o);
          }
        }
        float p[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          p[h] = ex2_approx(t[h] - m_ref[h]);
          l_thr[h] += p[h];
        }

        // P^T buffer k & 1 was last read by PV(k - 2)
        if (k >= 2) wait_pv(k - 2);
        // P^T: row h = head, column = key r, bf16, 128-byte swizzled (K-major B operand); rows
        // NH..15 are never written: they only feed O^T columns that are never read
        {
          unsigned char* pb = pbuf + (k & 1) * L::kPBytes;
          const int sub = r >> 6, kb = (r & 63) * 2;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int off = sub * (kN * 128) + h * 128 + ((((kb >> 4) ^ (h & 7))) << 4) + (kb & 15);
            *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(p[h]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[k & 1]);
        ++n_in;

        if (last) {  // hand the piece to the epilogue warps
          wait_slot();
          PieceInfo& pi = pinfo[pc & 1];
          const float ws = warp_reduce<NH, false>(l_thr, lane);
          if (reduce_writer<NH>(lane)) pi.l4[q4][reduce_head<NH>(lane)] = ws;
          if (sid < NH) pi.m[sid] = m_ref[sid];
          if (sid == 0) {
            pi.i = inf.i;
            pi.g = inf.g;
            pi.c_start = c_start;
            pi.nch = inf.nch;
            pi.n_in = n_in;
            pi.xi0 = inf.xi0;
            pi.flags = (c_start == 0 && n_in == inf.nch) ? kWhole : 0;
          }
          mbar_arrive(&bars->pc_full[pc & 1]);
          ++pc;
        }
      }
      if (ok) {  // end marker for the epilogue
        wait_slot();
        if (ok) {
          if (sid == 0) pinfo[pc & 1].flags = kEnd;
          mbar_arrive(&bars->pc_full[pc & 1]);
        }
      }
      if (!ok && lane == 0) raise_timeout(a, bars);
    } else {
      // ---------------------------------------------------------------- epilogue warps 7-10
      // Stores each finished piece: the output rows when the piece is a whole (question, kv
      // head), else its partial (O rows, reference max, sum) for the merge kernel.  No waiting
      // on global memory here, so the O^T buffers are released right away.
      const int q4 = warp & 3;
      const int r = q4 * 32 + lane;  // head dimension of O^T owned by this thread
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const int eid = tid - 224;     // 0..127
      float* partials = reinterpret_cast<float*>(a.ws + a.layout.partials);
      int2* item_xi0 = reinterpret_cast<int2*>(a.ws + a.layout.xi0);
      constexpr int pstride = kN * (kD + 2);
      bool ok = true;
      for (int pc = 0;; ++pc) {
        const int b = pc & 1;
        const uint32_t ph = (pc >> 1) & 1;
        if (!warp_wait(&bars->pc_full[b], ph, abort_flag, budget)) { ok = false; break; }
        const PieceInfo& pi = pinfo[b];
        if (pi.flags & kEnd) break;
        if (!warp_wait(&bars->o_full[b], ph, abort_flag, budget)) { ok = false; break; }  // last PV complete
        tc_fence_after();
        float ov[NH], l_sum[NH], m_p[NH];
        {
          uint32_t o[NH];
          tmem_ld_cols<NH>(tmem + (2 + b) * kN + lane_off, o);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            ov[h] = __uint_as_float(o[h]);
            l_sum[h] = (pi.l4[0][h] + pi.l4[1][h]) + (pi.l4[2][h] + pi.l4[3][h]);
            m_p[h] = pi.m[h];
          }
        }
        const int i = pi.i, g = pi.g, c_start = pi.c_start, xi0 = pi.xi0;
        const bool whole = pi.flags & kWhole;
        tc_fence_before();
        mbar_arrive(&bars->o_free[b]);  // O^T buffer b and piece slot b are free

        const int cidx = i * a.h_kv + g;
        if (whole) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)i * a.h_q + g * a.group) * kD + r;
#pragma unroll
          for (int h = 0; h < NH; ++h)
            if (h < a.group) out[h * kD] = __float2bfloat16_rn(ov[h] / l_sum[h]);
        } else {
          float* part = partials + ((int64_t)cidx * a.layout.max_chunks + c_start) * pstride;
#pragma unroll
          for (int h = 0; h < NH; ++h) part[h * kD + r] = ov[h];
          if (eid < NH) {
            part[kN * kD + eid] = m_p[eid];
            part[kN * kD + kN + eid] = l_sum[eid];
          }
        }
        if (c_start == 0 && eid == 0) item_xi0[cidx] = make_int2(xi0, pi.nch);
      }
      if (!ok && lane == 0) raise_timeout(a, bars);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else if (warp == 1) {  // invalid call: nothing ran on the tensor cores
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
  }

  // the merge kernel may be scheduled as soon as every CTA got here (it still waits for this
  // grid to complete before it reads anything)
  pdl_trigger();
}

// Merge of the pieces of every (question, kv head) that the decode kernel split (thread r =
// head dimension r; the pair's first chunk and chunk count come from the decode kernel through
// the workspace, so lens is not read here), in a fixed order: piece 0 starts at chunk 0, piece
// j > 0 at the j-th batch boundary of the grab plan after the pair's first chunk.  Online over
// rounds of pieces whose reference max and sum are gathered into shared memory while the O rows
// load.  Everything that decides a CTA's work -- the call's code and grab plan, the live flag and
// chunk range of pair blockIdx.x + t * gridDim.x for each thread t, a question's lens for the
// advance -- is loaded in one round trip; the CTA then merges only its pairs that were split.
// Block 0 also resets the decode kernel's batch counter for the next call.
template <int NH>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
  pdl_wait();  // the decode grid is complete and visible
  // the next kernel may be scheduled now: it waits for this grid before it touches memory
  // (the next step's segment builder launches during the merge instead of after it)
  pdl_trigger();
  int* sched = reinterpret_cast<int*>(a.ws + a.layout.sched);
  const int2* item_xi0 = reinterpret_cast<const int2*>(a.ws + a.layout.xi0);
  const int r = threadIdx.x;
  const int n_pairs = a.n * a.h_kv;
  const int code = sched[2];
  BatchPlan plan;
  plan.x1 = sched[1];
  plan.n1 = sched[3];
  plan.B = sched[4];
  plan.total = INT_MAX;  // not needed here (only start and of are)
  const int pair = blockIdx.x + r * gridDim.x;  // the grid covers every pair and every question
  const int live = pair < n_pairs ? a.active[pair / a.h_kv] : 0;
  const int2 xc = pair < n_pairs ? item_xi0[pair] : make_int2(-1, 0);  // written for every live pair
  const int qi = blockIdx.x * blockDim.x + r;
  const bool adv = a.advance_lens && qi < a.n && a.active[qi];
  const int len = adv ? a.advance_lens[qi] : 0;
  if (blockIdx.x == 0 && r == 0) sched[0] = 0;
  if (code != ST_OK) return;  // invalid call (or timeout): nothing to merge, lens kept
  if (adv) a.advance_lens[qi] = len + 1;  // kev_decode_step: the step is complete, so lens moves on

  __shared__ int s_pair[128], s_xi0[128], s_nch[128], s_n;
  if (r == 0) s_n = 0;
  __syncthreads();
  if (live && xc.x >= 0 && plan.of(xc.x + xc.y - 1) != plan.of(xc.x)) {  // more than one piece
    const int e = atomicAdd(&s_n, 1);
    s_pair[e] = pair;
    s_xi0[e] = xc.x;
    s_nch[e] = xc.y;
  }
  __syncthreads();
  const int n_split = s_n;

  __shared__ float mg_m[128], mg_l[128];
  const float* partials = reinterpret_cast<const float*>(a.ws + a.layout.partials);
  constexpr int pstride = kN * (kD + 2);
  constexpr int kRound = 32 / NH > 8 ? 8 : 32 / NH;  // pieces per round (O loads in flight)
  for (int e = 0; e < n_split; ++e) {
    const int cidx = s_pair[e], xi0 = s_xi0[e], nch = s_nch[e];
    const int i = cidx / a.h_kv, g = cidx % a.h_kv;
    const int b0 = plan.of(xi0);
    const int np = plan.of(xi0 + nch - 1) - b0 + 1;
    const float* base = partials + (int64_t)cidx * a.layout.max_chunks * pstride;
    auto piece_off = [&](int j) { return (j == 0 ? 0 : plan.start(b0 + j) - xi0) * pstride; };
    float M[NH], Ls[NH], O[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      M[h] = -INFINITY;
      Ls[h] = 0.f;
      O[h] = 0.f;
    }
    for (int j0 = 0; j0 < np; j0 += kRound) {
      const int jn = min(kRound, np - j0);
      if (r < jn * NH) {
        const int j = r / NH, h = r % NH;
        const int off = piece_off(j0 + j);
        mg_m[r] = base[off + kN * kD + h];
        mg_l[r] = base[off + kN * kD + kN + h];
      }
      float ovr[kRound][NH];
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        const int off = piece_off(j0 + u);
#pragma unroll
        for (int h = 0; h < NH; ++h) ovr[u][h] = (u < jn) ? base[off + h * kD + r] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float mr = M[h];
        for (int j = 0; j < jn; ++j) mr = fmaxf(mr, mg_m[j * NH + h]);
        const float sc = ex2_approx(M[h] - mr);  // 0 on the first round (M = -inf)
        Ls[h] *= sc;
        O[h] *= sc;
        M[h] = mr;
      }
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        if (u < jn) {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float wgt = ex2_approx(mg_m[u * NH + h] - M[h]);
            Ls[h] += mg_l[u * NH + h] * wgt;
            O[h] += ovr[u][h] * wgt;
          }
        }
      }
      __syncthreads();  // the round's gathered values are read before the next round overwrites them
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)i * a.h_q + g * a.group) * kD + r;
#pragma unroll
    for (int h = 0; h < NH; ++h)
      if (h < a.group) out[h * kD] = __float2bfloat16_rn(O[h] / Ls[h]);
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

template <int NS, int NH>
cudaError_t launch_ns(const DecodeArgs& a, int num_sms, cudaStream_t st, const DecodeMaps& m) {
  const int smem = TSmem<NS>::bytes(a.n);
  cudaError_t e =
      cudaFuncSetAttribute(decode_tc_kernel<NS, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  DTcParams p;
  p.a = a;
  p.a.test_stall = test_stall_requested();
  p.wait_budget = wait_budget_cycles();
  e = launch_pdl(decode_tc_kernel<NS, NH>, dim3(num_sms), dim3(kThreads), (size_t)smem, st, m, p);
  if (e != cudaSuccess) return e;
  // the merge kernel, programmatically dependent on the decode kernel (its launch overlaps the
  // decode kernel's end; its griddepcontrol.wait orders every read after the decode grid)
  // one pair per thread at most (the CTAs spread the merges), every question covered for the advance
  const int pairs = a.n * a.h_kv;
  const int grid = max(min(pairs, 4 * num_sms), max((pairs + 127) / 128, (a.n + 127) / 128));
  return launch_pdl(decode_merge_kernel<NH>, dim3((unsigned)grid), dim3(128), 0, st, a);
}

template <int NH>
cudaError_t launch_nh(const DecodeArgs& a, int num_sms, cudaStream_t st, const DecodeMaps& m) {
  constexpr int kMaxSmem = 232448;
  if (TSmem<3>::bytes(a.n) <= kMaxSmem) return launch_ns<3, NH>(a, num_sms, st, m);
  return launch_ns<2, NH>(a, num_sms, st, m);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int num_sms, cudaStream_t st) {
  static_assert(kDecodeTcMaxGroup == kN, "one MMA covers the q-heads of a group");
  if (a.group < 1 || a.group > kDecodeTcMaxGroup) return cudaErrorInvalidValue;
  DecodeMaps m;
  const uint64_t pool_rows = a.block_table ? (uint64_t)a.n_blocks * a.h_kv * kC : (uint64_t)a.n_slots * a.h_kv * a.cap;
  for (int j = 0; j < kBoxSizes; ++j)
    if (!make_map(&m.k[j], a.pool_k, pool_rows, 16u << j) || !make_map(&m.v[j], a.pool_v, pool_rows, 16u << j))
      return cudaErrorInvalidValue;
  if (!make_map(&m.q, a.q_new, (uint64_t)a.n * a.h_q, kN)) return cudaErrorInvalidValue;
  if (a.group <= 4) return launch_nh<4>(a, num_sms, st, m);
  if (a.group <= 8) return launch_nh<8>(a, num_sms, st, m);
  return launch_nh<16>(a, num_sms, st, m);
}

}  // namespace kev
