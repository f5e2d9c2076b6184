// Decode step over the KV slot pool: compaction, append, split-K attention, fixed-order merge.
//
// Decode with a cache (inference-engine notes, sakurs2.com, §2.2): only K/V are cached; the
// new row is appended at position n = lens_i and the new query attends to all n + 1
// positions, no mask.  Early stop (Kev pipeline article, gsyq.cn news 368355, §1.2, §2.3):
// a question with active[i] == 0 is removed from the step -- it contributes no work item,
// so its slot is neither read nor written.
//
// One launch, one persistent CTA per SM.  Every CTA first runs the same prologue over the N
// questions: validation of the live questions and a prefix sum of their work items, which
// is the compacted list of live (question, kv head, head block, chunk) items -- so no second
// launch or grid-wide wait is needed.  A chunk is kChunk consecutive positions of one slot;
// its K rows and its V rows are each one contiguous range of the pool and are streamed into
// shared memory with single bulk copies (TMA, 1-D), double buffered: while the eight warps
// work on chunk x, the copies of chunk x+1 are in flight.
//
// Eight compute warps per CTA, for the G q-heads that share the kv head (up to 8 per item):
//   scores   half a warp per K row, lane l holding 8 dims of the row and the same 8 dims of
//            every query in registers; the 16 partial dot products of 4 rows are combined
//            with a shuffle reduce-scatter (5 shuffles per head for 4 rows);
//   softmax  one warp per head: max, exp2 and sum over the chunk's rows;
//   PV       16 lanes across the 128 dims x 16 row groups; packed fp32x2 FMAs; the row
//            groups are summed with shuffles and one pass through shared memory.
// When a (question, kv head) has several chunks, the CTA that finishes last (arrival
// counter) merges the chunk results in chunk order, so the output does not depend on timing.
#include "kev_decode_common.cuh"
#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;
using dec::ItemInfo;
using dec::range_owner;
using dec::range_start;

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads;  // thread 0 also issues the bulk copies
constexpr int kChunk = kDecodeChunk;            // rows per work item
constexpr int kMaxStages = 3;
constexpr int kHB = 8;                          // q-heads per item at most
constexpr long long kDrainBudget = 4000000000ll;

template <int D, int EB, int GT, int NS>
struct DSmem {
  static constexpr int kRowBytes = D * EB;
  static constexpr int kQBytes = kHB * kRowBytes;                       // the item's queries
  static constexpr int kStageBytes = 2 * kChunk * kRowBytes + kQBytes;  // K rows, V rows, queries
  static constexpr int kStages = NS;                                    // stage ring depth
  static constexpr int kStage = 0;
  static constexpr int kS = kStage + kStages * kStageBytes;   // float [GT][kChunk]  scores
  static constexpr int kP = kS + GT * kChunk * 4;             // float [kChunk][GT]  weights
  static constexpr int kRed = kP + kChunk * GT * 4;           // float [4][GT][D]    cross-warp sums
  static constexpr int kStat = kRed + 4 * GT * D * 4;         // float m[kHB], l[kHB], alpha[kHB]
  static constexpr int kBar = kStat + 3 * kHB * 4;            // DBars
  static constexpr int kBase = kBar + 128;                    // int item_base[N + 1], then int2 meta[N]
  // total for N questions
  static __host__ __device__ constexpr int bytes(int n) { return kBase + ((n + 2) / 2) * 8 + n * 8; }
  static __host__ __device__ constexpr int meta_off(int n) { return kBase + ((n + 2) / 2) * 8; }
};

struct DBars {
  uint64_t full[kMaxStages];
  uint64_t stall;  // timeout test hook: nothing ever arrives on it
  int flags;
  int last;
  int abort;
  int never;
  int scan_tmp[(kThreads + 31) / 32];
};

__device__ __forceinline__ void named_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}
// Barrier over the compute warps that also ANDs a flag across them (a uniform decision).
__device__ __forceinline__ bool named_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kComputeThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// bf16 pair (low element first) -> packed fp32 pair, exact
__device__ __forceinline__ unsigned long long bf2_to_f2(uint32_t w) {
  return (unsigned long long)(w << 16) | ((unsigned long long)(w & 0xffff0000u) << 32);
}

// Element access for both storage types: 8 consecutive elements as 4 packed fp32 pairs.
template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void load8(const unsigned char* p, unsigned long long (&o)[4]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    o[0] = bf2_to_f2(w.x);
    o[1] = bf2_to_f2(w.y);
    o[2] = bf2_to_f2(w.z);
    o[3] = bf2_to_f2(w.w);
  }
  __device__ static __forceinline__ void store(void* base, int64_t idx, float v) {
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  }
  __device__ static __forceinline__ float load(const void* base, int64_t idx) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  }
};
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void load8(const unsigned char* p, unsigned long long (&o)[4]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint4 b = *reinterpret_cast<const uint4*>(p + 16);
    o[0] = (unsigned long long)a.x | ((unsigned long long)a.y << 32);
    o[1] = (unsigned long long)a.z | ((unsigned long long)a.w << 32);
    o[2] = (unsigned long long)b.x | ((unsigned long long)b.y << 32);
    o[3] = (unsigned long long)b.z | ((unsigned long long)b.w << 32);
  }
  __device__ static __forceinline__ void store(void* base, int64_t idx, float v) { static_cast<float*>(base)[idx] = v; }
  __device__ static __forceinline__ float load(const void* base, int64_t idx) { return static_cast<const float*>(base)[idx]; }
};

template <typename T, int D, int GT, int NS>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
  using E = Elem<T>;
  constexpr int EB = E::kBytes;
  using L = DSmem<D, EB, GT, NS>;
  constexpr int kRow = D * EB;  // bytes of one stored row
  extern __shared__ __align__(128) unsigned char smem[];
  DBars* bars = reinterpret_cast<DBars*>(smem + L::kBar);
  int* item_base = reinterpret_cast<int*>(smem + L::kBase);
  int2* meta = reinterpret_cast<int2*>(smem + L::meta_off(a.n));
  int* hash = reinterpret_cast<int*>(smem + L::kStage);
  float* sc = reinterpret_cast<float*>(smem + L::kS);
  float* pw = reinterpret_cast<float*>(smem + L::kP);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  float* st_m = reinterpret_cast<float*>(smem + L::kStat);
  float* st_l = st_m + kHB;
  float* st_a = st_l + kHB;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n;
  const int n_hblocks = (a.group + kHB - 1) / kHB;

  // ---- prologue: validation of live questions, compacted work list --------------------
  if (tid == 0) {
    bars->abort = 0;
    bars->never = 0;
  }
  int* sched = reinterpret_cast<int*>(a.ws + a.layout.sched);  // [2]: this call's validation code
  const int running =
      dec::prologue<kThreads>(a, n_hblocks, item_base, meta, hash, &bars->flags, bars->scan_tmp, &sched[2]);
  if (running < 0) return;
  if (tid == 0) {
    for (int s = 0; s < L::kStages; ++s) mbar_init(&bars->full[s], 1);
    mbar_init(&bars->stall, 1);
    fence_mbar_init();
  }
  __syncthreads();  // the hash is dead from here on: the stages may be written
  const int total = running;
  // at most one CTA per chunk, so that every CTA's range is non-empty and the CTAs that
  // touch a (question, kv head) are exactly the owners of its first..last chunk
  const int nb = min((int)gridDim.x, total);
  if ((int)blockIdx.x >= nb) return;
  const int x_begin = range_start(blockIdx.x, total, nb);
  const int x_end = range_start(blockIdx.x + 1, total, nb);
  volatile int* abort_flag = &bars->abort;
  const volatile int* never = &bars->never;
  const long long budget = a.wait_budget;

  // Thread 0 issues the bulk copies of a chunk: K rows, V rows (positions already in the
  // pool) and the item's queries, all counted on the stage's mbarrier.
  uint32_t issued[kMaxStages] = {0, 0, 0};
  auto issue = [&](int xx, int stage) {
    const ItemInfo fi = dec::decode_item<kHB>(a, item_base, meta, xx, n_hblocks);
    const int rows = min(fi.p1, fi.len) - fi.p0;  // the new row is not in the pool yet
    const uint32_t bytes = (uint32_t)rows * kRow;
    const uint32_t qbytes = (uint32_t)fi.nh * kRow;
    unsigned char* dst = smem + L::kStage + stage * L::kStageBytes;
    mbar_arrive_expect_tx(&bars->full[stage], 2 * bytes + qbytes);
    if (rows > 0) {
      const int64_t row0 = ((int64_t)fi.slot * a.h_kv + fi.g) * a.cap + fi.p0;
      bulk_copy_g2s(dst, static_cast<const unsigned char*>(a.pool_k) + row0 * kRow, bytes, &bars->full[stage]);
      bulk_copy_g2s(dst + kChunk * kRow, static_cast<const unsigned char*>(a.pool_v) + row0 * kRow, bytes,
                    &bars->full[stage]);
    }
    bulk_copy_g2s(dst + 2 * kChunk * kRow,
                  static_cast<const unsigned char*>(a.q_new) + ((int64_t)fi.i * a.h_q + fi.h0) * kRow, qbytes,
                  &bars->full[stage]);
    ++issued[stage];
  };
  if (L::kStages > 1 && tid == 0)
    for (int k = 0; k < L::kStages - 1 && x_begin + k < x_end; ++k) issue(x_begin + k, k);

  // ------------------------------------------------------------------ compute warps
  int* counters = reinterpret_cast<int*>(a.ws + a.layout.counters);
  float* partials = reinterpret_cast<float*>(a.ws + a.layout.partials);
  const int pstride = GT * (D + 2);
  const int half = lane >> 4, hl = lane & 15;  // half-warp and lane inside it
  constexpr int kDimL = D / 16;                // dims per lane in the score phase (8 or 4)
  constexpr int kDG = D / 8;                   // 8-dim groups per row in the PV phase (16 or 8)
  constexpr int kRG = kComputeThreads / kDG;   // PV row groups (16 or 32)
  const int dg = tid % kDG, rg = tid / kDG;
  unsigned long long o2[GT][4];               // this thread's share of the running output
  uint32_t iter = 0;

  for (int x = x_begin; x < x_end; ++x, ++iter) {
    const ItemInfo fi = dec::decode_item<kHB>(a, item_base, meta, x, n_hblocks);
    if (L::kStages == 1) {  // single stage: refill it once every thread is done with it
      named_sync();
      if (tid == 0) issue(x, 0);
    }
    const int s = iter % L::kStages;
    const uint32_t round = iter / L::kStages;
    unsigned char* kst = smem + L::kStage + s * L::kStageBytes;
    unsigned char* vst = kst + kChunk * kRow;
    const unsigned char* qst = kst + 2 * kChunk * kRow;
    const int nr = fi.p1 - fi.p0;  // rows of this chunk, the new row included
    const bool piece_first = (x == x_begin) || fi.c == 0;
    const bool piece_last = (x == x_end - 1) || fi.c == fi.nch - 1;
    if (piece_first) {
#pragma unroll
      for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[g][e] = 0ull;
    }

    bool landed = mbar_wait(&bars->full[s], round & 1, abort_flag, budget);
    // timeout test hook: before its first chunk CTA 0 waits on a barrier nothing arrives on
    if (a.test_stall && blockIdx.x == 0 && iter == 0) landed = mbar_wait(&bars->stall, 0, abort_flag, budget) && landed;
    if (!named_sync_and(landed)) {
      if (tid == 0) {
        set_status(a.dev_status, ST_TIMEOUT);
        sched[2] = ST_TIMEOUT;  // a step's lens advance is skipped
        *abort_flag = 1;
      }
      break;
    }
    // every thread is past chunk x-1: its stage takes chunk x + kStages - 1
    if (L::kStages > 1 && tid == 0 && x + L::kStages - 1 < x_end)
      issue(x + L::kStages - 1, (iter + L::kStages - 1) % L::kStages);
    // the new row: into this chunk's shared rows and, once per (question, kv head), the pool
    if (fi.len < fi.p1) {
      const int r = fi.len - fi.p0;
      const int64_t src = ((int64_t)fi.i * a.h_kv + fi.g) * kRow;
      const int64_t dst = (((int64_t)fi.slot * a.h_kv + fi.g) * a.cap + fi.len) * kRow;
      for (int e = tid; e < kRow / 16; e += kComputeThreads) {
        const uint4 kw = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.k_new) + src + 16 * e);
        const uint4 vw = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.v_new) + src + 16 * e);
        *reinterpret_cast<uint4*>(kst + r * kRow + 16 * e) = kw;
        *reinterpret_cast<uint4*>(vst + r * kRow + 16 * e) = vw;
        if (fi.hb == 0) {
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(a.pool_k) + dst + 16 * e) = kw;
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(a.pool_v) + dst + 16 * e) = vw;
        }
      }
      named_sync();
    }

    // ---- scores: half-warp per row, 4 rows per block, 16 rows per warp ----------------
    {
      unsigned long long q2[GT][kDimL / 2];
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        if (g < fi.nh) {
          if (kDimL == 8) {
            unsigned long long t[4];
            E::load8(qst + g * kRow + hl * kDimL * EB, t);
#pragma unroll
            for (int e = 0; e < kDimL / 2; ++e) q2[g][e] = t[e];
          } else {
            const unsigned char* qp = qst + g * kRow + hl * kDimL * EB;
            if (EB == 2) {
              const uint2 w = *reinterpret_cast<const uint2*>(qp);
              q2[g][0] = bf2_to_f2(w.x);
              q2[g][1 % (kDimL / 2)] = bf2_to_f2(w.y);
            } else {
              const uint4 w = *reinterpret_cast<const uint4*>(qp);
              q2[g][0] = (unsigned long long)w.x | ((unsigned long long)w.y << 32);
              q2[g][1 % (kDimL / 2)] = (unsigned long long)w.z | ((unsigned long long)w.w << 32);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < kDimL / 2; ++e) q2[g][e] = 0ull;
        }
      }
      const float sl2 = a.scale * 1.4426950408889634f;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int rbase = warp * 16 + half * 8 + blk * 4;
        float acc[4][GT];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = rbase + k;
          unsigned long long kv[4] = {0ull, 0ull, 0ull, 0ull};
          if (r < nr) {
            const unsigned char* kp = kst + r * kRow + hl * kDimL * EB;
            if (kDimL == 8) {
              E::load8(kp, kv);
            } else if (EB == 2) {
              const uint2 w = *reinterpret_cast<const uint2*>(kp);
              kv[0] = bf2_to_f2(w.x);
              kv[1] = bf2_to_f2(w.y);
            } else {
              const uint4 w = *reinterpret_cast<const uint4*>(kp);
              kv[0] = (unsigned long long)w.x | ((unsigned long long)w.y << 32);
              kv[1] = (unsigned long long)w.z | ((unsigned long long)w.w << 32);
            }
          }
#pragma unroll
          for (int g = 0; g < GT; ++g) {
            unsigned long long p2 = 0ull;
#pragma unroll
            for (int e = 0; e < kDimL / 2; ++e) p2 = fma2(q2[g][e], kv[e], p2);
            const float2 pf = unpack2(p2);
            acc[k][g] = pf.x + pf.y;
          }
        }
        // reduce-scatter over the 16 lanes of the half-warp
        float b[2][GT];
        const bool up8 = hl & 8, up4 = hl & 4;
#pragma unroll
        for (int g = 0; g < GT; ++g) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const float send = up8 ? acc[kk][g] : acc[kk + 2][g];
            const float keep = up8 ? acc[kk + 2][g] : acc[kk][g];
            b[kk][g] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
          }
        }
        const int r = rbase + (up8 ? 2 : 0) + (up4 ? 1 : 0);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          const float send = up4 ? b[0][g] : b[1][g];
          const float keep = up4 ? b[1][g] : b[0][g];
          float c = keep + __shfl_xor_sync(0xffffffffu, send, 4);
          c += __shfl_xor_sync(0xffffffffu, c, 2);
          c += __shfl_xor_sync(0xffffffffu, c, 1);
          if ((hl & 3) == 0) sc[g * kChunk + r] = r < nr ? c * sl2 : -INFINITY;
        }
      }
    }
    named_sync();

    // ---- online softmax over the piece: one warp per head --------------------------------
    if (warp < GT) {
      const int g = warp;
      float v[kChunk / 32];
      float mc = -INFINITY;
#pragma unroll
      for (int k = 0; k < kChunk / 32; ++k) {
        v[k] = sc[g * kChunk + lane + 32 * k];
        mc = fmaxf(mc, v[k]);
      }
      mc = warp_max(mc);
      const float m_old = piece_first ? -INFINITY : st_m[g];
      const float l_old = piece_first ? 0.f : st_l[g];
      const float m_new = fmaxf(m_old, mc);  // finite: every chunk holds at least one row
      float l = 0.f;
#pragma unroll
      for (int k = 0; k < kChunk / 32; ++k) {
        const float pv = ex2_approx(v[k] - m_new);  // rows past the chunk: exp2(-inf) = 0
        pw[(lane + 32 * k) * GT + g] = pv;
        l += pv;
      }
      l = warp_sum(l);
      __syncwarp();
      if (lane == 0) {
        const float alpha = ex2_approx(m_old - m_new);  // first chunk of a piece: exp2(-inf) = 0
        st_a[g] = alpha;
        st_m[g] = m_new;
        st_l[g] = l_old * alpha + l;
      }
    }
    named_sync();

    // ---- PV: lanes across dims, row groups; running output rescaled by alpha ------------
    {
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const float al = st_a[g];
        const unsigned long long aa = f2pack(al, al);
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[g][e] = fma2(aa, o2[g][e], 0ull);
      }
      for (int r = rg; r < nr; r += kRG) {
        unsigned long long vv[4];
        E::load8(vst + r * kRow + dg * 8 * EB, vv);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          const float pr = pw[r * GT + g];
          const unsigned long long pp = f2pack(pr, pr);
#pragma unroll
          for (int e = 0; e < 4; ++e) o2[g][e] = fma2(pp, vv[e], o2[g][e]);
        }
      }
      // rows are read; order these reads before the bulk copy that refills the stage
      fence_proxy_async_smem();
    }
    if (!piece_last) continue;

    // ---- end of a piece: sum the row groups, then output or partial + ordered merge -----
    {
      float o[GT][8];
#pragma unroll
      for (int g = 0; g < GT; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 t = unpack2(o2[g][e]);
          o[g][2 * e] = t.x;
          o[g][2 * e + 1] = t.y;
        }
#pragma unroll
      for (int off = kDG; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < GT; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], off);
      // warps 4-7 hand their sums to warps 0-3 (fixed order: the result is deterministic)
      if (warp >= 4 && lane < kDG) {
#pragma unroll
        for (int g = 0; g < GT; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) red[((warp - 4) * GT + g) * D + dg * 8 + e] = o[g][e];
      }
      named_sync();
      if (warp < 4 && lane < kDG) {
#pragma unroll
        for (int g = 0; g < GT; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) red[(warp * GT + g) * D + dg * 8 + e] += o[g][e];
      }
    }
    named_sync();
    const int x0 = x - fi.c;                         // first chunk of this (question, kv head, block)
    const int c_start = max(x_begin, x0) - x0;       // first chunk of this piece
    const bool whole = (c_start == 0) && (fi.c == fi.nch - 1);
    const int cidx = (fi.i * a.h_kv + fi.g) * n_hblocks + fi.hb;
    float* part = partials + ((int64_t)cidx * a.layout.max_chunks + c_start) * pstride;
    for (int e = tid; e < GT * D; e += kComputeThreads) {
      const int g = e / D, dd = e % D;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) acc += red[(w * GT + g) * D + dd];
      if (g >= fi.nh) continue;
      if (whole) {
        E::store(a.out, ((int64_t)fi.i * a.h_q + fi.h0 + g) * D + dd, acc / st_l[g]);
      } else {
        part[g * D + dd] = acc;
        if (dd == 0) {
          part[GT * D + g] = st_m[g];
          part[GT * D + GT + g] = st_l[g];
        }
      }
    }
    if (!whole) {
      __threadfence();  // this CTA's partial is visible before its arrival is counted
      named_sync();
      if (tid == 0) {
        const int b_first = range_owner(x0, total, nb), b_last = range_owner(x0 + fi.nch - 1, total, nb);
        bars->last = (atomicAdd(&counters[cidx], 1) == b_last - b_first);
      }
      named_sync();
      if (bars->last) {
        __threadfence();
        const int b_first = range_owner(x0, total, nb), b_last = range_owner(x0 + fi.nch - 1, total, nb);
        const float* base = partials + (int64_t)cidx * a.layout.max_chunks * pstride;
        for (int e = tid; e < GT * D; e += kComputeThreads) {
          const int g = e / D, dd = e % D;
          if (g >= fi.nh) continue;
          float M = -INFINITY;
          for (int b = b_first; b <= b_last; ++b) {
            const int cs = max(range_start(b, total, nb), x0) - x0;
            M = fmaxf(M, __ldcg(base + cs * pstride + GT * D + g));
          }
          float Lsum = 0.f, O = 0.f;
          for (int b = b_first; b <= b_last; ++b) {
            const int cs = max(range_start(b, total, nb), x0) - x0;
            const float* pc = base + cs * pstride;
            const float w = ex2_approx(__ldcg(pc + GT * D + g) - M);
            Lsum += __ldcg(pc + GT * D + GT + g) * w;
            O += __ldcg(pc + g * D + dd) * w;
          }
          E::store(a.out, ((int64_t)fi.i * a.h_q + fi.h0 + g) * D + dd, O / Lsum);
        }
        if (tid == 0) counters[cidx] = 0;
      }
    }
    named_sync();
  }
  // every copy lands before the CTA leaves
  if (tid == 0) {
    for (int st = 0; st < L::kStages; ++st)
      if (issued[st]) mbar_wait(&bars->full[st], (issued[st] - 1) & 1, never, kDrainBudget);
  }
}

// fp32 decode at head dims other than 64 and 128 (any multiple of 16 up to 256): the same
// validation prologue (nothing is written unless every live question is valid), then one warp
// per (live question, q-head), the online softmax over positions 0..n in blocks of 32 (lane j
// scores position j of the block; dims lane, lane + 32, ... for the output), the new position
// read from k_new / v_new; the first q-head of each kv group writes the new row into the pool.
// No split over the positions, so no workspace is used beyond the prologue's shared memory.
constexpr int kSimpleWarps = 8;
constexpr int kSimpleMaxD = 256;

template <int PER>
__global__ void __launch_bounds__(kSimpleWarps * 32) decode_simple_kernel(DecodeArgs a, int D) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float q_s[kSimpleWarps][kSimpleMaxD];
  __shared__ int s_flags;
  __shared__ int s_scan[kSimpleWarps + 1];
  const int n = a.n;
  int* item_base = reinterpret_cast<int*>(smem);
  int2* meta = reinterpret_cast<int2*>(smem + (size_t)((n + 2) / 2) * 8);
  int* hash = reinterpret_cast<int*>(smem + (size_t)((n + 2) / 2) * 8 + (size_t)n * 8);
  int* sched = reinterpret_cast<int*>(a.ws + a.layout.sched);  // [2]: this call's validation code
  if (dec::prologue<kSimpleWarps * 32>(a, 1, item_base, meta, hash, &s_flags, s_scan, &sched[2]) < 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* Qn = static_cast<const float*>(a.q_new);
  const float* Kn = static_cast<const float*>(a.k_new);
  const float* Vn = static_cast<const float*>(a.v_new);
  float* PK = static_cast<float*>(a.pool_k);
  float* PV = static_cast<float*>(a.pool_v);
  float* O = static_cast<float*>(a.out);
  const int64_t items = (int64_t)n * a.h_q;
  for (int64_t it = (int64_t)blockIdx.x * kSimpleWarps + warp; it < items; it += (int64_t)gridDim.x * kSimpleWarps) {
    const int i = (int)(it / a.h_q), h = (int)(it % a.h_q);
    if (!a.active[i]) continue;
    const int len = meta[i].x, slot = meta[i].y, g = h / a.group;
    const float* krow_new = Kn + ((int64_t)i * a.h_kv + g) * D;
    const float* vrow_new = Vn + ((int64_t)i * a.h_kv + g) * D;
    const int64_t pool0 = (((int64_t)slot * a.h_kv + g) * a.cap) * D;  // row 0 of the slot, kv head g
    __syncwarp();
    for (int c = lane; c < D; c += 32) q_s[warp][c] = Qn[((int64_t)i * a.h_q + h) * D + c];
    if (h % a.group == 0)  // the new row: appended once per (question, kv head)
      for (int c = lane; c < D; c += 32) {
        PK[pool0 + (int64_t)len * D + c] = krow_new[c];
        PV[pool0 + (int64_t)len * D + c] = vrow_new[c];
      }
    __syncwarp();
    float m = -INFINITY, l = 0.f;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int kb = 0; kb <= len; kb += 32) {
      const int pos = kb + lane;
      float sc = -INFINITY;
      if (pos <= len) {
        const float* kr = pos < len ? PK + pool0 + (int64_t)pos * D : krow_new;
        float dot = 0.f;
#pragma unroll 8
        for (int c = 0; c < D; ++c) dot = fmaf(q_s[warp][c], kr[c], dot);
        sc = dot * a.scale;
      }
      const float m_new = fmaxf(m, warp_max(sc));
      const float alpha = expf(m - m_new);  // m = -inf on the first block gives 0
      const float pw = (pos <= len) ? expf(sc - m_new) : 0.f;
      l = l * alpha + warp_sum(pw);
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] *= alpha;
      const int nk = min(32, len - kb + 1);
      for (int j = 0; j < nk; ++j) {
        const float pj = __shfl_sync(0xffffffffu, pw, j);
        const float* vr = (kb + j < len ? PV + pool0 + (int64_t)(kb + j) * D : vrow_new) + lane;
#pragma unroll
        for (int e = 0; e < PER; ++e)
          if (lane + 32 * e < D) acc[e] = fmaf(pj, vr[32 * e], acc[e]);
      }
      m = m_new;
    }
    const float inv = 1.f / l;
    float* orow = O + ((int64_t)i * a.h_q + h) * D + lane;
#pragma unroll
    for (int e = 0; e < PER; ++e)
      if (lane + 32 * e < D) orow[32 * e] = acc[e] * inv;
  }
}

cudaError_t launch_decode_simple(const DecodeArgs& a, int d, int num_sms, cudaStream_t s) {
  if (d < 16 || d > kSimpleMaxD || d % 16) return cudaErrorInvalidValue;
  int hs = 1;
  while (hs < 2 * a.n) hs <<= 1;
  const size_t smem = (size_t)((a.n + 2) / 2) * 8 + (size_t)a.n * 8 + (size_t)hs * 4;
  auto kern = d <= 64 ? decode_simple_kernel<2> : d <= 128 ? decode_simple_kernel<4> : decode_simple_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, kSimpleWarps * 32, smem, s>>>(a, d);
  return cudaGetLastError();
}

__global__ void advance_kernel(int32_t* lens, const uint8_t* active, int32_t n, const int32_t* code) {
  if (code && *code != ST_OK) return;  // kev_decode_step after an invalid (or timed-out) step: lens kept
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && active[i]) lens[i] += 1;
}

template <typename T, int D, int GT, int NS>
cudaError_t launch_stages(const DecodeArgs& args, int num_sms, cudaStream_t s) {
  using L = DSmem<D, (int)sizeof(T), GT, NS>;
  static_assert(L::kStages * L::kStageBytes >= 2 * kMaxQuestions * 4, "the validation hash lives in the stages");
  DecodeArgs a = args;
  a.wait_budget = wait_budget_cycles();
  a.test_stall = test_stall_requested();
  const int smem = L::bytes(a.n);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, GT, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_kernel<T, D, GT, NS><<<num_sms, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// Deepest stage ring that fits the shared-memory budget for this many questions.
template <typename T, int D, int GT>
cudaError_t launch_one(const DecodeArgs& a, int num_sms, cudaStream_t s) {
  constexpr int kMaxSmem = 232448;
  if (DSmem<D, (int)sizeof(T), GT, 3>::bytes(a.n) <= kMaxSmem) return launch_stages<T, D, GT, 3>(a, num_sms, s);
  if (DSmem<D, (int)sizeof(T), GT, 2>::bytes(a.n) <= kMaxSmem) return launch_stages<T, D, GT, 2>(a, num_sms, s);
  return launch_stages<T, D, GT, 1>(a, num_sms, s);
}

template <typename T, int D>
cudaError_t launch_d(const DecodeArgs& a, int num_sms, cudaStream_t s) {
  const int g = a.group < kHB ? a.group : kHB;
  if (g <= 1) return launch_one<T, D, 1>(a, num_sms, s);
  if (g <= 2) return launch_one<T, D, 2>(a, num_sms, s);
  if (g <= 4) return launch_one<T, D, 4>(a, num_sms, s);
  return launch_one<T, D, 8>(a, num_sms, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int d, kev_dtype dt, int num_sms, cudaStream_t s) {
  if (dt == KEV_FP32) {
    if (d != 64 && d != 128) return launch_decode_simple(a, d, num_sms, s);
    return d == 64 ? launch_d<float, 64>(a, num_sms, s) : launch_d<float, 128>(a, num_sms, s);
  }
  return d == 64 ? launch_d<__nv_bfloat16, 64>(a, num_sms, s) : launch_d<__nv_bfloat16, 128>(a, num_sms, s);
}

cudaError_t launch_advance(int32_t* lens, const uint8_t* active, int32_t n, cudaStream_t s, const int32_t* code) {
  if (n <= 0) return cudaSuccess;
  advance_kernel<<<(n + 255) / 256, 256, 0, s>>>(lens, active, n, code);
  return cudaGetLastError();
}

}  // namespace kev
