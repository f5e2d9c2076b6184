// Packed prefill attention on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// Computes, for every work item of the segment builder's list -- (question i, 128-row query
// tile m, one or two q-heads of one kv group) -- the exact attention of the inference-engine
// notes (sakurs2.com, §2.1, Z = softmax(QK^T / sqrt(d_h) + M) V) restricted by the causal AND
// block-diagonal mask of the Kev articles (icman.com.cn §2.3, gsyq.cn §2.2): the tile's rows
// read key tiles 0..m of their own question only, and only the diagonal tile m needs the
// element mask (key <= row).  Tiles are FlashAttention-style (notes §2.4): the T x T score
// matrix never leaves the chip, and the softmax is the online form with a running max m, sum
// l and a rescale of the accumulator when the max moves.
//
// GB300 mapping (one persistent CTA per SM, 384 threads = 3 warpgroups):
//   warp 8      TMA producer of the K and V tiles (128 x d each) of the shared kv head, in
//               the order K(0) V(0) K(1) V(1) ... into one 5-slot ring: a K slot is released
//               when both S MMAs have read it, a V slot after both PV MMAs, and each tile's
//               load starts 2-3 key steps ahead.  Warp 10 loads the item's query tiles (one per
//               q-head) once the previous item's last S MMA has read them.  128-byte swizzled
//               boxes, completion on mbarriers.
//   warp 9      MMA issuer, ping-pong over the two query tiles A and B: S_t = Q_t K^T into
//               TMEM (128 x 128 fp32 per tile), then O_t += P_t V with P_t read from TMEM
//               (it overwrites S_t as bf16) and V from shared memory; tcgen05.commit
//               releases stages and signals the softmax warps.  While softmax A works on
//               its tile, the tensor core runs tile B's MMAs, and the other way round.
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: each thread owns one query
//               row (its TMEM lane): tcgen05.ld of S, diagonal mask, row max on the raw
//               scores on an item's first tile only, exp2 of one fused multiply-add per
//               element (scale * log2 e folded), packed fp32x2 sums, P as bf16 back into
//               TMEM; a later tile recomputes the max and rescales O in TMEM only if its
//               exponentials approach the fp32 range (exact: O and l always share one
//               reference max).  The epilogue divides by l and stores bf16 rows;
//               rows past the question's end are not stored.
//   The control warpgroup (warps 8-11) hands registers to the softmax warpgroups (setmaxnreg),
//   so a softmax thread holds its whole 128-wide score row in registers.
// Every wait is bounded; a wait that gives up sets KEV_ERR_TIMEOUT and raises the CTA's abort
// flag, and the CTA drains its own copies and MMAs before freeing TMEM and exiting.
#include <cuda.h>
#include <stdlib.h>

#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;

constexpr int kBM = 128;            // query rows per tile
constexpr int kBN = 128;            // keys per tile
// K and V tiles share one ring, in the order K(0) V(0) K(1) V(1) ...: with 4 slots, K(j) reuses
// the slot of K(j-2) and V(j) that of V(j-2), so each tile's load starts about two key steps
// before its MMA needs it (measured: 4 slots beat 3 and 5, and free 32 KB for the output stage).
constexpr int kRingSlots = 4;
constexpr int kThreads = 384;       // 3 warpgroups
constexpr int kProducerWarp = 8;    // warpgroup 2: K/V producer, MMA issuer A, Q producer, MMA issuer B
constexpr int kMmaWarp = 9;
constexpr int kQProducerWarp = 10;
constexpr int kMmaWarpB = 11;       // MMA issuer of query tile B (warp 9 issues tile A's)
// Register split: the kernel is launched at <= 168 registers per thread (384 x 168 = 64512);
// the control warpgroup drops to 80 and the two softmax warpgroups rise to 208:
// 128 x 80 + 256 x 208 = 63488 <= 64512, so the increase can always be granted.
constexpr int kRegsControl = 80;
constexpr int kRegsSoftmax = 208;
constexpr uint32_t kTmemCols = 512;
constexpr float kOverflowSum = 1.8446744e19f;      // 2^64: a tile sum above it triggers the exact path
constexpr long long kDrainBudget = 4000000000ll;  // cycles to wait for in-flight work on abort

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
  int32_t test_stall;     // timeout test hook: CTA 0's K/V producer first waits on a barrier nothing arrives on
  // chunked prefill: K/V from the slots (the maps tm_k / tm_v are the pools' [rows, D] views)
  const int32_t* prefix_lens;
  const int32_t* slot_ids;
  int32_t h_kv;
  int32_t cap;
};

template <int D>
struct Smem {
  static constexpr int kSub = D / 64;             // 64-column (128-byte) sub-tiles per row
  static constexpr int kSubBytes = kBM * 128;     // one 128-row x 128-byte sub-tile
  static constexpr int kTileBytes = kBM * D * 2;  // one Q/K/V tile
  static constexpr int kQ = 0;                    // two query tiles
  static constexpr int kRing = kQ + 2 * kTileBytes;  // K/V ring
  static constexpr int kStage = kRing + kRingSlots * kTileBytes;  // one output tile, TMA-store box layout
  static constexpr int kBar = kStage + kTileBytes;
  static constexpr int kBytes = kBar + 1024;
  static constexpr int kLaunchBytes = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t r_full[kRingSlots], r_empty[kRingSlots];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t stg_free[4];  // slice q (rows 32q..32q+31) of the output stage has been read by its last store
  uint64_t drain[2];
  uint64_t stall;  // timeout test hook: nothing ever arrives on it
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

struct Item {
  int q, seg_begin;
  int h0;    // q-head of tile A (the kv group is h0 / group)
  int nh;    // query tiles in the item (1 or 2)
  int nkv;   // key tiles the item loads (the larger of its tiles' counts)
  bool two;  // tiles A and B are consecutive query tiles of one q-head (else: one tile, heads h0, h0+1)
  int row0a, rowsa, nkva;  // tile A: first row, rows, key tiles
  int row0b, rowsb, nkvb;  // tile B
  int kv_row0;             // chunked prefill: pool row of position 0 of the question's slot, kv head
  __device__ int row0_of(int t) const { return t ? row0b : row0a; }
  __device__ int rows_of(int t) const { return t ? rowsb : rowsa; }
  __device__ int head_of(int t) const { return two ? h0 : h0 + t; }
  __device__ int nkv_of(int t) const { return t ? nkvb : nkva; }
};
// Work item {question, row_begin, rows, first_head | n_heads << 16 | two_tiles << 30}; with
// two_tiles, the item is query tiles (row_begin, row_begin + 128) of one q-head, and `rows` is the
// second tile's row count.
__device__ __forceinline__ Item load_item(const int4* items, const kev_interval* iv, int it) {
  const int4 w = items[it];
  Item x;
  x.q = w.x;
  x.seg_begin = iv[w.x].begin;
  x.h0 = w.w & 0xffff;
  x.two = (w.w >> 30) & 1;
  x.row0a = w.y;
  x.nkva = (w.y - x.seg_begin) / kBM + 1;
  if (x.two) {
    x.nh = 2;
    x.rowsa = kBM;
    x.row0b = w.y + kBM;
    x.rowsb = w.z;
    x.nkvb = x.nkva + 1;
  } else {
    x.nh = (w.w >> 16) & 0x3fff;
    x.rowsa = x.rowsb = w.z;
    x.row0b = w.y;
    x.nkvb = x.nkva;
  }
  x.nkv = x.nkvb;
  return x;
}

// Work item of the kernel instance: a chunk's query tiles sit after the prefix_lens[q] cached
// positions of its slot (a multiple of the tile), so every tile has that many more key tiles, the
// last one still the diagonal one; its keys and values are rows of the slot.
template <bool kChunk>
__device__ __forceinline__ Item load_work(const int4* items, const TcParams& p, int it) {
  Item x = load_item(items, p.intervals, it);
  if (kChunk) {
    const int pt = p.prefix_lens[x.q] / kBM;
    x.nkva += pt;
    x.nkvb += pt;
    x.nkv += pt;
    x.kv_row0 = (p.slot_ids[x.q] * p.h_kv + x.h0 / p.group) * p.cap;
  }
  return x;
}

// Item order of a CTA: in round r it takes item r*G + b (r even) or r*G + G-1-b (r odd) of the
// longest-first list (G = grid size, b = its index), so a CTA that took one of the longest items
// of a round takes one of the shortest of the next; all roles walk the same sequence.
__device__ __forceinline__ int snake_item(int r, int b, int G) { return r * G + ((r & 1) ? G - 1 - b : b); }

template <int D, bool kChunk>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                      const TcParams p) {
  using L = Smem<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();  // the segment builder's work list is complete
  pdl_trigger();
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(p.ws);
  if (hdr->status != ST_OK) return;
  if (hdr->format != 0) {  // the work list was built for another kernel (another shape)
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.dev_status, KEV_ERR_INVALID_ARG);
    return;
  }
  const int n_items = hdr->n_items;
  if ((int)blockIdx.x >= n_items) return;
  const int4* items = reinterpret_cast<const int4*>(p.ws + p.layout.items);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 2);  // the Q tiles and the ring slots are released by both MMA issuers
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&bars->r_full[s], 1);
      mbar_init(&bars->r_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_free[t], 4);
    }
    for (int q = 0; q < 4; ++q) mbar_init(&bars->stg_free[q], 1);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    mbar_init(&bars->stall, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [256+D, 256+2D)
  volatile int* abort_flag = &bars->abort;
  const volatile int* never = &bars->never;
  const long long budget = p.wait_budget;

  if (warp >= kProducerWarp) {
  regs_dec<kRegsControl>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ K/V producer
    if (lane == 0) {
      uint32_t seq = 0;  // ring sequence: 2 ki is K(ki), 2 ki + 1 is V(ki)
      uint32_t loads[kRingSlots] = {};
      // timeout test hook: a wait that runs out (nothing arrives), then the abort path
      bool ok = !(p.test_stall && blockIdx.x == 0) || mbar_wait(&bars->stall, 0, abort_flag, budget);
      Item x_next = load_work<kChunk>(items, p, blockIdx.x);
      for (int rnd = 0, it = blockIdx.x; it < n_items && ok; it = snake_item(++rnd, blockIdx.x, gridDim.x)) {
        const Item x = x_next;  // loaded one item ahead: its latency hides behind this item
        const int it_next = snake_item(rnd + 1, blockIdx.x, gridDim.x);
        if (it_next < n_items) x_next = load_work<kChunk>(items, p, it_next);
        const int g = x.h0 / p.group;
        for (int j = 0; j < x.nkv && ok; ++j) {
          for (int is_v = 0; is_v < 2; ++is_v, ++seq) {
            const int s = seq % kRingSlots;
            const uint32_t round = seq / kRingSlots;
            if (round > 0 && !mbar_wait(&bars->r_empty[s], (round - 1) & 1, abort_flag, budget)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->r_full[s], L::kTileBytes);
            for (int c = 0; c < L::kSub; ++c)
              tma_load_2d(smem + L::kRing + s * L::kTileBytes + c * L::kSubBytes, is_v ? &tm_v : &tm_k,
                          kChunk ? c * 64 : g * D + c * 64, kChunk ? x.kv_row0 + j * kBN : x.seg_begin + j * kBN,
                          &bars->r_full[s]);
            ++loads[s];
          }
        }
      }
      if (!ok) raise_timeout(p, bars);
      if (*abort_flag) {  // every copy issued by this thread lands before the CTA leaves
        for (int s = 0; s < kRingSlots; ++s)
          if (loads[s]) mbar_wait(&bars->r_full[s], (loads[s] - 1) & 1, never, kDrainBudget);
      }
    }
  } else if (warp == kQProducerWarp) {
    // ------------------------------------------------------------------ Q producer
    if (lane == 0) {
      uint32_t n = 0, q_loads = 0;
      bool ok = true;
      Item x_next = load_work<kChunk>(items, p, blockIdx.x);
      for (int rnd = 0, it = blockIdx.x; it < n_items && ok; it = snake_item(++rnd, blockIdx.x, gridDim.x), ++n) {
        const Item x = x_next;
        const int it_next = snake_item(rnd + 1, blockIdx.x, gridDim.x);
        if (it_next < n_items) x_next = load_work<kChunk>(items, p, it_next);
        if (n > 0 && !mbar_wait(&bars->q_empty, (n - 1) & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full, x.nh * L::kTileBytes);
        for (int t = 0; t < x.nh; ++t)
          for (int c = 0; c < L::kSub; ++c)
            tma_load_2d(smem + L::kQ + t * L::kTileBytes + c * L::kSubBytes, &tm_q, x.head_of(t) * D + c * 64,
                        x.row0_of(t), &bars->q_full);
        ++q_loads;
        // pull the next item's query tiles into L2 while this item runs: their load into
        // shared memory starts only when this item's last S MMA has read the Q buffer
        if (it_next < n_items) {
          const Item& nx = x_next;
          for (int t = 0; t < nx.nh; ++t)
            for (int c = 0; c < L::kSub; ++c) tma_prefetch_l2_2d(&tm_q, nx.head_of(t) * D + c * 64, nx.row0_of(t));
        }
      }
      if (!ok) raise_timeout(p, bars);
      if (*abort_flag && q_loads) mbar_wait(&bars->q_full, (q_loads - 1) & 1, never, kDrainBudget);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarpB) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 9 issues the MMAs of query tile A, warp 11 those of tile B, taking strict turns on
    // the tensor core: A's group of a key step (PV_A, then S_A of the next key tile), then B's,
    // then A's next, handed over with named barriers (a few cycles, no shared memory).  Each
    // issuer does its waits while the other one issues, so their latency stays off the
    // tensor core, and the groups never interleave, so tile B's softmax runs while tile A's
    // MMAs execute and the other way round.  Both release the shared Q tiles and ring slots
    // (their empty barriers count two arrivals); an issuer whose tile is absent from an item
    // (a single q-head left in the group) takes its turns without issuing.  After a failed
    // wait an issuer keeps taking its turns (issuing nothing) until both reach the end.
    const int t = warp == kMmaWarp ? 0 : 1;
    const bool leader = lane == 0;
    constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
    uint32_t kv_iter = 0, n = 0, p_cnt = 0, items_done = 0;
    bool ok = true;
    bool first_turn = true;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (!ok) return;
      ok = warp_wait(bar, parity, abort_flag, budget);
      if (!ok) *abort_flag = 1;
    };
    // turn hand-over: barrier 2 = "A's group is issued", barrier 3 = "B's group is issued"
    auto take_turn = [&]() {
      if (t == 1) asm volatile("bar.sync 2, 64;" ::: "memory");
      else if (!first_turn) asm volatile("bar.sync 3, 64;" ::: "memory");
      first_turn = false;
    };
    auto pass_turn = [&]() {
      __syncwarp();
      if (t == 0) asm volatile("bar.arrive 2, 64;" ::: "memory");
      else asm volatile("bar.arrive 3, 64;" ::: "memory");
    };

    auto issue_s = [&](int stage) {
      const uint32_t q_addr = smem_u32(smem + L::kQ + t * L::kTileBytes);
      const uint32_t k_addr = smem_u32(smem + L::kRing + stage * L::kTileBytes);  // K tile's ring slot
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * L::kSubBytes + (kk & 3) * 32;
        umma_bf16(tmem + t * kBN, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idesc_s,
                  kk > 0);
      }
      umma_commit(&bars->s_full[t]);
    };
    auto issue_pv = [&](int stage, bool accumulate) {
      const uint32_t v_addr = smem_u32(smem + L::kRing + stage * L::kTileBytes);  // V tile's ring slot
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint64_t b = sdesc_sw128(v_addr + kk * 16 * 128, L::kSubBytes, 1024);
        umma_bf16_ts(tmem + 256 + t * D, tmem + t * kBN + kk * 8, b, idesc_o, (accumulate || kk > 0) ? 1u : 0u);
      }
    };
    // ring slot and phase of K(ki) (sequence 2 ki) and V(ki) (sequence 2 ki + 1)
    auto slot = [](uint32_t q) { return (int)(q % kRingSlots); };
    auto phase = [](uint32_t q) { return (q / kRingSlots) & 1; };

    Item x_next = load_work<kChunk>(items, p, blockIdx.x);
    for (int rnd = 0, it = blockIdx.x; it < n_items; it = snake_item(++rnd, blockIdx.x, gridDim.x), ++n) {
      const Item x = x_next;  // loaded one item ahead: its latency hides behind this item
      const int it_next = snake_item(rnd + 1, blockIdx.x, gridDim.x);
      if (it_next < n_items) x_next = load_work<kChunk>(items, p, it_next);
      const bool mine = t < x.nh;
      // this tile's key tiles (an absent tile runs the item's steps, releasing stages only)
      const int nkv_t = mine ? x.nkv_of(t) : x.nkv;
      {
        const uint32_t qk = 2 * kv_iter;
        wait_ok(&bars->q_full, n & 1);
        wait_ok(&bars->r_full[slot(qk)], phase(qk));
        take_turn();
        if (ok && leader) {
          tc_fence_after();
          if (mine) issue_s(slot(qk));
          umma_commit(&bars->r_empty[slot(qk)]);
          if (nkv_t == 1) umma_commit(&bars->q_empty);
        }
        pass_turn();
      }
      for (int j = 0; j < x.nkv; ++j) {
        const uint32_t ki = kv_iter + j;
        const uint32_t qv = 2 * ki + 1, qk = 2 * ki + 2;  // V(ki), K(ki + 1)
        const int vs = slot(qv), kn = slot(qk);
        const bool has_next = j + 1 < x.nkv;     // the item loads K(ki + 1)
        const bool act = mine && j < nkv_t;      // this tile uses key tile j
        const bool next_s = act && j + 1 < nkv_t;
        wait_ok(&bars->r_full[vs], phase(qv));
        if (has_next) wait_ok(&bars->r_full[kn], phase(qk));
        if (act) {
          wait_ok(&bars->p_full[t], p_cnt & 1);
          if (j == 0 && items_done > 0) wait_ok(&bars->o_free[t], (items_done - 1) & 1);
          ++p_cnt;
        }
        take_turn();
        if (ok && leader) {
          tc_fence_after();
          if (act) {
            issue_pv(vs, j > 0);
            umma_commit(&bars->r_empty[vs]);  // this issuer's use of the V tile ends with the PV
            if (next_s) issue_s(kn);          // overwrites S_t / P_t after the PV above read it (in order)
            else umma_commit(&bars->o_done[t]);
          } else {
            umma_commit(&bars->r_empty[vs]);
          }
          if (has_next) umma_commit(&bars->r_empty[kn]);
          if (j + 1 == nkv_t - 1) umma_commit(&bars->q_empty);  // this tile's last S is issued
        }
        pass_turn();
      }
      if (mine) ++items_done;
      kv_iter += x.nkv;
    }
    if (t == 0 && !first_turn) asm volatile("bar.sync 3, 64;" ::: "memory");  // B's last hand-over
    if (!ok && leader) raise_timeout(p, bars);
    // every MMA this thread issued is complete before TMEM is freed
    if (leader) {
      umma_commit(&bars->drain[t]);
      mbar_wait(&bars->drain[t], 0, never, kDrainBudget);
    }
    __syncwarp();
  }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------------ softmax warps
    const int t = warp >> 2;        // query tile of this warpgroup
    const int quarter = warp & 3;   // a warp may only touch TMEM lanes [32*(warp%4), +32)
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tm_s = tmem + t * kBN + lane_off;
    const uint32_t tm_o = tmem + 256 + t * D + lane_off;
    const float sl2 = p.scale_log2;
    const unsigned long long sl2x2 = f2pack(sl2, sl2);
    uint32_t s_cnt = 0, o_cnt = 0;
    uint32_t stg_uses = 0;  // output-stage uses before the current item (tile A's, then tile B's)
    bool ok = true;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;

    Item x_next = load_work<kChunk>(items, p, blockIdx.x);
    for (int rnd = 0, it = blockIdx.x; it < n_items && ok; it = snake_item(++rnd, blockIdx.x, gridDim.x)) {
      const Item x = x_next;  // loaded one item ahead: its latency hides behind this item
      const int it_next = snake_item(rnd + 1, blockIdx.x, gridDim.x);
      if (it_next < n_items) x_next = load_work<kChunk>(items, p, it_next);
      const bool full_a = x.rows_of(0) == kBM, full_b = x.nh == 2 && x.rows_of(1) == kBM;
      const uint32_t my_use = stg_uses + ((t == 1 && full_a) ? 1u : 0u);  // tile A's use comes first
      stg_uses += (full_a ? 1u : 0u) + (full_b ? 1u : 0u);
      if (t >= x.nh) continue;
      const int nkv = x.nkv_of(t), rows_t = x.rows_of(t), row0_t = x.row0_of(t), head_t = x.head_of(t);
      float m_run = -INFINITY, l_run = 0.f;

      for (int j = 0; j < nkv; ++j) {
        if (!warp_wait(&bars->s_full[t], s_cnt & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        // the whole 128-wide score row of this thread, one load round trip
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tm_s + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        if (j == nkv - 1) {  // diagonal tile: key k is visible to row r iff k <= r
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e > r) sr[c][e] = __float_as_uint(-INFINITY);
        }
        // Row max (8 independent partial maxima, then combined), in scaled log2 units.
        auto row_max = [&]() -> float {
          float mp[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            mp[q] = fmax3(__uint_as_float(sr[q >> 1][(q & 1) * 16]), __uint_as_float(sr[q >> 1][(q & 1) * 16 + 1]),
                          __uint_as_float(sr[q >> 1][(q & 1) * 16 + 2]));
#pragma unroll
          for (int e = 3; e < 15; e += 2)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              mp[q] = fmax3(mp[q], __uint_as_float(sr[q >> 1][(q & 1) * 16 + e]),
                            __uint_as_float(sr[q >> 1][(q & 1) * 16 + e + 1]));
#pragma unroll
          for (int q = 0; q < 8; ++q) mp[q] = fmaxf(mp[q], __uint_as_float(sr[q >> 1][(q & 1) * 16 + 15]));
          return fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * sl2;
        };
        // P = exp2(s * scale * log2e - m) as bf16 pairs into the first 64 columns of S_t (S is
        // already in registers; the PV MMA reads P from there); returns the row's sum of P.
        auto exp_tile = [&](float m) -> float {
          const unsigned long long negm = f2pack(-m, -m);
          unsigned long long accs[4] = {0ull, 0ull, 0ull, 0ull};  // independent partial sums
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const unsigned long long sv =
                  (unsigned long long)sr[c][2 * e] | ((unsigned long long)sr[c][2 * e + 1] << 32);
              const float2 a = unpack2(fma2(sv, sl2x2, negm));
              const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
              accs[e & 3] = add2(accs[e & 3], f2pack(p0, p1));
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tm_s + c * 16, pk);
          }
          const float2 acc = unpack2(add2(add2(accs[0], accs[1]), add2(accs[2], accs[3])));
          return acc.x + acc.y;
        };
        // The reference max only guards the exponentials against overflow (P is bf16 and O, l
        // accumulate in fp32: their precision is relative, whatever the reference).  So the
        // first tile of an item sets it, later tiles reuse it, and only a tile whose sum
        // signals overflow risk (its scores grew by ~2^60 over the reference) pays for a row
        // max, rescales O and l, and recomputes P: exact in every case.
        if (j == 0) m_run = row_max();
        float lt = exp_tile(m_run);
        const bool big = !(lt <= kOverflowSum);
        float alpha = 1.f;
        if (__any_sync(0xffffffffu, big)) {
          if (big) {
            const float mt = fmaxf(row_max(), m_run);
            alpha = ex2_approx(m_run - mt);
            m_run = mt;
            l_run *= alpha;
          }
          lt = exp_tile(m_run);
          // PV of the previous tile is complete (S_t came after it): rescale O
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tm_o + c * 32, o);
          }
        }
        l_run += lt;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars->p_full[t]);
      }
      if (!ok) break;

      // epilogue: O / l -> bf16 rows of this item
      if (!warp_wait(&bars->o_done[t], o_cnt & 1, abort_flag, budget)) {
        ok = false;
        break;
      }
      ++o_cnt;
      tc_fence_after();
      const float inv = 1.f / l_run;
      uint32_t o[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tm_o + c * 32, o[c]);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
      tc_fence_before();
      mbar_arrive_warp(&bars->o_free[t]);  // O_t is in registers: the next item's PV may start
      if (rows_t == kBM) {
        // A whole tile: each warp writes its 32 rows as bf16 into its slice of the output stage
        // (the 128-byte swizzled box layout) and one lane stores the slice with two bulk tensor
        // copies of 32 rows; the warp waits only for the copy engine to have read its 8 KB.
        // Tile A's use of a slice comes before tile B's (its warps 4-7 wait on warps 0-3).
        const int q = warp & 3;
        const bool okw = my_use == 0 || warp_wait(&bars->stg_free[q], (my_use - 1) & 1, abort_flag, budget);
        if (!okw) {
          ok = false;
          break;
        }
        unsigned char* stg = smem + L::kStage;
#pragma unroll
        for (int c = 0; c < L::kSub; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = c * 64 + k * 8;  // 8 columns = one 16-byte chunk
            const uint32_t w0 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 1]) * inv);
            const uint32_t w1 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 2]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 3]) * inv);
            const uint32_t w2 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 4]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 5]) * inv);
            const uint32_t w3 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 6]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 7]) * inv);
            st_shared_v4(smem_u32(stg + c * L::kSubBytes + r * 128 + ((k ^ (r & 7)) << 4)), w0, w1, w2, w3);
          }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = 0; c < L::kSub; ++c)
            tma_store_2d(&tm_out, stg + c * L::kSubBytes + q * 32 * 128, head_t * D + c * 64, row0_t + q * 32);
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(&bars->stg_free[q]);
        }
        __syncwarp();
      } else if (r < rows_t) {
        // the question's last, partial tile: row by row (a whole box would overwrite the
        // next question's rows)
        __nv_bfloat16* orow = out + ((int64_t)(row0_t + r) * p.h_q + head_t) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[c][2 * e]) * inv, __uint_as_float(o[c][2 * e + 1]) * inv);
          if (out32) {  // 32-byte stores when the output allows them (the ABI promises 16)
            st_global_v8(orow + c * 32, w);
            st_global_v8(orow + c * 32 + 16, w + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
    }
    if (!ok && lane == 0) raise_timeout(p, bars);
    if (lane == 0) bulk_wait_all();  // this lane's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

// 2-D bf16 view [rows, cols] (cols contiguous), boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const PrefillArgs& a, int num_sms, cudaStream_t s) {
  const bool chunk = a.prefix_lens != nullptr;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, (uint64_t)a.h_q * D, (uint64_t)a.T) || !make_map(&mo, a.out, (uint64_t)a.h_q * D, (uint64_t)a.T, 32))
    return cudaErrorInvalidValue;
  if (chunk) {  // keys and values: the slots as [n_slots * H_kv * cap, D] rows
    const uint64_t rows = (uint64_t)a.n_slots * a.h_kv * a.cap;
    if (!make_map(&mk, a.pool_k, D, rows) || !make_map(&mv, a.pool_v, D, rows)) return cudaErrorInvalidValue;
  } else if (!make_map(&mk, a.k, (uint64_t)a.h_kv * D, (uint64_t)a.T) ||
             !make_map(&mv, a.v, (uint64_t)a.h_kv * D, (uint64_t)a.T)) {
    return cudaErrorInvalidValue;
  }
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
  p.test_stall = test_stall_requested();
  p.prefix_lens = a.prefix_lens;
  p.slot_ids = a.slot_ids;
  p.h_kv = a.h_kv;
  p.cap = a.cap;
  const int smem = Smem<D>::kLaunchBytes;
  auto kern = chunk ? prefill_tc_kernel<D, true> : prefill_tc_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t max_items = a.layout.max_items;
  const int grid = (int)(max_items < num_sms ? max_items : num_sms);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, mq, mk, mv, mo, p);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, int d, int num_sms, cudaStream_t s) {
  if (a.T <= 0 || a.layout.max_items == 0) return cudaSuccess;
  return d == 64 ? launch_tc<64>(a, num_sms, s) : launch_tc<128>(a, num_sms, s);
}

}  // namespace kev
