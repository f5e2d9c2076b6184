// Packed prefill attention on CTA pairs of the 5th-generation tensor cores (bf16, d = 128).
//
// The same attention as the single-CTA kernel (kev_prefill_tc.cu): for every query tile m of
// question i and q-head h, softmax(scale q k^T + M) v over key tiles 0..m of the question,
// with the element mask key <= row on the diagonal tile only (inference-engine notes,
// sakurs2.com, §2.1; the causal AND block-diagonal mask of the Kev articles, icman.com.cn §2.3,
// gsyq.cn §2.2), FlashAttention-style with an online softmax (notes §2.4).
//
// Here two CTAs of a cluster share every MMA: tcgen05.mma.cta_group::2 with M = 256 rows, 128
// from each CTA.  The 128 keys of a K tile (the B operand of S = Q K^T) are split 64/64
// between the two CTAs' shared memory and the 128 dims of a V tile (the B operand of
// O += P V) 64/64, so each SM reads only half of every K and V tile from its shared memory
// and loads only half of it: per key step and SM, (4 + 2) KB per S MMA and 2 KB per PV MMA
// instead of 8 KB and 4 KB -- shared-memory traffic drops from the full MMA time to ~60 % of
// it, which is what held the single-CTA MMAs at ~1.5x their issue time.
//
// A work unit (built by the segment builder) is two 256-row MMA tiles A and B of one
// (question, kv head): each is two "halves" of 128 query rows -- (query tile, q-head) --
// the even CTA's and the odd CTA's.  A and B share every K/V tile; the tensor core
// alternates between them so one tile's softmax runs while the other's MMAs execute.
//
// Roles (384 threads per CTA):
//   warps 0-3 / 4-7   softmax of this CTA's half of tile A / B (a query row per thread)
//                     and the epilogue of that half
//   warp 8            K/V producer: this CTA's half of each K tile (64 keys) and V tile (64
//                     dims) into a 6-slot ring; completion is counted on the even CTA's barrier
//   warp 10           Q producer: this CTA's query halves of tiles A and B
//   warps 9 / 11      (even CTA only) MMA issuers of tile A / B, in strict turns
// The odd CTA's softmax warps signal the even CTA's barriers remotely; every MMA completion
// is committed to the barriers of both CTAs.  Every wait is bounded; on a timeout the kernel
// stores KEV_ERR_TIMEOUT, raises the abort flag, drains what it issued and leaves through
// the final cluster barrier with its pair.
#include <cuda.h>

#include "kev_internal.cuh"
#include "kev_sm100.cuh"

namespace kev {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kBM = 128;              // query rows per half
constexpr int kBN = 128;              // keys per tile
constexpr int kRingSlots = 6;         // K(j) reuses the slot of K(j-3): loads start ~3 key steps ahead
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kQProducerWarp = 10;
constexpr int kRegsControl = 80;
constexpr int kRegsSoftmax = 208;     // 128 x 80 + 256 x 208 = 63488 <= 384 x 168 (launch bound)
constexpr uint32_t kTmemCols = 512;   // S_A, S_B, O_A, O_B: 128 columns each
constexpr float kOverflowSum = 1.8446744e19f;

constexpr long long kDrainBudget = 4000000000ll;

struct PairParams {
  char* ws;
  PrefillLayout layout;
  const kev_interval* intervals;
  void* out;
  int32_t h_q;
  int32_t group;
  float scale_log2;
  int32_t* dev_status;
  long long wait_budget;
  int32_t test_stall;
  // slot write of every whole 128-row K/V tile (store_tiles): pool row of (slot, kv head g,
  // position j) is (slot * h_kv + g) * cap + j
  const int32_t* slot_ids;
  int32_t h_kv;
  int32_t cap;
  int32_t n_slots;
  int32_t store_tiles;
};

struct Smem {
  static constexpr int kQTile = kBM * kD * 2;        // 32 KB: a query half, 2 sub-tiles of 128 rows x 128 B
  static constexpr int kQSub = kBM * 128;
  static constexpr int kSlot = 16384;                // half a K tile (64 keys, 2 sub-tiles) or half a V tile
  static constexpr int kKSub = 64 * 128;             // 64 keys x 128 B
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + 2 * kQTile;
  static constexpr int kStage = kRing + kRingSlots * kSlot;  // output stage, TMA-store box layout
  static constexpr int kBar = kStage + kQTile;
  static constexpr int kBytes = kBar + 1024;
  static constexpr int kLaunchBytes = kBytes + 1024;
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t r_full[kRingSlots], r_empty[kRingSlots];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t stg_free[4];
  uint64_t drain[2];
  uint64_t stall;
  uint32_t tmem_base;
  int abort;
  int never;
};

__device__ __forceinline__ void raise_timeout(const PairParams& p, Bars* b) {
  PrefillHeader* hdr = reinterpret_cast<PrefillHeader*>(p.ws);
  atomicCAS(&hdr->status, 0, ST_TIMEOUT);
  set_status(p.dev_status, ST_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b->abort) = 1;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          long long budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(0xffffffffu, ok);
}

// One half: (query tile, q-head) of 128 rows, as this CTA sees it.
struct Half {
  bool on;
  int head, row0, rows, nkv;
};
struct Unit {
  int q, g, seg_begin, len;
  int nkv;        // key tiles the unit loads
  int nkv_t[2];   // per MMA tile (0: absent)
  int s[4];       // halves: A even, A odd, B even, B odd
};

__device__ __forceinline__ Unit load_unit(const int4* units, const kev_interval* iv, int u) {
  const int4 w0 = units[2 * u], w1 = units[2 * u + 1];
  Unit x;
  x.q = w0.x;
  x.g = w0.y;
  x.nkv_t[0] = w0.z & 0xffff;
  x.nkv_t[1] = w0.z >> 16;
  x.nkv = max(x.nkv_t[0], x.nkv_t[1]);
  x.s[0] = w1.x;
  x.s[1] = w1.y;
  x.s[2] = w1.z;
  x.s[3] = w1.w;
  x.seg_begin = iv[x.q].begin;
  x.len = iv[x.q].end - x.seg_begin;
  return x;
}

__device__ __forceinline__ Half half_of(const Unit& x, int t, int rank, const kev_interval* iv, int group) {
  const int s = x.s[2 * t + rank];
  Half h;
  h.on = s >= 0;
  if (!h.on) {
    h.head = h.row0 = h.rows = h.nkv = 0;
    return h;
  }
  const int m = s >> kUnitHeadBits;
  h.head = x.g * group + (s & ((1 << kUnitHeadBits) - 1));
  h.row0 = x.seg_begin + m * kBM;
  h.rows = min(kBM, iv[x.q].end - h.row0);
  h.nkv = m + 1;
  return h;
}

// Units of a cluster: round r takes unit r*C + c (r even) or r*C + C-1-c (r odd).
__device__ __forceinline__ int snake(int r, int c, int C) { return r * C + ((r & 1) ? C - 1 - c : c); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                        const __grid_constant__ CUtensorMap tm_pk, const __grid_constant__ CUtensorMap tm_pv,
                        const PairParams p) {
  using L = Smem;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_cta_rank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  pdl_wait();  // the segment builder's work list is complete
  pdl_trigger();
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(p.ws);
  // both CTAs of a cluster read the same words, so they leave here together or not at all
  if (hdr->status != ST_OK) return;
  if (hdr->format != 1) {  // the work list was built for another kernel (another shape)
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.dev_status, KEV_ERR_INVALID_ARG);
    return;
  }
  const int n_units = hdr->n_items;
  if (cid >= n_units) return;
  const int4* units = reinterpret_cast<const int4*>(p.ws + p.layout.items);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 2);
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&bars->r_full[s], 1);
      mbar_init(&bars->r_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 8);  // 4 softmax warps of each CTA
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_free[t], 8);
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
    if (p.store_tiles) {
      tma_prefetch_desc(&tm_pk);
      tma_prefetch_desc(&tm_pv);
    }
  }
  if (warp == kMmaWarp) {  // the same columns in both CTAs
    tmem_alloc_pair(&bars->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  const volatile int* never = &bars->never;
  const long long budget = p.wait_budget;
  const bool leader = rank == 0;
  // the even CTA's barriers, as shared::cluster addresses
  const uint32_t cl_q_full = mapa_rank(smem_u32(&bars->q_full), 0);

  if (warp >= kProducerWarp) {
    regs_dec<kRegsControl>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------------- K/V producer
      // Sequence 2j is K(j) (this CTA's 64 keys), 2j + 1 is V(j) (this CTA's 64 dims).  The even
      // CTA arms each slot's barrier for both CTAs' bytes; the odd CTA's copies complete on it.
      // With store_tiles, the tiles this CTA holds of every whole 128-row key tile j of a
      // (question, kv head) also go to the slot pool, once: from the unit with the half of q-head 0
      // of the group at query tile j, at its key step j.  A slot's tile is stored when its MMAs
      // are done with it and the slot is about to be refilled (or at the end).
      if (lane == 0) {
        uint32_t seq = 0;
        uint32_t loads[kRingSlots] = {};
        int pend[kRingSlots];  // pool row of the key tile a slot holds for the slot write, or -1
        for (int s = 0; s < kRingSlots; ++s) pend[s] = -1;
        auto flush = [&](int s) {  // slot s: K (even) or V (odd) of this CTA, into the pool
          unsigned char* src = smem + L::kRing + s * L::kSlot;
          if (s & 1) {  // all 128 keys, dims [64 rank, 64 rank + 64)
            tma_store_2d(&tm_pv, src, rank * 64, pend[s]);
          } else {      // keys [64 rank, 64 rank + 64), all 128 dims
            tma_store_2d(&tm_pk, src, 0, pend[s] + 64 * rank);
            tma_store_2d(&tm_pk, src + L::kKSub, 64, pend[s] + 64 * rank);
          }
          bulk_commit_group();
          pend[s] = -1;
        };
        bool ok = !(p.test_stall && blockIdx.x == 0) || mbar_wait(&bars->stall, 0, abort_flag, budget);
        for (int rnd = 0, u = cid; u < n_units && ok; u = snake(++rnd, cid, ncl)) {
          const Unit x = load_unit(units, p.intervals, u);
          const int slot = p.store_tiles ? p.slot_ids[x.q] : -1;
          for (int j = 0; j < x.nkv && ok; ++j) {
            bool store = slot >= 0 && slot < p.n_slots && (j + 1) * kBN <= min(x.len, p.cap);
            if (store) {
              bool head0 = false;
              for (int k = 0; k < 4; ++k)
                head0 |= x.s[k] >= 0 && (x.s[k] & ((1 << kUnitHeadBits) - 1)) == 0 && (x.s[k] >> kUnitHeadBits) == j;
              store = head0;
            }
            for (int is_v = 0; is_v < 2; ++is_v, ++seq) {
              const int s = seq % kRingSlots;
              const uint32_t round = seq / kRingSlots;
              if (round > 0 && !mbar_wait(&bars->r_empty[s], (round - 1) & 1, abort_flag, budget)) {
                ok = false;
                break;
              }
              if (pend[s] >= 0) {  // its MMAs are done: store the old tile, then let the new one in
                flush(s);
                bulk_wait_read_all();
              }
              pend[s] = store ? (int)(((int64_t)slot * p.h_kv + x.g) * p.cap + j * kBN) : -1;
              if (leader) mbar_arrive_expect_tx(&bars->r_full[s], 2 * L::kSlot);
              unsigned char* dst = smem + L::kRing + s * L::kSlot;
              const uint32_t bar = mapa_rank(smem_u32(&bars->r_full[s]), 0);
              const int key0 = x.seg_begin + j * kBN;
              if (is_v) {  // all 128 keys, dims [64 rank, 64 rank + 64)
                tma_load_2d_pair(dst, &tm_v, x.g * kD + rank * 64, key0, bar);
              } else {     // keys [64 rank, 64 rank + 64), all 128 dims
                tma_load_2d_pair(dst, &tm_k, x.g * kD, key0 + rank * 64, bar);
                tma_load_2d_pair(dst + L::kKSub, &tm_k, x.g * kD + 64, key0 + rank * 64, bar);
              }
              ++loads[s];
            }
          }
        }
        if (!ok) raise_timeout(p, bars);
        // the tiles still waiting for the slot write: stored once their MMAs are done
        for (int s = 0; s < kRingSlots && ok; ++s)
          if (pend[s] >= 0) {
            ok = mbar_wait(&bars->r_empty[s], (loads[s] - 1) & 1, abort_flag, budget);
            if (ok) flush(s);
          }
        bulk_wait_all();  // the stores are complete before the CTA leaves
        if (*abort_flag && leader) {  // the copies counted on this CTA's barriers land before it leaves
          for (int s = 0; s < kRingSlots; ++s)
            if (loads[s]) mbar_wait(&bars->r_full[s], (loads[s] - 1) & 1, never, kDrainBudget);
        }
      }
    } else if (warp == kQProducerWarp) {
      // ---------------------------------------------------------------- Q producer
      if (lane == 0) {
        uint32_t n = 0, q_loads = 0;
        bool ok = true;
        for (int rnd = 0, u = cid; u < n_units && ok; u = snake(++rnd, cid, ncl), ++n) {
          const Unit x = load_unit(units, p.intervals, u);
          if (n > 0 && !mbar_wait(&bars->q_empty, (n - 1) & 1, abort_flag, budget)) {
            ok = false;
            break;
          }
          if (leader) {
            int halves = 0;
            for (int k = 0; k < 4; ++k) halves += x.s[k] >= 0;
            mbar_arrive_expect_tx(&bars->q_full, halves * L::kQTile);
          }
          for (int t = 0; t < 2; ++t) {
            const Half h = half_of(x, t, rank, p.intervals, p.group);
            if (!h.on) continue;
            for (int c = 0; c < 2; ++c)
              tma_load_2d_pair(smem + L::kQ + t * L::kQTile + c * L::kQSub, &tm_q, h.head * kD + c * 64, h.row0,
                               cl_q_full);
          }
          ++q_loads;
          const int u_next = snake(rnd + 1, cid, ncl);
          if (u_next < n_units) {  // the next unit's query rows into L2 while this one runs
            const Unit nx = load_unit(units, p.intervals, u_next);
            for (int t = 0; t < 2; ++t) {
              const Half h = half_of(nx, t, rank, p.intervals, p.group);
              if (!h.on) continue;
              for (int c = 0; c < 2; ++c) tma_prefetch_l2_2d(&tm_q, h.head * kD + c * 64, h.row0);
            }
          }
        }
        if (!ok) raise_timeout(p, bars);
        if (*abort_flag && leader && q_loads) mbar_wait(&bars->q_full, (q_loads - 1) & 1, never, kDrainBudget);
      }
    } else if (leader) {
      // ---------------------------------------------------------------- MMA issuers (even CTA)
      // Warp 9 issues tile A's MMAs, warp 11 tile B's, in strict turns (A's group of a key step,
      // then B's), handed over with named barriers: each waits while the other issues, and tile
      // B's softmax runs while tile A's MMAs execute and the other way round.  Every commit goes
      // to the barriers of both CTAs.
      const int t = warp == kMmaWarp ? 0 : 1;  // warp 11 issues tile B
      const bool issuer = lane == 0;
      constexpr uint32_t idesc_s = idesc_bf16(2 * kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(2 * kBM, kD, false, true);
      uint32_t kv_iter = 0, n = 0, p_cnt = 0, units_done = 0;
      bool ok = true, first_turn = true;
      auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return;
        ok = warp_wait(bar, parity, abort_flag, budget);
        if (!ok) *abort_flag = 1;
      };
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
      auto issue_s = [&](int stage) {  // S_t = Q_t K^T: A = this tile's query halves, B = K (64 keys per CTA)
        const uint32_t q_addr = smem_u32(smem + L::kQ + t * L::kQTile);
        const uint32_t k_addr = smem_u32(smem + L::kRing + stage * L::kSlot);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t a = sdesc_sw128(q_addr + (kk >> 2) * L::kQSub + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(k_addr + (kk >> 2) * L::kKSub + (kk & 3) * 32, 16, 1024);
          umma_bf16_pair(tmem + t * kBN, a, b, idesc_s, kk > 0);
        }
        umma_commit_pair(&bars->s_full[t]);
      };
      auto issue_pv = [&](int stage, bool accumulate) {  // O_t += P_t V: P from TMEM, V's 64 dims per CTA
        const uint32_t v_addr = smem_u32(smem + L::kRing + stage * L::kSlot);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = sdesc_sw128(v_addr + kk * 16 * 128, 16384, 1024);
          umma_bf16_pair_ts(tmem + 256 + t * kD, tmem + t * kBN + kk * 8, b, idesc_o,
                            (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      auto slot = [](uint32_t q) { return (int)(q % kRingSlots); };
      auto phase = [](uint32_t q) { return (q / kRingSlots) & 1; };

      for (int rnd = 0, u = cid; u < n_units; u = snake(++rnd, cid, ncl), ++n) {
        const Unit x = load_unit(units, p.intervals, u);
        const bool mine = x.nkv_t[t] > 0;
        const int nkv_t = mine ? x.nkv_t[t] : x.nkv;  // an absent tile takes its turns, issuing nothing
        {
          const uint32_t qk = 2 * kv_iter;
          wait_ok(&bars->q_full, n & 1);
          wait_ok(&bars->r_full[slot(qk)], phase(qk));
          take_turn();
          if (ok && issuer) {
            tc_fence_after();
            if (mine) issue_s(slot(qk));
            umma_commit_pair(&bars->r_empty[slot(qk)]);
            if (nkv_t == 1) umma_commit_pair(&bars->q_empty);
          }
          pass_turn();
        }
        for (int j = 0; j < x.nkv; ++j) {
          const uint32_t ki = kv_iter + j;
          const uint32_t qv = 2 * ki + 1, qk = 2 * ki + 2;
          const int vs = slot(qv), kn = slot(qk);
          const bool has_next = j + 1 < x.nkv;
          const bool act = mine && j < nkv_t;
          const bool next_s = act && j + 1 < nkv_t;
          wait_ok(&bars->r_full[vs], phase(qv));
          if (has_next) wait_ok(&bars->r_full[kn], phase(qk));
          if (act) {
            wait_ok(&bars->p_full[t], p_cnt & 1);
            if (j == 0 && units_done > 0) wait_ok(&bars->o_free[t], (units_done - 1) & 1);
            ++p_cnt;
          }
          take_turn();
          if (ok && issuer) {
            tc_fence_after();
            if (act) {
              issue_pv(vs, j > 0);
              umma_commit_pair(&bars->r_empty[vs]);
              if (next_s) issue_s(kn);
              else umma_commit_pair(&bars->o_done[t]);
            } else {
              umma_commit_pair(&bars->r_empty[vs]);
            }
            if (has_next) umma_commit_pair(&bars->r_empty[kn]);
            if (j + 1 == nkv_t - 1) umma_commit_pair(&bars->q_empty);
          }
          pass_turn();
        }
        if (mine) ++units_done;
        kv_iter += x.nkv;
      }
      if (t == 0 && !first_turn) asm volatile("bar.sync 3, 64;" ::: "memory");
      if (!ok && issuer) raise_timeout(p, bars);
      if (issuer) {  // every MMA this thread issued is complete before TMEM is freed
        umma_commit_pair(&bars->drain[t]);
        mbar_wait(&bars->drain[t], 0, never, kDrainBudget);
      }
      __syncwarp();
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------------ softmax warps
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tm_s = tmem + t * kBN + lane_off;
    const uint32_t tm_o = tmem + 256 + t * kD + lane_off;
    const float sl2 = p.scale_log2;
    const unsigned long long sl2x2 = f2pack(sl2, sl2);
    uint32_t s_cnt = 0, o_cnt = 0, stg_uses = 0;
    bool ok = true;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
    const uint32_t cl_p_full = mapa_rank(smem_u32(&bars->p_full[t]), 0);
    const uint32_t cl_o_free = mapa_rank(smem_u32(&bars->o_free[t]), 0);
    auto arrive_leader = [&](uint32_t cl_bar) {  // one arrival per warp on the even CTA's barrier
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(cl_bar);
    };

    for (int rnd = 0, u = cid; u < n_units && ok; u = snake(++rnd, cid, ncl)) {
      const Unit x = load_unit(units, p.intervals, u);
      const Half ha = half_of(x, 0, rank, p.intervals, p.group);
      const Half hb = half_of(x, 1, rank, p.intervals, p.group);
      const bool full_a = ha.on && ha.rows == kBM, full_b = hb.on && hb.rows == kBM;
      const uint32_t my_use = stg_uses + ((t == 1 && full_a) ? 1u : 0u);
      stg_uses += (full_a ? 1u : 0u) + (full_b ? 1u : 0u);
      const int nkv = x.nkv_t[t];
      if (nkv == 0) continue;  // tile t absent from this unit: no MMA, nothing to wait for
      const Half h = t ? hb : ha;
      // rows of this warp all past the question's end (its last query tile): nothing of them is
      // stored, so their weights are neither computed nor written (their O rows stay garbage)
      const bool dead = h.rows <= quarter * 32;
      float m_run = -INFINITY, l_run = 0.f;

      for (int j = 0; j < nkv; ++j) {
        if (!warp_wait(&bars->s_full[t], s_cnt & 1, abort_flag, budget)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        if (!h.on || j >= h.nkv) {
          // an empty half, or a key tile past this half's diagonal: zero weights for the PV MMA
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_st16(tm_s + c * 16, z);
          tmem_st_wait();
          tc_fence_before();
          arrive_leader(cl_p_full);
          continue;
        }
        if (dead) {
          tc_fence_before();
          arrive_leader(cl_p_full);
          continue;
        }
        // On the diagonal tile key k is visible to row r iff k <= r, so the 32-key chunks past
        // this warp's own (c > quarter) are masked for all its rows: not loaded, their weights
        // written as zeros without an exponential (the sums and the max are unchanged: those
        // entries only ever contributed exact zeros and -inf).
        const int cmax = (j == h.nkv - 1) ? quarter : 3;
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tm_s + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        if (j == h.nkv - 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e > r) sr[c][e] = __float_as_uint(-INFINITY);
        }
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
        auto exp_tile = [&](float m) -> float {
          const unsigned long long negm = f2pack(-m, -m);
          unsigned long long accs[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
            if (c > cmax) {
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[e] = 0u;
              tmem_st16(tm_s + c * 16, pk);
              continue;
            }
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
        // The first key tile sets the reference max; later tiles reuse it unless their sum shows
        // overflow risk (scores ~2^60 above it), then the exact path: new max, O and l rescaled.
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
          // PV of the previous key tile is complete (S_t came after it): rescale O
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
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
        arrive_leader(cl_p_full);
      }
      if (!ok) break;

      // epilogue: O / l -> bf16 rows of this half
      if (!warp_wait(&bars->o_done[t], o_cnt & 1, abort_flag, budget)) {
        ok = false;
        break;
      }
      ++o_cnt;
      tc_fence_after();
      if (!h.on) {
        tc_fence_before();
        arrive_leader(cl_o_free);
        continue;
      }
      const float inv = 1.f / l_run;
      uint32_t o[kD / 32][32];
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) tmem_ld32(tm_o + c * 32, o[c]);
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) tmem_ld_wait(o[c]);
      tc_fence_before();
      arrive_leader(cl_o_free);  // O_t is in registers: the next unit's PV may start
      if (h.rows == kBM) {
        const int q = warp & 3;
        const bool okw = my_use == 0 || warp_wait(&bars->stg_free[q], (my_use - 1) & 1, abort_flag, budget);
        if (!okw) {
          ok = false;
          break;
        }
        unsigned char* stg = smem + L::kStage;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = c * 64 + k * 8;
            const uint32_t w0 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 1]) * inv);
            const uint32_t w1 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 2]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 3]) * inv);
            const uint32_t w2 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 4]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 5]) * inv);
            const uint32_t w3 = pack_bf16x2(__uint_as_float(o[col / 32][col % 32 + 6]) * inv,
                                            __uint_as_float(o[col / 32][col % 32 + 7]) * inv);
            st_shared_v4(smem_u32(stg + c * L::kQSub + r * 128 + ((k ^ (r & 7)) << 4)), w0, w1, w2, w3);
          }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = 0; c < 2; ++c)
            tma_store_2d(&tm_out, stg + c * L::kQSub + q * 32 * 128, h.head * kD + c * 64, h.row0 + q * 32);
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(&bars->stg_free[q]);
        }
        __syncwarp();
      } else if (r < h.rows) {
        __nv_bfloat16* orow = out + ((int64_t)(h.row0 + r) * p.h_q + h.head) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[c][2 * e]) * inv, __uint_as_float(o[c][2 * e + 1]) * inv);
          if (out32) {
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
    if (lane == 0) bulk_wait_all();
  }

  // The odd CTA cannot observe its own copies (they complete on the even CTA's barriers): after
  // an abort it gives them time to land before the pair leaves (a copy from global memory takes
  // microseconds; this waits ~100 us).
  if (*abort_flag && !leader && threadIdx.x == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < 200000ll) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still touch its memory
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// host side
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

bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
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

// Clusters of 2 that can be resident at once (one CTA per SM), per device.
int max_pairs(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::kLaunchBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cached[dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, int num_sms, cudaStream_t s) {
  if (a.T <= 0 || a.layout.max_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mo, mpk, mpv;
  if (!make_map(&mq, a.q, (uint64_t)a.h_q * kD, (uint64_t)a.T, 128) ||
      !make_map(&mo, a.out, (uint64_t)a.h_q * kD, (uint64_t)a.T, 32) ||
      !make_map(&mk, a.k, (uint64_t)a.h_kv * kD, (uint64_t)a.T, 64) ||
      !make_map(&mv, a.v, (uint64_t)a.h_kv * kD, (uint64_t)a.T, 128))
    return cudaErrorInvalidValue;
  if (a.store_tiles) {  // the pools as [n_slots * H_kv * cap, 128] rows, the boxes of the ring slots
    const uint64_t rows = (uint64_t)a.n_slots * a.h_kv * a.cap;
    if (!make_map(&mpk, a.pool_k, kD, rows, 64) || !make_map(&mpv, a.pool_v, kD, rows, 128))
      return cudaErrorInvalidValue;
  } else {
    mpk = mk;  // not used
    mpv = mv;
  }
  PairParams p;
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
  p.store_tiles = a.store_tiles ? 1 : 0;
  p.slot_ids = a.slot_ids;
  p.h_kv = a.h_kv;
  p.cap = a.cap;
  p.n_slots = a.n_slots;
  cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Smem::kLaunchBytes);
  if (e != cudaSuccess) return e;
  // units are at most max_items / 2; the grid is the resident pairs, or fewer
  const int64_t max_units = a.layout.max_items / 2;
  const int pairs = (int)(max_units < max_pairs(num_sms) ? max_units : max_pairs(num_sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (pairs > 0 ? pairs : 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::kLaunchBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_pair_kernel, mq, mk, mv, mo, mpk, mpv, p);
}

}  // namespace kev
