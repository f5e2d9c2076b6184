// Segment descriptors: validation, cu_seqlens, gap list and the longest-first work list.
//
// The block-diagonal mask of the Kev architecture article (icman.com.cn news 75864, §2.1,
// §2.3) is never materialised: a question's intervals become tiles of 128 query rows, and
// tile m of a question is paired only with key tiles 0..m of the same question (the causal
// lower triangle of its own diagonal block).  This is the varlen "cu_seqlens" form the
// article moves to for long inputs (§5.2, §6.4), extended to a tile work list.
//
// One CTA of 512 threads; at most kMaxQuestions questions.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kThreads = 512;
// Up to this many questions the checks run as one pass of all pairs per thread out of shared
// memory (no sort, no barrier per sorting stage); larger batches use bitonic sorts.
constexpr int kSmall = 1024;

// In-place ascending bitonic sort of `n2` (power of two) keys in shared memory.
__device__ void bitonic_sort(unsigned long long* key, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const bool up = (i & k) == 0;
          const unsigned long long a = key[i], b = key[p];
          if ((a > b) == up) {
            key[i] = b;
            key[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__device__ int block_exclusive_scan(int v, int* tmp /* [kThreads/32 + 1] */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) tmp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int base = warp > 0 ? tmp[warp - 1] : 0;
  const int r = base + x - v;
  if (total) *total = tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return r;
}

// Work units of the CTA-pair prefill kernel.  A question of n query tiles has, in each kv
// group of G q-heads, the (tile, head) pairs of its causal blocks.  They are grouped into
// "pair-tiles", the 256-row MMA tiles of a CTA pair: heads (2e, 2e+1) of tile m, whose halves
// both need key tiles 0..m; with G odd, the last head's tiles m and m+1 (m even) form one
// pair-tile (its first half does one key step more than it needs, with zero weights), or tile
// m alone if it is the question's last.  In order of key-tile count, consecutive pair-tiles
// form a unit (tiles A, B, which share every K/V tile and differ by at most one key tile, two
// when G = 1); an odd count leaves a last unit with tile B absent.  The enumeration depends
// only on the question's own length, so a question's arithmetic does not depend on its
// neighbours.  Rank m (key tiles m + 1) holds E = G/2 pair-tiles, plus one more when G is odd
// and m is odd or the last rank.
struct UnitShape {
  int n, G, E, odd;
  __device__ UnitShape(int n_, int G_) : n(n_), G(G_), E(G_ >> 1), odd(G_ & 1) {}
  __device__ int pair_tiles() const { return n * E + odd * ((n + 1) >> 1); }
  __device__ int units() const { return (pair_tiles() + 1) >> 1; }
  // pair-tile p (in order of key-tile count): its two halves and key-tile count
  __device__ void pair_tile(int p, int& h0, int& h1, int& nkv) const {
    int m, k;
    if (!odd) {
      m = p / E;
      k = p - m * E;
    } else {
      const int b = p / (2 * E + 1), r = p - b * (2 * E + 1);
      m = r < E ? 2 * b : 2 * b + 1;
      k = r < E ? r : r - E;
      if (m >= n) {  // the odd head's tile n-1 alone (n odd)
        m = n - 1;
        k = E;
      }
    }
    if (k < E) {
      h0 = (m << kUnitHeadBits) | (2 * k);
      h1 = (m << kUnitHeadBits) | (2 * k + 1);
    } else if (m & 1) {  // the odd head's tiles m - 1 and m
      h0 = ((m - 1) << kUnitHeadBits) | (G - 1);
      h1 = (m << kUnitHeadBits) | (G - 1);
    } else {  // the odd head's last tile, alone
      h0 = (m << kUnitHeadBits) | (G - 1);
      h1 = -1;
    }
    nkv = m + 1;
  }
  // unit u: pair-tiles 2u (tile A) and 2u + 1 (tile B, absent past the end)
  __device__ void unit(int u, int4& w1, int& na, int& nb) const {
    int a0, a1, b0 = -1, b1 = -1;
    pair_tile(2 * u, a0, a1, na);
    nb = 0;
    if (2 * u + 1 < pair_tiles()) pair_tile(2 * u + 1, b0, b1, nb);
    w1 = make_int4(a0, a1, b0, b1);
  }
};

// Shared-memory counter add aggregated over a warp: the lanes that pass the same `key` add `v`
// each with one atomic between them (units mostly share a handful of bins, so per-lane atomics
// on one word would serialise the warp); returns this lane's old value plus v x its rank among
// those lanes.  Every lane of the warp calls it; lanes with `valid` false add nothing.
__device__ __forceinline__ int warp_aggregated_add(int* counters, int key, int v, bool valid) {
  const int lane = threadIdx.x & 31;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? key : -1);
  const int leader = __ffs(peers) - 1;
  int old = 0;
  if (valid && lane == leader) old = atomicAdd(&counters[key], v * __popc(peers));
  old = __shfl_sync(0xffffffffu, old, leader);
  return old + v * __popc(peers & ((1u << lane) - 1u));
}

// One thread per (question, unit), longest first by cost bins; `base` (shared, n + 1 ints)
// holds the questions' first unit indices.
__device__ void emit_units(const SegmentsArgs& a, PrefillHeader* hdr, int4* out, int* bin_count, int* bin_cursor,
                           int n_gaps, int* base, int* scan_tmp) {
  const int tid = threadIdx.x;
  const int h_kv = a.h_q / a.group;
  auto n_tiles = [&](int i) { return (a.intervals[i].end - a.intervals[i].begin + kTileM - 1) / kTileM; };
  __syncthreads();
  if (tid < kCostBins) bin_count[tid] = 0;
  int running = 0;
  for (int b0 = 0; b0 < a.n; b0 += blockDim.x) {
    const int i = b0 + tid;
    const int cnt = i < a.n ? UnitShape(n_tiles(i), a.group).units() : 0;
    int blk;
    const int off = block_exclusive_scan(cnt, scan_tmp, &blk);
    if (i < a.n) base[i] = running + off;
    running += blk;
  }
  const int total = running;  // units per kv head
  if (tid == 0) base[a.n] = total;
  __syncthreads();
  auto question_of = [&](int u) {
    int lo = 0, hi = a.n;  // base[lo] <= u < base[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (base[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
  };
  // a unit's cost is its key-tile count (tile B's, the larger); the loops run in whole warps
  for (int u0 = 0; u0 < total; u0 += blockDim.x) {
    const int u = u0 + tid;
    int bin = 0;
    if (u < total) {
      const int i = question_of(u);
      int4 w1;
      int na, nb;
      UnitShape(n_tiles(i), a.group).unit(u - base[i], w1, na, nb);
      bin = min(max(na, nb) - 1, kCostBins - 1);
    }
    warp_aggregated_add(bin_count, bin, h_kv, u < total);
  }
  __syncthreads();
  __shared__ int s_total;
  if (tid < 32) {  // bins in descending order
    const int hi = kCostBins - 1 - 2 * tid, lo = hi - 1;
    const int c_hi = bin_count[hi], c_lo = bin_count[lo];
    int x = c_hi + c_lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
    }
    const int b = x - (c_hi + c_lo);
    bin_cursor[hi] = b;
    bin_cursor[lo] = b + c_hi;
    if (tid == 31) s_total = x;
  }
  __syncthreads();
  for (int u0 = 0; u0 < total; u0 += blockDim.x) {
    const int u = u0 + tid;
    int i = 0, na = 0, nb = 0, bin = 0;
    int4 w1 = make_int4(0, 0, 0, 0);
    if (u < total) {
      i = question_of(u);
      UnitShape(n_tiles(i), a.group).unit(u - base[i], w1, na, nb);
      bin = min(max(na, nb) - 1, kCostBins - 1);
    }
    const int pos = warp_aggregated_add(bin_cursor, bin, h_kv, u < total);
    if (u < total)
      for (int g = 0; g < h_kv; ++g) {  // the kv heads of one unit stay adjacent (same query rows)
        out[2 * (pos + g)] = make_int4(i, g, na | (nb << 16), 0);
        out[2 * (pos + g) + 1] = w1;
      }
  }
  __syncthreads();
  if (tid == 0) {
    hdr->n_items = s_total;
    hdr->n_tiles = 0;
    hdr->n_gaps = n_gaps;
    hdr->status = ST_OK;
    hdr->sched = 0;
    hdr->n_questions = a.n;
    hdr->total_tokens = a.T;
    hdr->h_q = a.h_q;
    hdr->format = 1;
    if (a.dev_status) *a.dev_status = ST_OK;
  }
}

__global__ void __launch_bounds__(kThreads) segments_kernel(SegmentsArgs a) {
  __shared__ unsigned long long keys[kMaxQuestions];
  __shared__ int s_flags;  // bit 0 intervals, bit 1 slot range, bit 2 overflow, bit 3 duplicate slot, bit 4 prefix
  __shared__ int scan_tmp[kThreads / 32 + 1];
  __shared__ int bin_count[kCostBins];
  __shared__ int bin_cursor[kCostBins];
  __shared__ int s_ngaps;
  __shared__ int s_ntiles;
  __shared__ int2 s_iv[kSmall];  // small batches: intervals and slot ids in shared memory
  __shared__ int s_slot[kSmall];

  PrefillHeader* hdr = reinterpret_cast<PrefillHeader*>(a.ws);
  int32_t* cu = reinterpret_cast<int32_t*>(a.ws + a.layout.cu_seqlens);
  int2* tiles = reinterpret_cast<int2*>(a.ws + a.layout.tiles);
  int4* items = reinterpret_cast<int4*>(a.ws + a.layout.items);
  int2* gaps = reinterpret_cast<int2*>(a.ws + a.layout.gaps);

  pdl_wait();     // the intervals and slot ids may come from the kernel before this one
  pdl_trigger();  // the attention kernel after this one may be scheduled on the other SMs
  const int n = a.n;
  const int tid = threadIdx.x;
  if (tid == 0) s_flags = 0;
  if (tid < kCostBins) bin_count[tid] = 0;
  __syncthreads();

  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  const bool small = n <= kSmall;

  // 1. per-question range checks (and, for a small batch, a shared-memory copy of the inputs)
  for (int i = tid; i < n; i += blockDim.x) {
    const kev_interval iv = a.intervals[i];
    if (!(iv.begin >= 0 && iv.begin <= iv.end && iv.end <= a.T)) atomicOr(&s_flags, 1);
    int s = -1;
    // chunked prefill: the chunk sits after prefix_lens[i] cached positions (a tile boundary)
    const int pre = a.prefix_lens ? a.prefix_lens[i] : 0;
    if (pre < 0 || pre % kTileM != 0) atomicOr(&s_flags, 16);
    if (a.slot_ids) {
      s = a.slot_ids[i];
      if (s < 0 || s >= a.n_slots) atomicOr(&s_flags, 2);
      if ((int64_t)iv.end - iv.begin + pre > a.cap) atomicOr(&s_flags, 4);
    }
    if (small) {
      s_iv[i] = make_int2(iv.begin, iv.end);
      s_slot[i] = s;
    }
  }
  __syncthreads();

  if (small) {
    // 2-4 for a small batch.  Fast path, the usual layout: the intervals come in index order,
    // each ending at or before the next one begins -- no overlap, the ranks are the index order
    // of the non-empty ones, and a shared-memory hash finds a slot two non-empty questions share.
    const bool ranges_ok = (s_flags & 1) == 0;
    __shared__ int s_unordered;
    if (tid == 0) s_unordered = 0;
    __syncthreads();
    for (int i = tid; i + 1 < n; i += blockDim.x) {
      const int2 me = s_iv[i], nx = s_iv[i + 1];
      if (!(me.x <= nx.x && me.y <= nx.x)) s_unordered = 1;
    }
    __syncthreads();
    if (!s_unordered) {
      if (a.slot_ids) {
        int* hash = reinterpret_cast<int*>(keys);  // free until the ranks are written
        int hs = 1;
        while (hs < 2 * n) hs <<= 1;
        for (int j = tid; j < hs; j += blockDim.x) hash[j] = -1;
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x) {
          if (s_iv[i].y <= s_iv[i].x) continue;
          const int slot = s_slot[i];
          unsigned h = ((unsigned)slot * 2654435761u) & (unsigned)(hs - 1);
          for (int probe = 0; probe < hs; ++probe) {
            const int prev = atomicCAS(&hash[h], -1, slot);
            if (prev == -1) break;
            if (prev == slot) {
              atomicOr(&s_flags, 8);
              break;
            }
            h = (h + 1) & (unsigned)(hs - 1);
          }
        }
        __syncthreads();
      }
      if (ranges_ok) {
        int running = 0;
        for (int base = 0; base < n; base += blockDim.x) {
          const int i = base + tid;
          const bool ne = i < n && s_iv[i].y > s_iv[i].x;
          int blk;
          const int off = block_exclusive_scan(ne ? 1 : 0, scan_tmp, &blk);
          if (ne) keys[running + off] = ((unsigned long long)(unsigned)s_iv[i].x << 32) | (unsigned)s_iv[i].y;
          running += blk;
        }
        for (int i = running + tid; i < n2; i += blockDim.x) keys[i] = ~0ull;
        __syncthreads();
      }
    } else {
      // every non-empty interval against every other one (overlap, and a slot shared by two
      // non-empty questions), and its rank by (begin, index) places it in `keys`, begin-sorted;
      // empty intervals sort last
      const bool has_slots = a.slot_ids != nullptr;
      for (int i = tid; i < n; i += blockDim.x) {
        const int2 me = s_iv[i];
        if (me.y <= me.x) continue;
        const int my_slot = s_slot[i];
        int rank = 0;
        bool overlap = false, dup = false;
        // branch-free and unrolled: the shared-memory loads of several j are in flight at once
#pragma unroll 8
        for (int j = 0; j < n; ++j) {
          const int2 o = s_iv[j];
          const int so = s_slot[j];
          const bool other = j != i && o.y > o.x;
          overlap |= other & (me.x < o.y) & (o.x < me.y);
          dup |= other & has_slots & (so == my_slot);
          rank += other & ((o.x < me.x) | ((o.x == me.x) & (j < i)));
        }
        if (overlap) atomicOr(&s_flags, 1);
        if (dup) atomicOr(&s_flags, 8);
        if (ranges_ok) keys[rank] = ((unsigned long long)(unsigned)me.x << 32) | (unsigned)me.y;
      }
      __syncthreads();
      // the ranks of the non-empty intervals fill keys[0, n_ne); the rest marks the end
      if (ranges_ok) {
        int ne = 0;
        for (int i = tid; i < n; i += blockDim.x) ne += s_iv[i].y > s_iv[i].x;
        int n_ne;
        block_exclusive_scan(ne, scan_tmp, &n_ne);
        for (int i = n_ne + tid; i < n2; i += blockDim.x) keys[i] = ~0ull;
        __syncthreads();
      }
    }
  } else {
    // 2. overlap: sort non-empty intervals by begin, neighbours must not intersect
    if ((s_flags & 1) == 0 && n > 1) {
      for (int i = tid; i < n2; i += blockDim.x) {
        unsigned long long kk = ~0ull;
        if (i < n) {
          const kev_interval iv = a.intervals[i];
          if (iv.end > iv.begin) kk = ((unsigned long long)(unsigned)iv.begin << 32) | (unsigned)iv.end;
        }
        keys[i] = kk;
      }
      __syncthreads();
      bitonic_sort(keys, n2);
      for (int i = tid + 1; i < n; i += blockDim.x) {
        const unsigned long long cur = keys[i], prev = keys[i - 1];
        if (cur != ~0ull && prev != ~0ull) {
          if ((unsigned)(cur >> 32) < (unsigned)(prev & 0xffffffffu)) atomicOr(&s_flags, 1);
        }
      }
      __syncthreads();
    } else {
      for (int i = tid; i < n2; i += blockDim.x) {
        unsigned long long kk = ~0ull;
        if (i < n) {
          const kev_interval iv = a.intervals[i];
          if (iv.end > iv.begin) kk = ((unsigned long long)(unsigned)iv.begin << 32) | (unsigned)iv.end;
        }
        keys[i] = kk;
      }
      __syncthreads();
    }
  }

  // 3. gaps: tokens in no interval, from the begin-sorted intervals; gap k lies before the
  //    k-th non-empty interval (k = n_ne: after the last one), placed with a scan
  if ((s_flags & 1) == 0) {
    int ng_total = 0;
    for (int base = 0; base <= n; base += blockDim.x) {
      const int k = base + tid;
      int g0 = 0, g1 = 0;
      bool has = false;
      if (k <= n && (k == 0 || keys[k - 1] != ~0ull)) {  // k ranges over [0, n_ne]
        const bool at_end = k == n || keys[k] == ~0ull;
        g0 = k == 0 ? 0 : (int)(keys[k - 1] & 0xffffffffu);
        g1 = at_end ? a.T : (int)(keys[k] >> 32);
        has = g1 > g0;
      }
      int blk_total;
      const int off = block_exclusive_scan(has ? 1 : 0, scan_tmp, &blk_total);
      if (has) gaps[ng_total + off] = make_int2(g0, g1);
      ng_total += blk_total;
    }
    if (tid == 0) s_ngaps = ng_total;
  }
  __syncthreads();

  // 4. duplicate slots among non-empty questions (small batches did it in the pair pass)
  if (!small && a.slot_ids && s_flags == 0 && n > 1) {
    for (int i = tid; i < n2; i += blockDim.x) {
      unsigned long long kk = ~0ull;
      if (i < n) {
        const kev_interval iv = a.intervals[i];
        if (iv.end > iv.begin) kk = (unsigned long long)(unsigned)a.slot_ids[i];
      }
      keys[i] = kk;
    }
    __syncthreads();
    bitonic_sort(keys, n2);
    for (int i = tid + 1; i < n; i += blockDim.x) {
      if (keys[i] != ~0ull && keys[i] == keys[i - 1]) atomicOr(&s_flags, 8);
    }
    __syncthreads();
  }

  const int f = s_flags;
  const int code = (f & 1)    ? ST_INTERVALS
                   : (f & 2)  ? ST_SLOT
                   : (f & 16) ? ST_PREFIX
                   : (f & 4)  ? ST_OVERFLOW
                   : (f & 8)  ? ST_SLOT
                              : ST_OK;
  if (code != ST_OK) {
    if (tid == 0) {
      hdr->status = code;
      hdr->n_items = 0;
      hdr->n_tiles = 0;
      hdr->n_gaps = 0;
      hdr->sched = 0;
      hdr->n_questions = n;
      hdr->total_tokens = a.T;
      hdr->h_q = a.h_q;
      hdr->format = a.units2;
      if (a.dev_status) *a.dev_status = code;
    }
    return;
  }

  // 5. cu_seqlens (lengths in interval order) and per-question tile counts
  int total_len = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const int L = i < n ? a.intervals[i].end - a.intervals[i].begin : 0;
    int blk_total;
    const int off = block_exclusive_scan(L, scan_tmp, &blk_total);
    if (i < n) cu[i] = total_len + off;
    total_len += blk_total;
  }
  if (tid == 0) cu[n] = total_len;

  if (a.units2) {  // the CTA-pair kernel's units instead of tiles and items
    emit_units(a, hdr, items, bin_count, bin_cursor, s_ngaps, reinterpret_cast<int*>(keys), scan_tmp);
    return;
  }

  // 6. tile histogram over cost bins, then longest-first placement
  // a tile's cost is its number of key tiles: m + 1, plus the cached prefix's tiles
  for (int i = tid; i < n; i += blockDim.x) {
    const int L = a.intervals[i].end - a.intervals[i].begin;
    const int nt = (L + kTileM - 1) / kTileM;
    const int pt = a.prefix_lens ? a.prefix_lens[i] / kTileM : 0;
    for (int m = 0; m < nt; ++m) atomicAdd(&bin_count[min(m + pt, kCostBins - 1)], 1);
  }
  __syncthreads();
  static_assert(kCostBins == 64, "one warp places the 64 bins, two per lane");
  if (tid < 32) {  // bins in descending order: bin b starts after every bin above it
    const int hi = kCostBins - 1 - 2 * tid, lo = hi - 1;
    const int c_hi = bin_count[hi], c_lo = bin_count[lo];
    int x = c_hi + c_lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
    }
    const int base = x - (c_hi + c_lo);
    bin_cursor[hi] = base;
    bin_cursor[lo] = base + c_hi;
    if (tid == 31) {
      hdr->n_tiles = x;
      s_ntiles = x;
    }
  }
  __syncthreads();
  // the tile list stays in shared memory (the sort keys are dead) when it fits
  const int n_tiles = s_ntiles;
  int2* tl_list = n_tiles <= kMaxQuestions ? reinterpret_cast<int2*>(keys) : tiles;
  for (int i = tid; i < n; i += blockDim.x) {
    const int L = a.intervals[i].end - a.intervals[i].begin;
    const int nt = (L + kTileM - 1) / kTileM;
    const int pt = a.prefix_lens ? a.prefix_lens[i] / kTileM : 0;
    for (int m = nt - 1; m >= 0; --m) {
      const int pos = atomicAdd(&bin_cursor[min(m + pt, kCostBins - 1)], 1);
      tl_list[pos] = make_int2(i, m);
    }
  }
  __syncthreads();

  // 7. expand tiles into (tile, head block) items: a block is heads_per_item consecutive
  //    q-heads of one kv group (they share every K/V tile); the blocks of one tile stay
  //    adjacent so the q-heads that share a kv-head run close together (L2 reuse).  When the
  //    group leaves a single q-head over (odd group, two heads per item), that head's query
  //    tiles m-1 and m of a question form one item instead (m odd; bit 30 of the last word,
  //    `rows` = rows of tile m): the two tiles share the K/V tiles of tile m-1.  A question's
  //    last tile of an odd count keeps a single-head item.
  const int per_group = (a.group + a.heads_per_item - 1) / a.heads_per_item;
  const int h_kv = a.h_q / a.group;
  const bool odd_single = a.heads_per_item == 2 && (a.group & 1);
  // items of the tile at longest-first position `pos`
  auto tile_items = [&](int pos, int2& tl, int& nt) {
    tl = tl_list[pos];
    const kev_interval iv = a.intervals[tl.x];
    nt = (iv.end - iv.begin + kTileM - 1) / kTileM;
    int cnt = h_kv * per_group;
    if (odd_single && (tl.y & 1) == 0 && tl.y + 1 < nt) cnt -= h_kv;  // covered by the pair at m+1
    return cnt;
  };
  long long running = 0;
  for (int base = 0; base < n_tiles; base += blockDim.x) {
    const int pos = base + tid;
    int2 tl = make_int2(0, 0);
    int nt = 0;
    const int cnt = pos < n_tiles ? tile_items(pos, tl, nt) : 0;
    int blk_total;
    const int off = block_exclusive_scan(cnt, scan_tmp, &blk_total);
    if (pos < n_tiles) {
      const kev_interval iv = a.intervals[tl.x];
      const int r0 = iv.begin + tl.y * kTileM;
      const int rows = min(kTileM, iv.end - r0);
      long long k = running + off;
      for (int g = 0; g < h_kv; ++g)
        for (int b = 0; b < per_group; ++b) {
          const int h0 = g * a.group + b * a.heads_per_item;
          const int nh = min(a.heads_per_item, a.group - b * a.heads_per_item);
          if (odd_single && nh == 1 && tl.y + 1 < nt && (tl.y & 1) == 0) continue;
          if (odd_single && nh == 1 && (tl.y & 1) == 1)
            items[k++] = make_int4(tl.x, r0 - kTileM, rows, h0 | (1 << 16) | (1 << 30));  // tiles m-1, m
          else
            items[k++] = make_int4(tl.x, r0, rows, h0 | (nh << 16));
        }
    }
    running += blk_total;
  }
  if (tid == 0) hdr->n_items = (int)running;
  if (tid == 0) {
    hdr->status = ST_OK;
    hdr->n_gaps = s_ngaps;
    hdr->sched = 0;
    hdr->n_questions = n;
    hdr->total_tokens = a.T;
    hdr->h_q = a.h_q;
    hdr->format = 0;
    if (a.dev_status) *a.dev_status = ST_OK;
  }
}

}  // namespace

cudaError_t launch_segments(const SegmentsArgs& a, cudaStream_t s) {
  return launch_pdl(segments_kernel, dim3(1), dim3(kThreads), 0, s, a);
}

}  // namespace kev
