// Pieces shared by the two decode kernels (CUDA-core and tensor-core): validation of the live
// questions, the compacted list of work chunks, and the static split of that list into one
// contiguous range per CTA.
//
// Early stop (Kev pipeline article, gsyq.cn news 368355, §1.2, §2.3): a question with
// active[i] == 0 contributes no chunk, so its slot is neither read nor written.
#pragma once

#include "kev_internal.cuh"

namespace kev {
namespace dec {

constexpr int kChunk = kDecodeChunk;  // positions per work chunk

template <int NT>
__device__ int block_exclusive_scan(int v, int* tmp, int* total) {
  constexpr int nw = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < nw; ++w) {
    if (w < warp) base += tmp[w];
    tot += tmp[w];
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

struct ItemInfo {
  int i, g, hb, c, len, slot, nch, p0, p1, h0, nh;
};

// Chunk `x` of the compacted list: item_base is the prefix over questions of
// H_kv * n_hblocks * n_chunks (dropped questions: 0), meta holds {len, slot} per question.
template <int HB>
__device__ __forceinline__ ItemInfo decode_item(const DecodeArgs& a, const int* item_base, const int2* meta, int x,
                                                int n_hblocks) {
  int lo = 0, hi = a.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (item_base[mid] <= x) lo = mid; else hi = mid;
  }
  ItemInfo f;
  f.i = lo;
  const int2 m = meta[lo];
  f.len = m.x;
  f.slot = m.y;
  f.nch = (f.len + 1 + kChunk - 1) / kChunk;
  const int r = x - item_base[lo];
  f.c = r % f.nch;
  const int gh = r / f.nch;
  f.hb = gh % n_hblocks;
  f.g = gh / n_hblocks;
  f.p0 = f.c * kChunk;
  f.p1 = min(f.p0 + kChunk, f.len + 1);
  f.h0 = f.g * a.group + f.hb * HB;
  f.nh = min(HB, a.group - f.hb * HB);
  return f;
}

// Static split of the chunk space [0, total) into one contiguous range per CTA.
__device__ __forceinline__ int range_start(int b, int total, int nb) { return (int)((int64_t)b * total / nb); }
__device__ __forceinline__ int range_owner(int x, int total, int nb) {
  return (int)((((int64_t)x + 1) * nb - 1) / total);
}

// Every CTA runs this over the N questions: {len, slot} into `meta`, validation of the live
// questions (slot range, room for the new row, no slot shared by two live questions; a
// shared-memory hash finds duplicates), and the prefix sum of their chunks into
// `item_base`.  `hash` (int[2 * kMaxQuestions]) may alias memory the caller uses later.
// Returns the number of chunks, or -1 when the call is invalid (block 0 stores the status, and
// also the validation code into *code_out when that is not null).
template <int NT>
__device__ int prologue(const DecodeArgs& a, int n_hblocks, int* item_base, int2* meta, int* hash, int* flags,
                        int* scan_tmp, int* code_out = nullptr) {
  const int tid = threadIdx.x;
  const int n = a.n;
  const bool paged = a.block_table != nullptr;
  int hs = 1;
  // contiguous pool: a hash of the live slots; paged pool: of the blocks live questions use
  // (n * max_blocks <= kMaxPagedEntries, checked on the host, so the caller's area holds it)
  while (hs < 2 * (paged ? n * a.max_blocks : n)) hs <<= 1;
  if (tid == 0) *flags = 0;
  for (int j = tid; j < hs; j += NT) hash[j] = -1;
  __syncthreads();
  if (paged) {
    // every live question needs a block for each page of positions 0..len (the new row
    // included): a row too short is SLOT_OVERFLOW, an entry out of range or used twice SLOT
    for (int i = tid; i < n; i += NT) {
      const int len = a.lens[i];
      meta[i] = make_int2(len, i);
      if (a.active[i] && (len < 0 || len / kChunk >= a.max_blocks)) atomicOr(flags, 2);
    }
    const int64_t entries = (int64_t)n * a.max_blocks;
    for (int64_t e = tid; e < entries; e += NT) {
      const int i = (int)(e / a.max_blocks), b = (int)(e % a.max_blocks);
      if (!a.active[i]) continue;
      const int len = a.lens[i];
      if (len < 0 || b > len / kChunk) continue;
      const int blk = a.block_table[e];
      if (blk < 0 || blk >= a.n_blocks) {
        atomicOr(flags, 1);
        continue;
      }
      unsigned h = ((unsigned)blk * 2654435761u) & (unsigned)(hs - 1);
      for (int probe = 0; probe < hs; ++probe) {
        const int prev = atomicCAS(&hash[h], -1, blk);
        if (prev == -1) break;
        if (prev == blk) {
          atomicOr(flags, 4);
          break;
        }
        h = (h + 1) & (unsigned)(hs - 1);
      }
    }
  }
  for (int i = tid; i < n && !paged; i += NT) {
    const int live = a.active[i];
    const int slot = a.slot_ids[i];
    const int len = a.lens[i];
    meta[i] = make_int2(len, slot);
    if (!live) continue;
    if (slot < 0 || slot >= a.n_slots) {
      atomicOr(flags, 1);
      continue;
    }
    if (len < 0 || len >= a.cap) atomicOr(flags, 2);
    unsigned h = ((unsigned)slot * 2654435761u) & (unsigned)(hs - 1);
    for (int probe = 0; probe < hs; ++probe) {
      const int prev = atomicCAS(&hash[h], -1, slot);
      if (prev == -1) break;
      if (prev == slot) {
        atomicOr(flags, 4);
        break;
      }
      h = (h + 1) & (unsigned)(hs - 1);
    }
  }
  __syncthreads();
  const int f = *flags;
  const int code = paged ? ((f & 2) ? ST_OVERFLOW : (f & 5) ? ST_SLOT : ST_OK)
                         : ((f & 1) ? ST_SLOT : (f & 2) ? ST_OVERFLOW : (f & 4) ? ST_SLOT : ST_OK);
  if (blockIdx.x == 0 && tid == 0) {
    if (a.dev_status) *a.dev_status = code;
    if (code_out) *code_out = code;
  }
  if (code != ST_OK) return -1;

  int running = 0;
  for (int base = 0; base < n; base += NT) {
    const int i = base + tid;
    int cnt = 0;
    if (i < n && a.active[i]) cnt = a.h_kv * n_hblocks * ((meta[i].x + 1 + kChunk - 1) / kChunk);
    int tot;
    const int off = block_exclusive_scan<NT>(cnt, scan_tmp, &tot);
    if (i < n) item_base[i] = running + off;
    running += tot;
  }
  if (tid == 0) item_base[n] = running;
  __syncthreads();
  return running;
}

}  // namespace dec
}  // namespace kev
