// KV slot write and zero rows of tokens that belong to no question.
//
// Slot pool of the Kev pipeline article (gsyq.cn news 368355, §2.2): a preallocated pool
// cut into fixed-size slots, one per question.  Question i's rows are copied bit for bit:
//   pool_{k,v}[slot_i, g, j, :] = {k,v}[begin_i + j, g, :]    for j < L_i.
// Positions >= L_i and slots no question uses are not touched.  With a paged pool (block
// table, inference-engine notes §2.5) position j of question i goes to block
// block_table[i][j / 128], row j % 128 (n_slots then counts blocks).
//
// Tokens outside every interval (boundary / padding tokens between questions) are keys for
// nobody (the article's §4.1 PAD-leak fix) and their own output rows are written as 0.
//
// Work unit of the slot write: one (row, kv head) of K and of V, row_bytes each, in
// cu_seqlens order (consecutive units are consecutive in the packed K/V).  A warp copies
// 32 / (row_bytes / 16) units per pass with one 16-byte vector per lane, kUnroll passes with
// all their loads in flight before the stores.  Each block keeps cu_seqlens, the interval
// starts and the slot ids in shared memory, so a unit's question is a binary search there.
//
// After the attention kernel, this kernel overlaps the attention's tail: it reads nothing the
// attention writes and writes nothing the attention reads (the pools; output rows of gap
// tokens, which no query tile covers), so it waits for the attention grid only at its end,
// which keeps the completion order of the stream (this grid completes after the attention).
// The segment builder's results it reads are complete by then: the attention kernel lets it
// launch only after every attention CTA has waited for the builder.
#include "kev_internal.cuh"

namespace kev {
namespace {

constexpr int kAuxThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ int question_of(const int32_t* cu, int n, int r) {
  int lo = 0, hi = n;  // cu[lo] <= r < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kAuxThreads) aux_kernel(AuxArgs a) {
  extern __shared__ int32_t s_cu[];             // [n + 1]
  int2* s_bs = reinterpret_cast<int2*>(s_cu + ((a.n + 2) & ~1));  // [n] {begin, slot}
  __shared__ int s_ok;
  if (!a.after_attention) pdl_wait();  // the segment builder's results are complete
  pdl_trigger();
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(a.ws);
  const int32_t* cu = reinterpret_cast<const int32_t*>(a.ws + a.layout.cu_seqlens);
  if (threadIdx.x == 0) s_ok = hdr->status == ST_OK;
  const bool paged = a.block_table != nullptr;
  const bool to_pool = a.slot_ids != nullptr || paged;
  if (to_pool) {
    for (int i = threadIdx.x; i <= a.n; i += blockDim.x) s_cu[i] = cu[i];
    for (int i = threadIdx.x; i < a.n; i += blockDim.x)
      s_bs[i] = make_int2(a.intervals[i].begin, paged ? i : a.slot_ids[i]);
  }
  __syncthreads();

  if (s_ok && to_pool) {
    // A unit is up to 32 16-byte vectors of one (row, kv head): a row of vpr vectors is `parts`
    // units; a warp pass copies upp units of lpu lanes each (the other lanes idle).
    const int vpr = a.row_bytes / 16;
    const int lpu = vpr < 32 ? vpr : 32;
    const int upp = 32 / lpu;
    const int parts = (vpr + 31) / 32;
    const int lane = threadIdx.x & 31, sub = lane / lpu, v_in = lane % lpu;
    const int64_t units = (int64_t)s_cu[a.n] * a.h_kv * parts;
    const int64_t per_chunk = (int64_t)upp * kUnroll;
    const int64_t n_chunks = (units + per_chunk - 1) / per_chunk;
    const int warps = gridDim.x * (kAuxThreads / 32);
    const int4* k = reinterpret_cast<const int4*>(a.k);
    const int4* vv = reinterpret_cast<const int4*>(a.v);
    int4* pk = reinterpret_cast<int4*>(a.pool_k);
    int4* pv = reinterpret_cast<int4*>(a.pool_v);
    for (int64_t c = blockIdx.x * (kAuxThreads / 32) + (threadIdx.x >> 5); c < n_chunks; c += warps) {
      int4 bk[kUnroll], bv[kUnroll];
      int64_t dst[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int64_t u = c * per_chunk + t * upp + sub;
        dst[t] = -1;
        const int v = (int)(u % parts) * 32 + v_in;
        if (sub < upp && u < units && v < vpr) {
          const int64_t rg = u / parts;
          const int r = (int)(rg / a.h_kv), g = (int)(rg % a.h_kv);
          const int i = question_of(s_cu, a.n, r);
          const int j = r - s_cu[i];
          if (a.tails_only && j < ((s_cu[i + 1] - s_cu[i]) & ~127)) continue;  // stored by the attention kernel
          const int2 bs = s_bs[i];
          const int64_t src = ((int64_t)(bs.x + j) * a.h_kv + g) * vpr + v;
          if (paged) {  // block of position j (the tables were checked before the attention)
            if (j / kPage >= a.max_blocks) continue;
            const int blk = a.block_table[(int64_t)bs.y * a.max_blocks + j / kPage];
            if (blk < 0 || blk >= a.n_slots) continue;
            dst[t] = (((int64_t)blk * a.h_kv + g) * kPage + j % kPage) * vpr + v;
          } else {
            const int pos = j + (a.prefix_lens ? a.prefix_lens[i] : 0);  // chunked prefill: after the prefix
            if (bs.y < 0 || bs.y >= a.n_slots || pos >= a.cap) continue;  // a work list built for other slots
            dst[t] = (((int64_t)bs.y * a.h_kv + g) * a.cap + pos) * vpr + v;
          }
          bk[t] = __ldg(k + src);
          bv[t] = __ldg(vv + src);
        }
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        if (dst[t] >= 0) {
          pk[dst[t]] = bk[t];
          pv[dst[t]] = bv[t];
        }
      }
    }
  }
  if (s_ok && a.prefix_lens && a.slot_ids) {
    // chunked prefill: slot rows from the chunk's end up to the next multiple of 128 become zero
    // (no position lives there yet, but the attention's last key tile of the chunk reads them)
    const int vpr = a.row_bytes / 16;
    for (int i = blockIdx.x; i < a.n; i += gridDim.x) {
      const int L = s_cu[i + 1] - s_cu[i];
      const int slot = s_bs[i].y;
      if (L == 0 || slot < 0 || slot >= a.n_slots) continue;
      const int p0 = a.prefix_lens[i] + L;
      const int p1 = min(a.cap, (p0 + 127) / 128 * 128);
      const int per_head = (p1 - p0) * vpr;
      for (int w = threadIdx.x; w < per_head * a.h_kv; w += blockDim.x) {
        const int g = w / per_head, r = w % per_head;
        const int64_t dst = (((int64_t)slot * a.h_kv + g) * a.cap + p0) * vpr + r;
        reinterpret_cast<int4*>(a.pool_k)[dst] = make_int4(0, 0, 0, 0);
        reinterpret_cast<int4*>(a.pool_v)[dst] = make_int4(0, 0, 0, 0);
      }
    }
  }
  if (s_ok && a.out) {
    const int2* gaps = reinterpret_cast<const int2*>(a.ws + a.layout.gaps);
    const int ng = hdr->n_gaps;
    const int64_t out_vec_row = (int64_t)a.h_q * (a.row_bytes / 16);  // output row: H_q * d elements
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int gi = 0; gi < ng; ++gi) {
      const int2 gp = gaps[gi];
      const int64_t base = (int64_t)gp.x * out_vec_row;
      const int64_t cnt = (int64_t)(gp.y - gp.x) * out_vec_row;
      for (int64_t w = tid0; w < cnt; w += stride) reinterpret_cast<int4*>(a.out)[base + w] = make_int4(0, 0, 0, 0);
    }
  }
  if (a.after_attention) pdl_wait();  // this grid completes after the attention grid
}

}  // namespace

cudaError_t launch_aux(const AuxArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = a.slot_ids || a.block_table
                          ? sizeof(int32_t) * (size_t)((a.n + 2) & ~1) + sizeof(int2) * (size_t)a.n
                          : 0;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(aux_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(aux_kernel, dim3(num_sms * 4), dim3(kAuxThreads), smem, s, a);
}

}  // namespace kev
