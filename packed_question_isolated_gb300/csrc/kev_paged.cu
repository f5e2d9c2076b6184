// Paged slot pool: validation of the block tables before a prefill writes anything.
//
// Inference-engine notes (sakurs2.com), §2.5: K/V are kept in fixed-size blocks allocated on
// demand, and a block table records where each block lies, so attention reads K/V through the
// table instead of from one contiguous reservation.  Here a block holds kPage = 128 positions of
// one question for every kv head: pool [n_blocks, H_kv, kPage, d], position p of question i in
// block block_table[i * max_blocks + p / kPage], row p % kPage.
//
// paged_check_kernel (one CTA) checks the tables the prefill will write through: every non-empty
// question has a block for each of its ceil(L_i / kPage) pages (else SLOT_OVERFLOW), every used
// entry is in [0, n_blocks), and no block is used twice -- by two questions or by one (else SLOT:
// two questions on one block is the shared-state bug of the KV-cache isolation article,
// hnwysp.cn, §2.3).  Used entries go into an open-addressing hash in shared memory.  An error
// goes into the prefill workspace's status word, so the attention and slot-write kernels after
// this one write nothing, and into the caller's status word.
#include "kev_internal.cuh"

namespace kev {
namespace {

static_assert(kPage == kDecodeChunk, "a block is one decode chunk of positions");

constexpr int kCheckThreads = 1024;

__global__ void __launch_bounds__(kCheckThreads) paged_check_kernel(PagedCheckArgs a, int hs) {
  extern __shared__ int hash[];
  __shared__ int s_flags;  // bit 0: entry out of range or used twice, bit 1: a table row too short
  pdl_wait();              // the segment builder's status and the tables are complete
  pdl_trigger();
  PrefillHeader* hdr = reinterpret_cast<PrefillHeader*>(a.ws);
  if (hdr->status != ST_OK) return;  // the intervals were already rejected
  if (threadIdx.x == 0) s_flags = 0;
  for (int j = threadIdx.x; j < hs; j += blockDim.x) hash[j] = -1;
  __syncthreads();
  const int64_t entries = (int64_t)a.n * a.max_blocks;
  for (int64_t e = threadIdx.x; e < entries; e += blockDim.x) {
    const int i = (int)(e / a.max_blocks), b = (int)(e % a.max_blocks);
    const kev_interval iv = a.intervals[i];
    const int need = (iv.end - iv.begin + kPage - 1) / kPage;  // the builder checked begin <= end
    if (b == 0 && need > a.max_blocks) atomicOr(&s_flags, 2);
    if (b >= need) continue;
    const int blk = a.block_table[e];
    if (blk < 0 || blk >= a.n_blocks) {
      atomicOr(&s_flags, 1);
      continue;
    }
    unsigned h = ((unsigned)blk * 2654435761u) & (unsigned)(hs - 1);
    for (int probe = 0; probe < hs; ++probe) {
      const int prev = atomicCAS(&hash[h], -1, blk);
      if (prev == -1) break;
      if (prev == blk) {
        atomicOr(&s_flags, 1);
        break;
      }
      h = (h + 1) & (unsigned)(hs - 1);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_flags) {
    const int code = (s_flags & 2) ? ST_OVERFLOW : ST_SLOT;
    atomicCAS(&hdr->status, ST_OK, code);
    set_status(a.dev_status, code);
  }
}

}  // namespace

cudaError_t launch_paged_check(const PagedCheckArgs& a, cudaStream_t s) {
  int hs = 1;
  while (hs < 2 * a.n * a.max_blocks) hs <<= 1;  // n * max_blocks <= kMaxPagedEntries (host-checked)
  const size_t smem = sizeof(int) * (size_t)hs;
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(paged_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(paged_check_kernel, dim3(1), dim3(kCheckThreads), smem, s, a, hs);
}

}  // namespace kev
