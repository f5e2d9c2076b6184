// KV slot write and zero rows of tokens that belong to no question.
//
// Slot pool of the Kev pipeline article (gsyq.cn news 368355, §2.2): a preallocated pool
// cut into fixed-size slots, one per question.  Question i's rows are copied bit for bit:
//   pool_{k,v}[slot_i, g, j, :] = {k,v}[begin_i + j, g, :]    for j < L_i.
// Positions >= L_i and slots no question uses are not touched.
//
// Tokens outside every interval (boundary / padding tokens between questions) are keys for
// nobody (the article's §4.1 PAD-leak fix) and their own output rows are written as 0.
//
// Grid-stride over 16-byte vectors; the item space is (question, kv head, row) for the
// slot write and (gap, row) for the zero fill, enumerated from the segment builder's
// cu_seqlens and gap list.
#include "kev_internal.cuh"

namespace kev {
namespace {

__global__ void __launch_bounds__(256) aux_kernel(AuxArgs a) {
  pdl_wait();  // the work list and status of the kernels before this one are complete
  pdl_trigger();
  const PrefillHeader* hdr = reinterpret_cast<const PrefillHeader*>(a.ws);
  if (hdr->status != ST_OK) return;
  const int32_t* cu = reinterpret_cast<const int32_t*>(a.ws + a.layout.cu_seqlens);
  const int vec_per_row = a.row_bytes / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;

  if (a.slot_ids) {
    // rows of all questions, in cu_seqlens order: r in [0, cu[n]) -> (question, j)
    const int total = cu[a.n];
    const int64_t work = (int64_t)total * a.h_kv * vec_per_row;
    for (int64_t w = tid0; w < work; w += stride) {
      const int vec = (int)(w % vec_per_row);
      const int64_t rest = w / vec_per_row;
      const int g = (int)(rest % a.h_kv);
      const int r = (int)(rest / a.h_kv);
      // question owning packed-length position r (binary search in cu_seqlens)
      int lo = 0, hi = a.n;  // cu[lo] <= r < cu[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= r) lo = mid; else hi = mid;
      }
      const int j = r - cu[lo];
      const int tok = a.intervals[lo].begin + j;
      const int slot = a.slot_ids[lo];
      const int64_t src = ((int64_t)tok * a.h_kv + g) * vec_per_row + vec;
      const int64_t dst = (((int64_t)slot * a.h_kv + g) * a.cap + j) * vec_per_row + vec;
      reinterpret_cast<int4*>(a.pool_k)[dst] = __ldg(reinterpret_cast<const int4*>(a.k) + src);
      reinterpret_cast<int4*>(a.pool_v)[dst] = __ldg(reinterpret_cast<const int4*>(a.v) + src);
    }
  }
  if (a.out) {
    const int2* gaps = reinterpret_cast<const int2*>(a.ws + a.layout.gaps);
    const int ng = hdr->n_gaps;
    const int64_t out_vec_row = (int64_t)a.h_q * vec_per_row;  // output row: H_q * d elements
    for (int gi = 0; gi < ng; ++gi) {
      const int2 gp = gaps[gi];
      const int64_t base = (int64_t)gp.x * out_vec_row;
      const int64_t cnt = (int64_t)(gp.y - gp.x) * out_vec_row;
      for (int64_t w = tid0; w < cnt; w += stride) reinterpret_cast<int4*>(a.out)[base + w] = make_int4(0, 0, 0, 0);
    }
  }
}

}  // namespace

cudaError_t launch_aux(const AuxArgs& a, int num_sms, cudaStream_t s) {
  return launch_pdl(aux_kernel, dim3(num_sms * 4), dim3(256), 0, s, a);
}

}  // namespace kev
