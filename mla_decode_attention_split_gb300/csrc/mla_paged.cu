// Paged KV cache: the logical KV row offsets of the segments, built on the
// device from the page table.
//
// The page-table form is the one kernelbot-amd-mixed-mla-753817 hands to the
// vendor decode (`kv_indices`, `kv_last_page_len`, `page_size`; there with one
// row per page): segment b owns page-table entries
// [page_indptr[b], page_indptr[b+1]); its KV row i lives in page
// page_indices[page_indptr[b] + i / page_size] at slot i % page_size. With
// n_b pages the segment has (n_b - 1) * page_size + last_page_len[b] rows;
// with page_size 1 it has n_b rows and last_page_len is not read (that page
// passes the segment lengths there).
//
// The offsets go into the workspace and stage 1 then partitions the logical
// rows exactly as it does for a contiguous cache.
#include "mla_internal.h"
#include "mla_partition.cuh"

namespace mla {

constexpr int kPrepThreads = 1024;

// One block. On any inconsistency (page_indptr not starting at 0 or not
// monotone, a last-page length outside [1, page_size], more than 2^31 - 1
// rows) offset 0 is written as -1, which stage 1's own indptr check rejects
// with the bad-indptr flag before it reads any KV row.
__global__ void __launch_bounds__(kPrepThreads) mla_paged_prepare_kernel(const int32_t* __restrict__ pip,
                                                                         const int32_t* __restrict__ last, int batch,
                                                                         int page_size, int32_t* __restrict__ kvp,
                                                                         uint32_t* flags) {
  __shared__ int64_t sh[kPrepThreads / 32 + 1];
  griddep_launch_dependents();  // stage 1 may start; it waits for this grid before reading the offsets
  const int tid = threadIdx.x;
  const int per = (batch + kPrepThreads - 1) / kPrepThreads;
  const int lo = min(tid * per, batch), hi = min(lo + per, batch);
  int valid = 1;
  int64_t local = 0;
  for (int b = lo; b < hi; ++b) {
    const int32_t n = __ldg(pip + b + 1) - __ldg(pip + b);
    valid &= n >= 0;
    if (n > 0) {
      if (page_size == 1) {
        local += n;
      } else {
        const int32_t l = __ldg(last + b);
        valid &= (l >= 1) & (l <= page_size);
        local += static_cast<int64_t>(n - 1) * page_size + l;
      }
    }
  }
  if (tid == 0) valid &= __ldg(pip) == 0;
  valid = __syncthreads_and(valid);
  int64_t total = 0;
  const int64_t excl = block_exclusive_scan_i64<kPrepThreads>(valid ? local : 0, sh, total);
  valid &= total <= 0x7FFFFFFF;
  if (valid) {
    int64_t run = excl;
    for (int b = lo; b < hi; ++b) {
      kvp[b] = static_cast<int32_t>(run);
      const int32_t n = __ldg(pip + b + 1) - __ldg(pip + b);
      if (n > 0) run += page_size == 1 ? n : static_cast<int64_t>(n - 1) * page_size + __ldg(last + b);
    }
    if (tid == 0) kvp[batch] = static_cast<int32_t>(total);
  }
  __syncthreads();
  if (tid == 0 && !valid) {
    kvp[0] = -1;
    atomicOr(flags, kFlagBadIndptr);
  }
}

cudaError_t launch_paged_prepare(const int32_t* page_indptr, const int32_t* last_page_len, int32_t batch,
                                 int32_t page_size, int32_t* kv_indptr_out, uint32_t* flags, cudaStream_t stream) {
  mla_paged_prepare_kernel<<<1, kPrepThreads, 0, stream>>>(page_indptr, last_page_len, batch, page_size,
                                                           kv_indptr_out, flags);
  return cudaGetLastError();
}

}  // namespace mla
