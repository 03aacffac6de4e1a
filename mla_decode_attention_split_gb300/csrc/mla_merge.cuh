// The zero output of tokens whose segment has no KV rows, shared by all
// stage-1 kernels (the merge of split tokens is in mla_tc_common.cuh).
#pragma once

#include "mla_device.cuh"
#include "mla_internal.h"
#include "mla_partition.cuh"

namespace mla {

// Output rows of tokens whose segment has no KV rows are zero. CTA c writes
// them for segments c, c + P, c + 2P, ... (every CTA runs this, with or
// without work of its own).
template <int kThreads>
__device__ __forceinline__ void zero_empty_tokens(const Stage1Params& p) {
  for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
    if (__ldg(p.kv_indptr + b + 1) != __ldg(p.kv_indptr + b)) continue;
    const int64_t q0 = __ldg(p.qo_indptr + b), q1 = __ldg(p.qo_indptr + b + 1);
    uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + q0 * kHeads * kDv);
    const int64_t n = (q1 - q0) * (kHeads * kDv / 8);  // 16-byte units
    for (int64_t i = threadIdx.x; i < n; i += kThreads) o[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace mla
