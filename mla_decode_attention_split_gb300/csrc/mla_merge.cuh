// Merge of split tokens inside stage 1, and the zero output of empty
// segments: the pages' stage 2 (kernelbot-amd-mixed-mla-753817,
// `mla_flash_decode_stage2`: L = max_s lse_s, w_s = 2^(lse_s - L),
// out = sum_s w_s O_s / sum_s w_s, LSEs in the log2 domain) done by the
// stage-1 CTA that completes a token's count of partials, so no second kernel
// runs. Format-independent parts, shared by all stage-1 kernels.
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

// The merge of one token from global memory by kThreads threads: thread t
// keeps a running-max merge of float4 elements t, t + kThreads, ... of the
// 16 x 512 output; partial slots G c + token, c = c0..c1, two per round trip.
// Partials come from L2 (other SMs wrote them), not L1.
template <int kThreads>
__device__ void merge_token_global(const Stage1Params& p, int token, int64_t c0, int64_t c1) {
  constexpr int kF = (kHeads * kDv / 4 + kThreads - 1) / kThreads;
  float acc[kF][4], mrun[kF], wsum[kF];
#pragma unroll
  for (int i = 0; i < kF; ++i) {
    mrun[i] = -INFINITY;
    wsum[i] = 0.f;
    acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  }
  for (int64_t c = c0; c <= c1; c += 2) {
    const bool two = c + 1 <= c1;
    const int64_t s0 = p.group * c + token, s1 = two ? s0 + p.group : s0;
    const float4* o0 = reinterpret_cast<const float4*>(p.part_o + s0 * kHeads * kDv);
    const float4* o1 = reinterpret_cast<const float4*>(p.part_o + s1 * kHeads * kDv);
    float4 v0[kF], v1[kF];
    float l0[kF], l1[kF];
#pragma unroll
    for (int i = 0; i < kF; ++i) {
      const int f = threadIdx.x + i * kThreads;
      if (f < kHeads * kDv / 4) {
        v0[i] = __ldcg(o0 + f);
        v1[i] = __ldcg(o1 + f);
        l0[i] = __ldcg(p.part_lse + s0 * kHeads + (f >> 7));
        l1[i] = two ? __ldcg(p.part_lse + s1 * kHeads + (f >> 7)) : -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < kF; ++i) {
      const int f = threadIdx.x + i * kThreads;
      if (f < kHeads * kDv / 4) {
        const float mn = fmaxf(mrun[i], fmaxf(l0[i], l1[i]));
        const float sc = fast_exp2(mrun[i] - mn), w0 = fast_exp2(l0[i] - mn), w1 = fast_exp2(l1[i] - mn);
        acc[i][0] = acc[i][0] * sc + w0 * v0[i].x + w1 * v1[i].x;
        acc[i][1] = acc[i][1] * sc + w0 * v0[i].y + w1 * v1[i].y;
        acc[i][2] = acc[i][2] * sc + w0 * v0[i].z + w1 * v1[i].z;
        acc[i][3] = acc[i][3] * sc + w0 * v0[i].w + w1 * v1[i].w;
        wsum[i] = wsum[i] * sc + w0 + w1;
        mrun[i] = mn;
      }
    }
  }
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(token) * kHeads * kDv;
#pragma unroll
  for (int i = 0; i < kF; ++i) {
    const int f = threadIdx.x + i * kThreads;
    if (f < kHeads * kDv / 4) {
      const float inv = 1.0f / wsum[i];
      *reinterpret_cast<uint2*>(dst + 4 * f) =
          make_uint2(pack_bf16x2(acc[i][0] * inv, acc[i][1] * inv), pack_bf16x2(acc[i][2] * inv, acc[i][3] * inv));
    }
  }
}

// End of a CTA that wrote all its partials: publish them (every thread
// fences, then a block barrier), count each split piece on its token's
// counter, and merge the tokens whose count this CTA completed (at most the
// CTA's first and last piece are split). `scratch` is 16 x i64 of shared
// memory. All kThreads threads call this.
template <int kThreads>
__device__ void merge_split_tokens_at_end(const Stage1Params& p, PieceCursor cur, int64_t total, int64_t* scratch) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t P = p.num_splits;
    int64_t n = 0;
    Piece pc;
    while (cur.next(pc)) {
      if (pc.direct) continue;
      const int64_t c0 = part_of_row(pc.tok_vs, total, P), c1 = part_of_row(pc.tok_vs + pc.kvlen - 1, total, P);
      const uint32_t arrived = atomicAdd(p.tok_cnt + pc.token, 1u) + 1u;
      if (arrived == static_cast<uint32_t>(c1 - c0 + 1) && n < 4) {
        scratch[1 + 3 * n] = pc.token;
        scratch[2 + 3 * n] = c0;
        scratch[3 + 3 * n] = c1;
        ++n;
      }
    }
    scratch[0] = n;
    __threadfence();
  }
  __syncthreads();
  const int64_t n = scratch[0];
  for (int64_t e = 0; e < n; ++e) {
    const int token = static_cast<int>(scratch[1 + 3 * e]);
    merge_token_global<kThreads>(p, token, scratch[2 + 3 * e], scratch[3 + 3 * e]);
    if (threadIdx.x == 0) p.tok_cnt[token] = 0u;
  }
}

}  // namespace mla
