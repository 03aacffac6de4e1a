// Per-tensor fp8 quantisation scale of bf16 queries, computed on the device
// for the in-call a8w8 mode: s = max(amax |q|, 1e-12) / 448 in fp32, the rule
// of kernelbot-amd-mixed-mla-753817 `_quantize_fp8` (there evaluated in the
// tensor's dtype; here in fp32). Stage 1 then quantises q with s as it loads it.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

constexpr int kAmaxThreads = 256;

// Every block folds its maximum |q| (as bf16 magnitude bits) into header word
// kHdrQAmax; the last block to finish writes the scale and clears its own
// scratch words, so the header is ready for the next call.
__global__ void __launch_bounds__(kAmaxThreads) mla_q_amax_kernel(const uint4* __restrict__ q, int64_t n16,
                                                                   uint32_t* hdr) {
  __shared__ uint32_t wmax[kAmaxThreads / 32];
  __shared__ bool last;
  griddep_launch_dependents();  // stage 1 may start; it waits for this grid before reading the scale
  uint32_t m = 0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kAmaxThreads) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * kAmaxThreads) {
    const uint4 v = __ldg(q + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAmaxThreads / 32; ++w) m = max(m, wmax[w]);
    atomicMax(hdr + kHdrQAmax, m << 16);  // positive f32 bits order like integers
    __threadfence();
    last = atomicAdd(hdr + kHdrQBlocks, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    const float amax = __uint_as_float(atomicOr(hdr + kHdrQAmax, 0u));
    hdr[kHdrQScale] = __float_as_uint(fmaxf(amax, 1e-12f) / 448.0f);
    hdr[kHdrQAmax] = 0u;
    hdr[kHdrQBlocks] = 0u;
  }
}

cudaError_t launch_q_scale(const void* q, int64_t n, uint32_t* header, cudaStream_t stream) {
  const int64_t n16 = n / 8;  // 8 bf16 per 16 bytes; n = total_q x 16 x 576 is a multiple of 8
  // one 16-byte load per thread up to 8 blocks per SM of a 152-SM part, so the
  // loads are in flight together rather than one after another per thread
  int64_t blocks = (n16 + kAmaxThreads - 1) / kAmaxThreads;
  blocks = blocks < 1 ? 1 : (blocks > 1216 ? 1216 : blocks);
  mla_q_amax_kernel<<<static_cast<int>(blocks), kAmaxThreads, 0, stream>>>(static_cast<const uint4*>(q), n16, header);
  return cudaGetLastError();
}

}  // namespace mla
