// Stage 1 of split-K MLA decode: the dispatch to the tcgen05 kernels, one per
// KV format (fp8: mla_stage1_tc.cu, bf16: mla_stage1_bf.cu, mxfp4:
// mla_stage1_mx.cu; token groups: mla_stage1_pair.cu, mla_stage1_duo.cu,
// mla_stage1_quad.cu).
//
// The method is the split-K flash-decoding stage 1 of kernelbot-amd-mixed-mla
// -753817 (`mla_flash_decode_stage1`: 16 heads packed against the single KV
// head, K = all 576 dims, V = the first 512, online softmax in the exp2 domain
// with the sm_scale*log2(e) factor folded into the scores) and -586148
// (`_flash_splitk`).
#include "mla_internal.h"

namespace mla {

bool stage1_supported(int kv_fmt, int q_fmt) {
  if (q_fmt == kQBf16Quant) return kv_fmt == kKvFp8;  // the in-call a8w8 mode
  return (kv_fmt == kKvFp8 || kv_fmt == kKvBf16 || kv_fmt == kKvMxfp4) && (q_fmt == kQBf16 || q_fmt == kQFp8);
}

cudaError_t launch_stage1(int kv_fmt, int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (kv_fmt == kKvFp8) return launch_stage1_tc_fp8(q_fmt, p, stream);
  if (kv_fmt == kKvMxfp4) return launch_stage1_tc_mxfp4(q_fmt, p, stream);
  if (kv_fmt == kKvBf16) return launch_stage1_tc_bf16(q_fmt, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mla
