// The dequantisation check kernels. bf16 and fp8: KV rows go through stage
// 1's operand path (same byte layout, same MMA) against an identity operand.
// mxfp4: rows go through the mxfp4 stage-1 conversion (the same device code)
// to its rebased e5m2 operand bytes and row exponent. Either way the decode
// of the stored codes can be compared bit for bit.
#include "mla_device.cuh"
#include "mla_internal.h"
#include "mla_mx_convert.cuh"
#include "mla_partition.cuh"

namespace mla {

// ---------------------------------------------------------------------------
// Dequantisation check. One warp per 8 KV rows; lane (g, t) takes row g and
// the same bytes it would take as a score warp (see the stage-1 query
// fragment layout), then multiplies by an identity operand on the tensor core.
// C[h][n] = B[kappa][n] where kappa = h (+16 for the second half) selects a
// contraction index; kappa maps back to the KV dim through the permutation.
template <int KV>
__global__ void mla_dequant_kernel(const uint8_t* __restrict__ kv, int32_t total_kv, int32_t row0, int32_t nrows,
                                   float* __restrict__ out) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int base_row = row0 + 8 * blockIdx.x;
  const int my_row = base_row + g;
  const bool valid = (my_row < row0 + nrows) && (my_row < total_kv);
  if (KV == kKvFp8) {
    // identity halves: A[h][kappa] = 1.0 (e4m3 0x38) iff kappa == h + 16*half
    uint32_t id[2][4];
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int arow = g + ((r & 1) ? 8 : 0);
        const int kbase = 4 * t + ((r & 2) ? 16 : 0);
        uint32_t wv = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (kbase + i == arow + 16 * half) wv |= 0x38u << (8 * i);
        id[half][r] = wv;
      }
    const uint8_t* rowp = kv + static_cast<int64_t>(valid ? my_row : 0) * 576;
#pragma unroll
    for (int W = 0; W < 5; ++W) {
      uint4 kb[2];
      const int off = (W < 4) ? 128 * W + 32 * t : 512 + 16 * t;
      kb[0] = valid ? __ldg(reinterpret_cast<const uint4*>(rowp + off)) : make_uint4(0, 0, 0, 0);
      kb[1] = (valid && W < 4) ? __ldg(reinterpret_cast<const uint4*>(rowp + off + 16)) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < (W < 4 ? 4 : 2); ++k) {
        const uint32_t b0 = (k >> 1) ? (((2 * k) & 3) == 0 ? kb[1].x : kb[1].z) : (((2 * k) & 3) == 0 ? kb[0].x : kb[0].z);
        const uint32_t b1 = (k >> 1) ? (((2 * k) & 3) == 0 ? kb[1].y : kb[1].w) : (((2 * k) & 3) == 0 ? kb[0].y : kb[0].w);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          mma_e4m3(c, id[half], b0, b1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int hrow = g + ((e & 2) ? 8 : 0);  // C row = kappa - 16*half
            const int n = 2 * t + (e & 1);           // C col = KV row within the group
            const int kappa = hrow;                  // within the half
            const int tk = kappa >> 2, i = kappa & 3;
            const int d = (W < 4 ? 128 * W + 32 * tk + 8 * k : 512 + 16 * tk + 8 * k) + 4 * half + i;
            const int r = base_row + n;
            if (r < row0 + nrows && r < total_kv) out[static_cast<int64_t>(r - row0) * 576 + d] = c[e];
          }
        }
      }
    }
  } else {
    // bf16: A = 16x16 identity (bf16 1.0 = 0x3F80); kappa = h.
    uint32_t id[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int arow = g + ((r & 1) ? 8 : 0);
      const int kbase = 2 * t + ((r & 2) ? 8 : 0);
      uint32_t wv = 0;
      if (kbase == arow) wv |= 0x3F80u;
      if (kbase + 1 == arow) wv |= 0x3F80u << 16;
      id[r] = wv;
    }
    const uint8_t* rowp = kv + static_cast<int64_t>(valid ? my_row : 0) * 1152;
#pragma unroll
    for (int W = 0; W < 9; ++W) {
      uint4 kb[2];
      const int off = 128 * W + 32 * t;
      kb[0] = valid ? __ldg(reinterpret_cast<const uint4*>(rowp + off)) : make_uint4(0, 0, 0, 0);
      kb[1] = valid ? __ldg(reinterpret_cast<const uint4*>(rowp + off + 16)) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4& src = kb[k >> 1];
        const uint32_t b0 = ((2 * k) & 3) == 0 ? src.x : src.z;
        const uint32_t b1 = ((2 * k) & 3) == 0 ? src.y : src.w;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16(c, id, b0, b1);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kappa = g + ((e & 2) ? 8 : 0);
          const int n = 2 * t + (e & 1);
          // kappa = 2tk + ee -> d = 64W + 16tk + 4k + ee; kappa = 8 + 2tk + ee -> +2
          const int hi = kappa >= 8, kk = kappa & 7, tk = kk >> 1, ee = kk & 1;
          const int d = 64 * W + 16 * tk + 4 * k + 2 * hi + ee;
          const int r = base_row + n;
          if (r < row0 + nrows && r < total_kv) out[static_cast<int64_t>(r - row0) * 576 + d] = c[e];
        }
      }
    }
  }
}

// mxfp4: one warp per row, lane b < 18 takes block b (32 dims). The value of
// dim d is operand byte d times the row factor 2^(R - 140), R = the row's
// largest block exponent: exactly code * 2^(s - 127) unless the block is
// flushed (more than 28 binades below R, then 0).
__global__ void mla_dequant_mx_kernel(const uint8_t* __restrict__ kv, const uint8_t* __restrict__ kv_scale,
                                      int32_t row0, int32_t nrows, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int i = 4 * blockIdx.x + (threadIdx.x >> 5);
  if (i >= nrows) return;
  const int64_t row = static_cast<int64_t>(row0) + i;
  const uint32_t s = lane < 18 ? kv_scale[row * 18 + lane] : 0u;
  uint32_t R = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) R = max(R, __shfl_xor_sync(0xffffffffu, R, o));
  if (lane >= 18) return;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(kv + row * 288 + 16 * lane));
  uint4 lo, hi;
  mxcvt::convert_block(v, mxcvt::rebase_scale2(R - s), lo, hi);
  const float f = mxcvt::exp2i(mxcvt::row_exp(R));
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  float* o = out + static_cast<int64_t>(i) * 576 + 32 * lane;
#pragma unroll
  for (int k = 0; k < 32; ++k) o[k] = mxcvt::e5m2_value(w[k >> 2] >> (8 * (k & 3))) * f;
}

cudaError_t launch_dequant(const void* kv, const void* kv_scale, int kv_fmt, int32_t total_kv, int32_t row0,
                           int32_t nrows, float* out, cudaStream_t stream) {
  if (nrows <= 0) return cudaSuccess;
  const int blocks = (nrows + 7) / 8;
  if (kv_fmt == kKvFp8) {
    mla_dequant_kernel<kKvFp8><<<blocks, 32, 0, stream>>>(static_cast<const uint8_t*>(kv), total_kv, row0, nrows, out);
  } else if (kv_fmt == kKvBf16) {
    mla_dequant_kernel<kKvBf16><<<blocks, 32, 0, stream>>>(static_cast<const uint8_t*>(kv), total_kv, row0, nrows, out);
  } else if (kv_fmt == kKvMxfp4) {
    mla_dequant_mx_kernel<<<(nrows + 3) / 4, 128, 0, stream>>>(static_cast<const uint8_t*>(kv),
                                                               static_cast<const uint8_t*>(kv_scale), row0, nrows, out);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mla
