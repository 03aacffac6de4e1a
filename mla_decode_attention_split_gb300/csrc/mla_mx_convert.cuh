// The mxfp4 element conversion of the mxfp4 stage-1 kernel, shared with the
// dequantisation check entry so that the check runs the kernel's own code.
//
// Format (OCP Microscaling, as the mxfp4 submission of
// kernelbot-amd-mixed-mla-675627 stores the cache): each byte holds two e2m1
// codes (element 2i in the low nibble), and each run of 32 elements along the
// head dimension shares one e8m0 scale 2^(s - 127).
//
// Conversion: every e2m1 element becomes an e5m2 byte rebased to the row's
// largest block exponent R with kHeadroom binades to spare:
// e5m2 = e2m1 * 2^(s - R + kHeadroom). The row factor 2^(R - 127 - kHeadroom)
// is applied separately (stage 1 puts it into the row's scores and softmax
// weights).
//  * The largest element, 6 * 2^13 = 49152, stays below the e5m2 maximum
//    (57344), so no block overflows.
//  * A block d = R - s binades below the largest is exact while
//    0.5 * 2^(13 - d) >= 2^-16 (the e5m2 subnormal step), i.e. d <= 28: e2m1
//    values have at most 2 significant bits.
//  * Blocks more than 28 binades below R are flushed to (signed) zero. Their
//    elements are below 2^-28 of the row's largest block.
//  * Route: the hardware conversion turns each byte (two e2m1 codes) into two
//    exact f16 values, an f16 multiply by 2^(13 - d) rebases them (exact, by
//    the points above, f16 reaching 2^-24), and e5m2 is the high byte of f16
//    (same exponent bias, two mantissa bits), so the bytes are exact.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "mla_device.cuh"

namespace mla {
namespace mxcvt {

constexpr int kHeadroom = 13;  // binades between the row's largest block and the e5m2 top
constexpr int kMaxDepth = 28;  // e5m2 holds e2m1 * 2^(kHeadroom - d) exactly for d <= 28

// f16x2 2^(kHeadroom - d) in both halves for a block d = R - s binades below
// the row's largest (0 for a flushed block). 2^-15 is the f16 subnormal
// 0x0200; 2^e for -14 <= e <= 13 is normal, exponent field e + 15.
__device__ __forceinline__ uint32_t rebase_scale2(uint32_t d) {
  const int e = kHeadroom - static_cast<int>(d);
  const uint32_t s = d <= static_cast<uint32_t>(kMaxDepth)
                         ? (e >= -14 ? static_cast<uint32_t>(e + 15) << 10 : 0x0200u)
                         : 0u;
  return s | (s << 16);
}

// The exponent of the row factor: K = e5m2 * 2^(R - 127 - kHeadroom).
__device__ __forceinline__ int row_exp(uint32_t R) { return static_cast<int>(R) - 127 - kHeadroom; }

// Eight e2m1 codes (one 32-bit word, element 0 in the lowest nibble) -> eight
// e5m2 bytes: byte i of out_lo is element i, of out_hi element 4 + i.
__device__ __forceinline__ void e2m1x8_to_e5m2x8(uint32_t w, uint32_t s2, uint32_t& out_lo, uint32_t& out_hi) {
  uint32_t h0, h1, h2, h3;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      " mul.rn.f16x2 %0, %0, %5;\n mul.rn.f16x2 %1, %1, %5;\n"
      " mul.rn.f16x2 %2, %2, %5;\n mul.rn.f16x2 %3, %3, %5;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w), "r"(s2));
  out_lo = prmt(h0, h1, 0x7531u);  // high bytes of the four f16 values
  out_hi = prmt(h2, h3, 0x7531u);
}

// One block: 32 e2m1 codes (16 bytes) -> 32 e5m2 bytes as two 16-byte units
// (elements 0..15 in lo, 16..31 in hi).
__device__ __forceinline__ void convert_block(const uint4& v, uint32_t s2, uint4& lo, uint4& hi) {
  e2m1x8_to_e5m2x8(v.x, s2, lo.x, lo.y);
  e2m1x8_to_e5m2x8(v.y, s2, lo.z, lo.w);
  e2m1x8_to_e5m2x8(v.z, s2, hi.x, hi.y);
  e2m1x8_to_e5m2x8(v.w, s2, hi.z, hi.w);
}

// 2^e for an integer e in [-149, 127] (exact; fp32 subnormals below -126).
__device__ __forceinline__ float exp2i(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                   : __uint_as_float(1u << static_cast<uint32_t>(max(e + 149, 0)));
}

// The value of an e5m2 byte (exact: it is the high byte of an f16).
__device__ __forceinline__ float e5m2_value(uint32_t byte) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>((byte & 0xFFu) << 8)));
}

}  // namespace mxcvt
}  // namespace mla
