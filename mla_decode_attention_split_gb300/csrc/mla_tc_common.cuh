// Pieces shared by the tcgen05 stage-1 kernels (fp8 KV in mla_stage1_tc.cu,
// mxfp4 KV in mla_stage1_mx.cu): tile geometry, the shared-memory context,
// the tile walker, the per-head warp reductions and the q operand setup.
//
// Both kernels compute, per query token and split, the online-softmax partial
// of split-K flash decoding (kernelbot-amd-mixed-mla-753817,
// `mla_flash_decode_stage1`) with 128 KV rows as the MMA M dimension and the
// 16 heads (hi and lo halves of the bf16 operand, N = 32) as N.
#pragma once

#include <cuda.h>

#include "mla_device.cuh"
#include "mla_internal.h"
#include "mla_merge.cuh"
#include "mla_partition.cuh"
#include "mla_tcgen05.cuh"

namespace mla {
namespace tc {

constexpr int kTileRows = 128;
constexpr int kVChunks = 4;                   // 128-byte column chunks of the 512 V dims
constexpr int kChunkBytes = kTileRows * 128;  // 16 KB (one 128 x 128 B swizzled box)
constexpr int kVBytes = kVChunks * kChunkBytes;  // 64 KB
constexpr int kQChunkBytes = 32 * 128;        // 32 B-operand rows (hi, lo) x 128 B
constexpr int kQBytes = 5 * kQChunkBytes;     // 20 KB (chunk 4: rope dims, 64 B used)
constexpr int kRopeBytes = kTileRows * 64;    // [row group 16][16-B column 4][8 rows][16 B]
constexpr int kPBytes = kTileRows * 32;       // [row group][hi | lo][8 rows][16 heads]
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;                // 2 buffers x 32 columns
constexpr uint32_t kTmemO = 64;               // 2 buffers x (4 blocks x 32 columns)
constexpr float kLoScale = 16.0f;
// Lazy rescaling (the e4m3-P kernels): a head's reference max m moves only
// when a tile's max exceeds it by more than kMaxSlack (log2 units). Until then
// the weights exp2(x - m) may reach 2^kMaxSlack, so they are scaled by
// kPScale, with kPScale * 2^kMaxSlack (362) below e4m3's largest value (448).
// O, l and the LSE share the reference, so the softmax is the same; O in
// tensor memory is rescaled only when the reference moves.
constexpr float kMaxSlack = 3.5f;
constexpr float kPScale = 32.0f;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory context of one CTA; LL is the kernel's layout (offsets and
// barrier indices).
template <class LL>
struct Ctx {
  uint8_t* g;  // generic pointer to the 1024-aligned base
  uint32_t s;  // shared address of the aligned base
  volatile uint32_t* abort_word;
  uint32_t* flags;
  uint32_t tmem;
  int64_t total;  // virtual rows of the whole launch
  int64_t parts;  // CTAs that share them: min(num_splits, total), so that no range is empty
  __device__ __forceinline__ uint32_t bar(int i) const { return s + LL::kOffBars + 8u * i; }
  __device__ __forceinline__ bool wait(int i, uint32_t parity) const { return mbar_wait(bar(i), parity, abort_word, flags); }
};

// Bounded wait used while draining on exit (no abort check: the CTA leaves
// either way).
__device__ __forceinline__ void mbar_wait_drain_tc(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// Walks the CTA's tiles in order (one 128-row tile at a time).
struct TileRef {
  int32_t row, seg, k0, nvalid, pbase;
};

struct TileWalker {
  PieceCursor cur;
  Piece pc;
  int r0 = 0;
  bool have = false;
  __device__ void init(const PieceCursor& c) {
    cur = c;
    have = cur.next(pc);
    r0 = 0;
  }
  // First KV row of the next tile. Returns false when done.
  __device__ bool next(int32_t& row) {
    if (!have) return false;
    row = pc.kv_row + r0;
    r0 += kTileRows;
    if (r0 >= pc.nrows) {
      have = cur.next(pc);
      r0 = 0;
    }
    return true;
  }
  // The next tile: its first KV row, segment, the segment's first row and
  // how many of its rows belong to the piece. Returns false when done.
  __device__ bool next(TileRef& t) {
    if (!have) return false;
    t.row = pc.kv_row + r0;
    t.seg = pc.seg;
    t.k0 = pc.k0;
    t.nvalid = pc.nrows - r0;
    t.pbase = pc.pbase;
    r0 += kTileRows;
    if (r0 >= pc.nrows) {
      have = cur.next(pc);
      r0 = 0;
    }
    return true;
  }
};

// Paged KV, in two steps so that the page-table load is in flight while other
// work proceeds. page_of issues the load of the page id of row i of the
// segment whose first page-table entry is pbase (the entry read is inside
// [page_indptr[seg], page_indptr[seg+1]) because i is below the segment's row
// count); phys_row turns it into the
// physical row, or -1: for a row outside the piece (page_of_none), and, with
// the error flag raised, for a page id outside the pool.
struct PagedRow {
  int32_t id, slot;  // slot < 0: no row
};

__device__ __forceinline__ PagedRow page_of(const Stage1Params& p, int32_t pbase, int32_t i) {
  const int32_t pg = p.page_shift >= 0 ? (i >> p.page_shift) : i / p.page_size;
  return PagedRow{__ldg(p.page_indices + pbase + pg), i - pg * p.page_size};
}

__device__ __forceinline__ PagedRow page_of_none() { return PagedRow{0, -1}; }

// (The pool holds fewer than 2^31 rows: the host checks num_pages * page_size.)
__device__ __forceinline__ int32_t phys_row(const Stage1Params& p, PagedRow r) {
  if (r.slot < 0) return -1;
  if (static_cast<uint32_t>(r.id) >= static_cast<uint32_t>(p.num_pages)) {
    atomicOr(p.dev_flags, kFlagBadPage);
    return -1;
  }
  return r.id * p.page_size + r.slot;
}

// The page ids of tile rows lane + 32 j (j = 0..3) of the next tile.
__device__ __forceinline__ bool paged_tile_ids(const Stage1Params& p, TileWalker& tw, int lane, PagedRow (&id)[4]) {
  TileRef t;
  const bool have = tw.next(t);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = 32 * j + lane;
    id[j] = (have && row < t.nvalid) ? page_of(p, t.pbase, t.row - t.k0 + row) : page_of_none();
  }
  return have;
}

// Per-tile bookkeeping of the UMMA issuer, packed in one word: bit 0 = first
// tile of its piece, bit 1 = last tile of its piece, bits 2.. = piece index
// within the CTA.
struct TileMeta {
  uint32_t k;
  bool first, last;
  __device__ static TileMeta unpack(uint32_t w) { return TileMeta{w >> 2, (w & 1u) != 0, (w & 2u) != 0}; }
};

// The CTA's tiles in order, with their bookkeeping words.
struct MetaTileWalker {
  PieceCursor cur;
  Piece pc;
  int r0 = 0;
  uint32_t k = 0;
  bool have = false;
  __device__ void init(const PieceCursor& c) {
    cur = c;
    have = cur.next(pc);
    r0 = 0;
    k = 0;
  }
  // First KV row and bookkeeping word of the next tile. Returns false when done.
  __device__ bool next(int32_t& row, uint32_t& meta) {
    if (!have) return false;
    row = pc.kv_row + r0;
    meta = (k << 2) | (r0 == 0 ? 1u : 0u) | (r0 + kTileRows >= pc.nrows ? 2u : 0u);
    r0 += kTileRows;
    if (r0 >= pc.nrows) {
      have = cur.next(pc);
      r0 = 0;
      ++k;
    }
    return true;
  }
};

__device__ __forceinline__ int count_tiles(PieceCursor cur) {
  Piece t;
  int n = 0;
  while (cur.next(t)) n += (t.nrows + kTileRows - 1) / kTileRows;
  return n;
}

// Max (or sum) of 16 per-head values over the 32 lanes of a warp: each halving
// step trades half of the heads with the partner lane, so after four steps
// lane l holds head l >> 1 over 16 lanes and a last step completes the warp.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 16;
    const float keep = up ? v[i + 8] : v[i], send = up ? v[i] : v[i + 8];
    const float r = __shfl_xor_sync(0xffffffffu, send, 16);
    a[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  float b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 8;
    const float keep = up ? a[i + 4] : a[i], send = up ? a[i] : a[i + 4];
    const float r = __shfl_xor_sync(0xffffffffu, send, 8);
    b[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  float c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 4;
    const float keep = up ? b[i + 2] : b[i], send = up ? b[i] : b[i + 2];
    const float r = __shfl_xor_sync(0xffffffffu, send, 4);
    c[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  const bool up = lane & 2;
  const float keep = up ? c[1] : c[0], send = up ? c[0] : c[1];
  const float r = __shfl_xor_sync(0xffffffffu, send, 2);
  float d = kMax ? fmaxf(keep, r) : keep + r;
  const float r1 = __shfl_xor_sync(0xffffffffu, d, 1);
  return kMax ? fmaxf(d, r1) : d + r1;
}

// Max of each of 16 per-head values over the 32 lanes of a warp (every lane
// gets all 16): 16 independent warp reductions (redux.sync, sm_100 family).
// NaN inputs are ignored, as fmaxf does.
__device__ __forceinline__ void warp_max16(const float (&v)[16], float (&r)[16]) {
#pragma unroll
  for (int h = 0; h < 16; ++h) asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r[h]) : "f"(v[h]));
}

// Lane 0 stores 16 per-head values of the warp as 4 x 16 bytes (16-byte aligned dst).
__device__ __forceinline__ void store16(float* dst, const float (&r)[16], int lane) {
  if (lane == 0) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
  }
}

// The 4 softmax warps: thread = tile row = tensor-memory lane.
struct SoftmaxCtx {
  int row, wi, lane;
  uint32_t lane_base;
  uint32_t gcount;
};

// Barrier among the 4 softmax warps (two alternating mbarriers of count 4).
template <class LL>
__device__ __forceinline__ bool group_sync(const Ctx<LL>& cx, SoftmaxCtx& sx) {
  const uint32_t k = sx.gcount & 1u, par = (sx.gcount >> 1) & 1u;
  ++sx.gcount;
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(LL::kGrp + k));
  return cx.wait(LL::kGrp + k, par);
}

// q of one token -> the Q buffer as the B operand (K-major, 128B swizzle,
// rows 0-15 = e4m3(q 2^shift), rows 16-31 = e4m3(16 (q 2^shift - hi))).
// Returns the score scale (exp2 domain, times `kvsc`) or a negative value on
// abort. Piece kk >= 1 waits until the previous piece's last Q.K^T is done.
// x / s rounded to nearest even, from inv = RN(1 / s), by one residual
// correction (Markstein's theorem; P. Markstein, "IA-64 and Elementary
// Functions", 2000, ch. 8): with q0 = RN(x inv) and the exact residual
// r = x - q0 s from an FMA, RN(q0 + r inv) is the correctly rounded quotient
// when neither the quotient nor the residual leaves the normal range. Here
// |x / s| <= 448 (s is the tensor's amax / 448); quotients below the normal
// range are far under the smallest e4m3 subnormal, so their code is 0 either
// way.
__device__ __forceinline__ float quotient_rn(float x, float s, float inv) {
  const float q0 = x * inv;
  const float r = fmaf(-q0, s, x);
  return fmaf(r, inv, q0);
}

// q of one token into rows row0..row0+31 of the Q buffer (chunks of
// kChunk bytes); returns the score scale or a negative value on abort. With
// fp8 codes and kLo false only rows row0..row0+15 are written (no lo rows).
template <class LL, int QF, int kChunk, bool kLo = true>
__device__ float fill_q(const Stage1Params& p, const Ctx<LL>& cx, SoftmaxCtx& sx, int token, int row0, uint32_t kk,
                        float kvsc) {
  const int t = 32 * sx.wi + sx.lane;  // 0..127
  const int h = t >> 3, d0 = 72 * (t & 7);
  uint8_t* qb = cx.g + LL::kOffQ;
  auto qaddr = [&](int r, int d) -> uint32_t* {
    const int row = row0 + r;
    const int unit = (d & 127) >> 4;
    return reinterpret_cast<uint32_t*>(qb + (d >> 7) * kChunk + (row >> 3) * 1024 + (row & 7) * 128 +
                                       ((unit ^ (row & 7)) << 4) + (d & 15));
  };
  float c;
  if (QF == kQBf16Quant) {
    // e4m3 codes of q / s (RNE, saturated), lo rows zero; s from the workspace,
    // written by the amax kernel that may still run (programmatic launch)
    if (kk == 0) griddep_wait();
    const uint16_t* src = static_cast<const uint16_t*>(p.q) + (static_cast<int64_t>(token) * kHeads + h) * kDqk + d0;
    const float qs = *static_cast<const volatile float*>(p.q_scale);
    const float inv = 1.0f / qs;  // correctly rounded, once
    uint4 v[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t code[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float a = quotient_rn(bf16_bits_to_f32(w[2 * k] & 0xFFFFu), qs, inv);
        const float b = quotient_rn(bf16_bits_to_f32(w[2 * k] >> 16), qs, inv);
        const float e = quotient_rn(bf16_bits_to_f32(w[2 * k + 1] & 0xFFFFu), qs, inv);
        const float f = quotient_rn(bf16_bits_to_f32(w[2 * k + 1] >> 16), qs, inv);
        code[k] = f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(e, f) << 16);
      }
      *qaddr(h, d0 + 8 * i) = code[0];
      *qaddr(h, d0 + 8 * i + 4) = code[1];
      if (kLo) {
        *qaddr(16 + h, d0 + 8 * i) = 0u;
        *qaddr(16 + h, d0 + 8 * i + 4) = 0u;
      }
    }
    c = p.sm_scale * kLog2e * kvsc * qs;
  } else if (QF == kQBf16) {
    const uint16_t* src = static_cast<const uint16_t*>(p.q) + (static_cast<int64_t>(token) * kHeads + h) * kDqk + d0;
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 36; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
    mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // per-warp maxima; rows 32.. of a two-token Q buffer use their own four words
    uint32_t* am = reinterpret_cast<uint32_t*>(cx.g + LL::kOffAmax) + 4 * (row0 >> 5);
    if (sx.lane == 0) am[sx.wi] = mx;
    if (!group_sync(cx, sx)) return -1.f;
    mx = max(max(am[0], am[1]), max(am[2], am[3]));
    const int e = static_cast<int>((mx >> 7) & 0xFF);  // biased exponent of max |q|
    int shift = (mx == 0) ? 0 : 134 - e;               // max |q| 2^shift in [128, 256)
    shift = max(-126, min(126, shift));
    const float up = __uint_as_float(static_cast<uint32_t>(shift + 127) << 23);
    const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
#pragma unroll
    for (int g = 0; g < 18; ++g) {  // groups of 4 dims: d0 + 4g
      const float x0 = bf16_bits_to_f32(w[2 * g] & 0xFFFFu) * up, x1 = bf16_bits_to_f32(w[2 * g] >> 16) * up;
      const float x2 = bf16_bits_to_f32(w[2 * g + 1] & 0xFFFFu) * up, x3 = bf16_bits_to_f32(w[2 * g + 1] >> 16) * up;
      const uint32_t h01 = f32x2_to_e4m3x2(x0, x1), h23 = f32x2_to_e4m3x2(x2, x3);
      const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
      const uint32_t l01 = f32x2_to_e4m3x2(kLoScale * (x0 - d01.x), kLoScale * (x1 - d01.y));
      const uint32_t l23 = f32x2_to_e4m3x2(kLoScale * (x2 - d23.x), kLoScale * (x3 - d23.y));
      *qaddr(h, d0 + 4 * g) = h01 | (h23 << 16);
      *qaddr(16 + h, d0 + 4 * g) = l01 | (l23 << 16);
    }
    c = p.sm_scale * kLog2e * kvsc * down;
  } else {
    const uint8_t* src = static_cast<const uint8_t*>(p.q) + (static_cast<int64_t>(token) * kHeads + h) * kDqk + d0;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + i);
      *qaddr(h, d0 + 8 * i) = v.x;
      *qaddr(h, d0 + 8 * i + 4) = v.y;
      if (kLo) {
        *qaddr(16 + h, d0 + 8 * i) = 0u;
        *qaddr(16 + h, d0 + 8 * i + 4) = 0u;
      }
    }
    c = p.sm_scale * kLog2e * kvsc * __ldg(p.q_scale);
  }
  return c;
}

// q of one token -> the Q buffer, handed to the MMA warp (see fill_q).
template <class LL, int QF>
__device__ float setup_q(const Stage1Params& p, const Ctx<LL>& cx, SoftmaxCtx& sx, int token, uint32_t kk, float kvsc) {
  if (kk >= 1 && !cx.wait(LL::kQEmpty, (kk - 1) & 1u)) return -1.f;
  const float c = fill_q<LL, QF, kQChunkBytes>(p, cx, sx, token, 0, kk, kvsc);
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(LL::kQFull));
  return c;
}

// One row's 64 rope bytes into a no-swizzle K-major A operand: 8-row x 16-byte
// core matrices, 128 B apart along K, 512 B apart along rows.
__device__ __forceinline__ void put_rope_row(uint8_t* rope_base, int row, const uint4 (&r)[4]) {
  uint8_t* base = rope_base + (row >> 3) * 512 + (row & 7) * 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(base + i * 128) = r[i];
}

// UMMA descriptors for the two products of a tile, shared by both kernels.
//   Q.K^T k-step ks (32 dims): A = KV rows (K-major, 128B swizzle), B = Q.
__device__ __forceinline__ uint64_t qk_desc_a(uint32_t vbase, int ks) {
  return smem_desc(vbase + (ks >> 2) * kChunkBytes + (ks & 3) * 32, 16, 1024, kLayoutSw128);
}
__device__ __forceinline__ uint64_t qk_desc_b(uint32_t qbuf, int ks) {
  return smem_desc(qbuf + (ks >> 2) * kQChunkBytes + (ks & 3) * 32, 16, 1024, kLayoutSw128);
}
//   rope k-step ks (32 dims): A = the no-swizzle rope operand, B = Q chunk 4.
__device__ __forceinline__ uint64_t rope_desc_a(uint32_t rope, int ks) {
  return smem_desc(rope + ks * 256, 128, 512, kLayoutNone);
}
//   P.V: A = V^T dims 128 mb.. of rows 32 ks.. (MN-major, 8-row atoms 1024 B
//   apart); B = P^T with N = 32 (hi heads, lo heads: core matrices 128 B
//   apart), K = rows (8-row groups 256 B apart).
__device__ __forceinline__ uint64_t pv_desc_a(uint32_t vbase, int mb, int ks) {
  return smem_desc(vbase + mb * kChunkBytes + ks * 4096, kChunkBytes, 1024, kLayoutSw128);
}
__device__ __forceinline__ uint64_t pv_desc_b(uint32_t pbuf, int ks) { return smem_desc(pbuf + ks * 1024, 256, 128, kLayoutNone); }

// One row of softmax weights (16 heads, already times kPScale) as hi/lo e4m3
// into the P operand.
__device__ __forceinline__ void put_p_row(uint8_t* pbuf, int row, const float (&pv)[16]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t h01 = f32x2_to_e4m3x2(pv[4 * q4], pv[4 * q4 + 1]), h23 = f32x2_to_e4m3x2(pv[4 * q4 + 2], pv[4 * q4 + 3]);
    const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
    hi[q4] = h01 | (h23 << 16);
    lo[q4] = f32x2_to_e4m3x2(kLoScale * (pv[4 * q4] - d01.x), kLoScale * (pv[4 * q4 + 1] - d01.y)) |
             (f32x2_to_e4m3x2(kLoScale * (pv[4 * q4 + 2] - d23.x), kLoScale * (pv[4 * q4 + 3] - d23.y)) << 16);
  }
  uint8_t* pb = pbuf + (row >> 3) * 256 + (row & 7) * 16;
  *reinterpret_cast<uint4*>(pb) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(pb + 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Multiplies the 4 x 32 O columns of this thread's lane by alpha[head].
__device__ __forceinline__ void rescale_o(uint32_t ob, const float (&alpha)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[32];
    tmem_ld32(ob + 32 * mb, o);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j & 15]);
    tmem_st32(ob + 32 * mb, o);
  }
  tmem_wait_st();
}

// One 128-dim block mb of a piece's epilogue: O (hi + lo/16 columns) times
// f[head] to the bf16 output (a whole-run piece) or the fp32 partial slot.
__device__ __forceinline__ void store_o_block(const Stage1Params& p, const Piece& pc, uint32_t ob, int row,
                                              const float (&f)[16], int mb) {
  uint32_t o[32];
  tmem_ld32(ob + 32 * mb, o);
  tmem_wait_ld();
  const int dim = 128 * mb + row;
  if (pc.direct) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(pc.token) * kHeads * kDv + dim;
#pragma unroll
    for (int h = 0; h < 16; ++h)
      dst[h * kDv] = __float2bfloat16_rn((__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h]);
  } else {
    float* dst = p.part_o + pc.slot * kHeads * kDv + dim;
#pragma unroll
    for (int h = 0; h < 16; ++h)
      dst[h * kDv] = (__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h];
  }
}

// Epilogue for one piece: O (hi + lo/16 columns) times f[head] to the bf16
// output (a whole-run piece) or the fp32 partial slot.
__device__ __forceinline__ void store_o(const Stage1Params& p, const Piece& pc, uint32_t ob, int row, const float (&f)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[32];
    tmem_ld32(ob + 32 * mb, o);
    tmem_wait_ld();
    const int dim = 128 * mb + row;
    if (pc.direct) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(pc.token) * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        dst[h * kDv] = __float2bfloat16_rn((__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h]);
    } else {
      float* dst = p.part_o + pc.slot * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        dst[h * kDv] = (__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h];
    }
  }
}

// Merge of split tokens (the pages' stage 2). The CTA whose partial completes a
// token's count merges it, at the very end of the CTA when its stage buffers
// are free: with L = max_s lse_s, out = sum_s 2^(lse_s - L) O_s /
// sum_s 2^(lse_s - L) over the partial slots G c + token of the CTAs c0..c1 that
// hold pieces of the token. A CTA holds at most two split pieces (the first
// and the last of its range) of at most four tokens each, so it merges at most
// eight tokens.
constexpr uint32_t kMergeMax = 8;
struct MergeList {
  uint32_t n;                                           // tokens this CTA merges
  int32_t token[kMergeMax], c0[kMergeMax], c1[kMergeMax];  // token and the CTAs that hold its pieces
  uint32_t pad[7];
};
static_assert(sizeof(MergeList) == 128, "merge list slot");

// After the 128 softmax threads wrote this CTA's partial of a split token:
// publish it and count it on the token's counter; if it completes the count,
// list the token for the end-of-CTA merge. The group barrier orders all 128
// threads' writes before thread 0's gpu-scope fence, which is cumulative, so
// only thread 0 waits for the writes to reach L2. Returns false on abort.
template <class LL>
__device__ __forceinline__ bool finish_partial(const Stage1Params& p, const Ctx<LL>& cx, SoftmaxCtx& sx,
                                               const Piece& pc) {
  if (!group_sync(cx, sx)) return false;
  if (sx.wi == 0 && sx.lane == 0) {
    __threadfence();
    const int64_t P = cx.parts;
    const int64_t c0 = part_of_row(pc.tok_vs, cx.total, P), c1 = part_of_row(pc.tok_vs + pc.kvlen - 1, cx.total, P);
    MergeList* ml = reinterpret_cast<MergeList*>(cx.g + LL::kOffMList);
    for (int i = 0; i < pc.ntok; ++i) {  // every token of the group
      const uint32_t arrived = atomicAdd(p.tok_cnt + pc.token + i, 1u) + 1u;
      // cooperative merge: every CTA of the token lists it; otherwise the one that completes its count
      if ((p.coop_merge || arrived == static_cast<uint32_t>(c1 - c0 + 1)) && ml->n < kMergeMax) {
        ml->token[ml->n] = pc.token + i;
        ml->c0[ml->n] = static_cast<int32_t>(c0);
        ml->c1[ml->n] = static_cast<int32_t>(c1);
        ++ml->n;
      }
    }
  }
  return true;
}

// The end-of-CTA merges, by all kThreads threads. Slots come into the stage
// buffers in batches of up to kSlots by bulk copies (one round trip a batch).
// The merge weights depend only on (slot, head): per batch, 16 threads (one
// per head) update the running maximum M of the LSEs, the rescale factor of
// what was merged so far, the batch's weights 2^(lse - M) and their running
// sum, and every thread then accumulates its float4 elements with FMAs.
template <class LL>
__device__ void merge_listed(const Stage1Params& p, const Ctx<LL>& cx) {
  constexpr int kThr = LL::kThreads;
  constexpr int kSlotBytes = kHeads * kDv * 4;  // 32 KB
  constexpr int kSlots = LL::kMergeBytes / kSlotBytes < 6 ? LL::kMergeBytes / kSlotBytes : 6;
  constexpr int kF = (kHeads * kDv / 4 + kThr - 1) / kThr;  // float4 elements per thread
  static_assert(kSlots >= 1, "merge buffers");
  const MergeList* ml = reinterpret_cast<const MergeList*>(cx.g + LL::kOffMList);
  const uint32_t nm = ml->n < kMergeMax ? ml->n : kMergeMax;
  // scratch in the (free) Q buffer: the batch's LSEs [kSlots][16], weights
  // [kSlots][16], and per head the rescale factor, running max and sum
  float* lsebuf = reinterpret_cast<float*>(cx.g + LL::kOffQ);
  float* wbuf = lsebuf + kSlots * kHeads;
  float* scbuf = wbuf + kSlots * kHeads;
  float* mbuf = scbuf + kHeads;
  float* sbuf = mbuf + kHeads;
  uint32_t batch = 0;
  for (uint32_t e = 0; e < nm; ++e) {
    const int token = ml->token[e];
    const int64_t c0 = ml->c0[e], np = static_cast<int64_t>(ml->c1[e]) - c0 + 1;
    float4 acc[kF];
#pragma unroll
    for (int i = 0; i < kF; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < kHeads) {
      mbuf[threadIdx.x] = -INFINITY;
      sbuf[threadIdx.x] = 0.f;
    }
    for (int64_t s0 = 0; s0 < np; s0 += kSlots) {
      const int nb = static_cast<int>(np - s0 < kSlots ? np - s0 : static_cast<int64_t>(kSlots));
      if (threadIdx.x == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");  // partials written through the generic proxy
        mbar_arrive_expect_tx(cx.bar(LL::kMerge), nb * (kSlotBytes + kHeads * 4));
        for (int j = 0; j < nb; ++j) {
          const int64_t slot = p.group * (c0 + s0 + j) + token;
          bulk_g2s(cx.s + LL::kOffKv + j * kSlotBytes, p.part_o + slot * kHeads * kDv, kSlotBytes, cx.bar(LL::kMerge),
                   policy_evict_first());
          bulk_g2s(cx.s + LL::kOffQ + j * kHeads * 4, p.part_lse + slot * kHeads, kHeads * 4, cx.bar(LL::kMerge),
                   policy_evict_first());
        }
      }
      // all threads agree before any of them moves on (a lone timeout must not
      // leave the others at the barrier below)
      if (!__syncthreads_and(cx.wait(LL::kMerge, batch & 1u) ? 1 : 0)) return;
      ++batch;
      if (threadIdx.x < kHeads) {
        const int h = threadIdx.x;
        float mn = mbuf[h];
        for (int j = 0; j < nb; ++j) mn = fmaxf(mn, lsebuf[j * kHeads + h]);
        const float sc = fast_exp2(mbuf[h] - mn);
        float sum = sbuf[h] * sc;
        for (int j = 0; j < nb; ++j) {
          const float w = fast_exp2(lsebuf[j * kHeads + h] - mn);
          wbuf[j * kHeads + h] = w;
          sum += w;
        }
        scbuf[h] = sc;
        mbuf[h] = mn;
        sbuf[h] = sum;
      }
      __syncthreads();
      const float4* obuf = reinterpret_cast<const float4*>(cx.g + LL::kOffKv);
#pragma unroll
      for (int i = 0; i < kF; ++i) {
        const int f = threadIdx.x + i * kThr;
        if (f < kHeads * kDv / 4) {
          const int h = f >> 7;  // 128 float4 per head
          const float sc = scbuf[h];
          float4 a = make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc);
          for (int j = 0; j < nb; ++j) {
            const float w = wbuf[j * kHeads + h];
            const float4 v = obuf[j * (kSlotBytes / 16) + f];
            a.x = fmaf(w, v.x, a.x);
            a.y = fmaf(w, v.y, a.y);
            a.z = fmaf(w, v.z, a.z);
            a.w = fmaf(w, v.w, a.w);
          }
          acc[i] = a;
        }
      }
      __syncthreads();  // the buffers are free for the next batch
    }
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(token) * kHeads * kDv;
#pragma unroll
    for (int i = 0; i < kF; ++i) {
      const int f = threadIdx.x + i * kThr;
      if (f < kHeads * kDv / 4) {
        const float inv = 1.0f / sbuf[f >> 7];
        *reinterpret_cast<uint2*>(dst + 4 * f) =
            make_uint2(pack_bf16x2(acc[i].x * inv, acc[i].y * inv), pack_bf16x2(acc[i].z * inv, acc[i].w * inv));
      }
    }
    if (threadIdx.x == 0) p.tok_cnt[token] = 0u;
    __syncthreads();  // the per-head sums are read before the next token resets them
  }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The cooperative end-of-CTA merge, when every CTA of the launch is resident
// at once (p.coop_merge). The n CTAs c0..c1 that hold pieces of a split token
// share its merge: once the token's count has reached n (all its partials
// published), CTA c0 + r takes units [64 r / n, 64 (r + 1) / n) of the 64
// units (head h, 128-dim quarter q) = 4 h + q. Each unit is the pages' stage 2
// over the token's n slots G c + token: L = max lse, w = 2^(lse - L),
// out = sum w O / sum w, bf16 RNE. The units' slot rows (512 B each) come into
// the free stage buffers by 16-byte asynchronous copies, one warp per row and
// all of a batch in flight at once, as many units at a time as fit; one
// thread per unit computes its weights from the LSEs (L2 loads), and one warp
// then merges a unit (lane l: float4 l of the quarter). A second round of
// counts returns the
// token's counter to zero: the CTA that brings it to 2 n resets it, after all n
// have passed their wait. All LL::kThreads threads call this.
template <class LL>
__device__ void merge_coop(const Stage1Params& p, const Ctx<LL>& cx) {
  constexpr int kWarps = LL::kThreads / 32;
  constexpr int kRowBytes = 128 * 4;                      // one unit row of one slot
  constexpr int kCap = LL::kMergeBytes / kRowBytes;       // rows per batch
  constexpr int kMaxUnits = kCap / 2;                     // a split token has n >= 2 slots
  static_assert(kMaxUnits <= LL::kThreads, "one thread per unit of a batch");
  static_assert(LL::kOffMList - LL::kOffQ >= 24 * kCap, "merge scratch between the Q buffer and the merge list");
  const MergeList* ml = reinterpret_cast<const MergeList*>(cx.g + LL::kOffMList);
  const int nm = static_cast<int>(ml->n < kMergeMax ? ml->n : kMergeMax);
  bool ok = true;
  if (threadIdx.x < nm) {
    const uint32_t need = static_cast<uint32_t>(ml->c1[threadIdx.x] - ml->c0[threadIdx.x] + 1);
    const uint32_t* cnt = p.tok_cnt + ml->token[threadIdx.x];
    const long long t0 = clock64();
    while (ld_acquire_u32(cnt) < need) {
      if (*cx.abort_word) {
        ok = false;
        break;
      }
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicOr(cx.flags, kFlagTimeout);
        ok = false;
        break;
      }
    }
  }
  if (!__syncthreads_and(ok ? 1 : 0)) return;
  // this CTA's units of each listed token: units [ub[e], ub[e] + cnt[e]) of n[e] rows each
  int cnt[kMergeMax], ub[kMergeMax], nn[kMergeMax], units = 0;
#pragma unroll
  for (int e = 0; e < static_cast<int>(kMergeMax); ++e) {
    cnt[e] = ub[e] = nn[e] = 0;
    if (e < nm) {
      const int n = ml->c1[e] - ml->c0[e] + 1, r = static_cast<int>(blockIdx.x) - ml->c0[e];
      nn[e] = n;
      ub[e] = 64 * r / n;
      cnt[e] = 64 * (r + 1) / n - ub[e];
      units += cnt[e];
    }
  }
  // scratch in the (free) Q buffer: per unit of a batch {token, n, unit}, its first row and 1 / sum of its
  // weights; per row its weight and the float offset of its source in the partials
  int4* uinfo = reinterpret_cast<int4*>(cx.g + LL::kOffQ);
  int* urow = reinterpret_cast<int*>(uinfo + kMaxUnits);
  float* uinv = reinterpret_cast<float*>(urow + kMaxUnits);
  float* rw = uinv + kMaxUnits;
  int64_t* rsrc = reinterpret_cast<int64_t*>(rw + kCap);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t pol = policy_evict_first();
  int e0 = 0, i0 = 0;  // the batch's first unit: unit i0 of entry e0
  while (e0 < nm) {
    // the batch: whole units while their rows fit (the same walk in every thread)
    int rows = 0, nb = 0, e1 = e0, i1 = i0;
    while (e1 < nm) {
      const int take = min(min(cnt[e1] - i1, (kCap - rows) / nn[e1]), kMaxUnits - nb);
      rows += take * nn[e1];
      nb += take;
      i1 += take;
      if (i1 < cnt[e1]) break;  // full
      ++e1;
      i1 = 0;
    }
    if (static_cast<int>(threadIdx.x) < nb) {
      // unit t of the batch: entry e, index i; rows before it in the batch
      int t = threadIdx.x, e = e0, i = i0, before = 0;
      while (t >= cnt[e] - i) {
        t -= cnt[e] - i;
        before += (cnt[e] - i) * nn[e];
        ++e;
        i = 0;
      }
      i += t;
      before += t * nn[e];
      const int token = ml->token[e], n = nn[e], u = ub[e] + i, h = u >> 2, q = u & 3;
      const int64_t c0 = ml->c0[e];
      float mx = -INFINITY;
      for (int j0 = 0; j0 < n; j0 += 8) {  // eight LSE loads in flight, then their stores
        float l8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          l8[k] = j0 + k < n ? __ldcg(p.part_lse + (p.group * (c0 + j0 + k) + token) * kHeads + h) : -INFINITY;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (j0 + k < n) {
            rsrc[before + j0 + k] = ((p.group * (c0 + j0 + k) + token) * kHeads + h) * kDv + 128 * q;
            rw[before + j0 + k] = l8[k];
          }
          mx = fmaxf(mx, l8[k]);
        }
      }
      float sum = 0.f;
      for (int j = 0; j < n; ++j) {
        const float w = fast_exp2(rw[before + j] - mx);
        rw[before + j] = w;
        sum += w;
      }
      uinfo[threadIdx.x] = make_int4(token, n, u, 0);
      urow[threadIdx.x] = before;
      uinv[threadIdx.x] = 1.0f / sum;
    }
    __syncthreads();
    for (int r = warp; r < rows; r += kWarps)
      cp_async16(cx.s + LL::kOffKv + r * kRowBytes + 16 * lane, p.part_o + rsrc[r] + 4 * lane, pol);
    cp_async_wait_all();
    __syncthreads();
    for (int t = warp; t < nb; t += kWarps) {
      const int4 ui = uinfo[t];
      const int rb = urow[t];
      const float4* src = reinterpret_cast<const float4*>(cx.g + LL::kOffKv + static_cast<int64_t>(rb) * kRowBytes);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < ui.y; ++j) {
        const float w = rw[rb + j];
        const float4 v = src[j * (kRowBytes / 16) + lane];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
      const float inv = uinv[t];
      const int h = ui.z >> 2, q = ui.z & 3;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(ui.x) * kHeads + h) * kDv +
                           128 * q + 4 * lane;
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    __syncthreads();  // the buffers are free for the next batch
    e0 = e1;
    i0 = i1;
  }
  if (threadIdx.x < nm) {
    const uint32_t need = static_cast<uint32_t>(ml->c1[threadIdx.x] - ml->c0[threadIdx.x] + 1);
    uint32_t* cnt_w = p.tok_cnt + ml->token[threadIdx.x];
    if (atomicAdd(cnt_w, 1u) + 1u == 2u * need) *cnt_w = 0u;
  }
}

// Barrier setup, the block's partition and tensor-memory allocation, common to
// both kernels. Returns false (before any allocation) when the CTA has no work
// or the indptrs are invalid.
template <class LL>
__device__ __forceinline__ bool cta_begin(const Stage1Params& p, Ctx<LL>& cx, uint8_t* smem_raw, int alloc_warp,
                                          PieceCursor& cur) {
  const uint32_t raw = smem_addr(smem_raw);
  cx.s = (raw + 1023u) & ~1023u;
  cx.g = smem_raw + (cx.s - raw);
  cx.abort_word = reinterpret_cast<volatile uint32_t*>(cx.g + LL::kOffAbort);
  cx.flags = p.dev_flags;
  if (threadIdx.x == 0) {
    LL::init_barriers(cx);
    mbar_init(cx.bar(LL::kMerge), 1);
    *cx.abort_word = 0u;
    reinterpret_cast<MergeList*>(cx.g + LL::kOffMList)->n = 0u;
    fence_mbar_init();
  }
  // Launched as a programmatic dependent, the CTA may start while the kernel
  // before it in the stream still runs. Nothing in global memory is touched
  // before that kernel has completed, except with in-call q quantisation:
  // there the kernel before is this call's amax kernel, which writes only the
  // scale, and the q set-up waits for it instead.
  griddep_launch_dependents();
  if (!p.wait_late) griddep_wait();
  const int64_t c = blockIdx.x;
  // with fewer virtual rows than CTAs, the last CTAs get none (no range is empty)
  auto eff_parts = [&](int64_t total) { return total < p.num_splits ? (total > 0 ? total : 1) : p.num_splits; };
  int64_t* sh = reinterpret_cast<int64_t*>(cx.g + LL::kOffScan);
  const SegLocate loc = block_locate<LL::kThreads, 1>(
      p.qo_indptr, p.kv_indptr, p.batch, p.total_q, p.total_kv, p.group,
      [=](int64_t total) { return part_start(c, total, eff_parts(total)); }, 0, sh);
  if (!loc.ok) {
    if (threadIdx.x == 0) atomicOr(p.dev_flags, kFlagBadIndptr);
    return false;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) p.dev_flags[1] = static_cast<uint32_t>(p.total_q);  // counters in use
  zero_empty_tokens<LL::kThreads>(p);
  cx.total = loc.total;
  cx.parts = eff_parts(loc.total);
  if (c >= cx.parts) return false;
  const int64_t x0 = part_start(c, loc.total, cx.parts), x1 = part_start(c + 1, loc.total, cx.parts);
  if (x0 >= x1 || loc.seg < 0) return false;  // uniform across the block
  if ((threadIdx.x >> 5) == alloc_warp) tmem_alloc(cx.s + LL::kOffSlot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *reinterpret_cast<volatile uint32_t*>(cx.g + LL::kOffSlot);
  cur = PieceCursor{p.qo_indptr, p.kv_indptr, p.batch, x0, x1, loc.seg, loc.seg_vs, c};
  cur.group = p.group;
  return true;
}

template <class LL>
__device__ __forceinline__ void cta_end(const Stage1Params& p, const Ctx<LL>& cx, int alloc_warp) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == alloc_warp) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
  if (*cx.abort_word) return;
  if (p.coop_merge)
    merge_coop(p, cx);
  else
    merge_listed(p, cx);
}

// Host: the tensor map of a KV cache of `rows` rows of 576 bytes, boxes of
// 128 bytes x box_rows rows, 128B swizzle (defined in mla_stage1_tc.cu).
cudaError_t make_kv_map(CUtensorMap* map, const void* kv, int64_t rows, uint32_t box_rows);

// Host: a 2-D byte tensor map, `rows` rows of `inner` bytes `pitch` bytes
// apart (pitch a multiple of 16), boxes of box_inner bytes x box_rows rows;
// rows past the end read as zero (defined in mla_stage1_tc.cu).
cudaError_t make_u8_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t pitch,
                        uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

}  // namespace tc
}  // namespace mla
