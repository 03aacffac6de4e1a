// Stage 1 of split-K MLA decode for an mxfp4 KV cache (OCP MX: e2m1 elements,
// one e8m0 scale per 32 along the head dimension) on the tcgen05 tensor cores.
//
// Method: the same split-K flash decoding partials as the fp8 kernel
// (kernelbot-amd-mixed-mla-753817, `mla_flash_decode_stage1`); the KV row is
// K[d] = e2m1[d] * 2^(scale[d / 32] - 127).
//
// GB300 design:
//  * The MX block scales run along the head dimension. For Q.K^T that is the
//    contraction, but for P.V it is the output (M) dimension, which no
//    block-scaled MMA form can take, so each row is converted once into an
//    8-bit operand that serves both products: every e2m1 element becomes an
//    e5m2 value rebased to the row's largest block exponent R with 13 binades
//    of headroom, e5m2 = e2m1 * 2^(scale - R + 13) (mla_mx_convert.cuh: exact
//    for every block within 28 binades of the row's largest).
//  * The row factor 2^r, r = R - 140, multiplies that row's scores, and enters
//    P.V through the weights: per head, the softmax keeps m = max x (for the
//    denominator l) and mu = max (x + r) (the reference of O), writes
//    P = 2^(x + r - mu) (<= 1, the largest term of O exactly 1), and the
//    epilogue multiplies O by 2^(mu - m) / l.
//  * The data path of a 128-row tile:
//      - the raw fp4x2 bytes come in by TMA, in two halves of 64 rows, each
//        three boxes (bytes 0-127 and 128-255 with 128-byte swizzle, bytes
//        256-287 with 32-byte swizzle) into a ring of three 20 KB stages; rows
//        past the end of the cache read as zero. The lanes of the producer
//        warp load the halves' e8m0 bytes with plain loads into the same stage
//        (a row's 18 bytes are not 16-byte aligned);
//      - a converter thread per tile row (= tensor-memory lane) reads its row
//        from the stage (the swizzle makes the reads conflict-free) and writes
//        the e5m2 bytes twice: all 576 into tensor memory, where Q.K^T reads
//        its A operand (144 columns a row), and the 512 V dims into a 64 KB
//        shared-memory stage in the 128-byte-swizzled layout that P.V reads as
//        V^T. The K operand therefore never crosses shared memory.
//  * Buffers: two V stages, two K buffers in tensor memory, two S and two P
//    buffers, one O accumulator (2 x 144 + 2 x 32 + 128 = 480 of the 512
//    tensor-memory columns). A tile's stage and K buffer are rewritten once
//    the P.V of the tile two back is done.
//  * Roles: warps 0-3 convert, warps 4-7 run the online softmax (thread =
//    row = tensor-memory lane), warp 8 issues both UMMA kinds from a
//    non-blocking loop (an issue blocks while the tensor pipe's queue is full,
//    so the issuer is neither a converter nor a softmax warp) and owns tensor
//    memory, warp 9 loads the raw tiles. Every mbarrier wait is bounded.
//  * Registers: setmaxnreg moves registers from the converting and the
//    issuing warpgroups to the softmax warpgroup at the start. At the end the
//    softmax warpgroup gives them back before a CTA barrier, and only after
//    that barrier do the other two ask for theirs again, so no increase ever
//    waits on registers that a warp waiting at a barrier holds.
#include "mla_mx_convert.cuh"
#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace mx {

using mxcvt::convert_block;
using mxcvt::exp2i;
using mxcvt::rebase_scale2;
using mxcvt::row_exp;

constexpr int kThreads = 384;                          // three warpgroups
constexpr int kIssuerWarp = 8;                         // warp 9 loads the raw tiles, warps 10-11 only hold registers
// Registers per thread: the launch gives 168 to every warpgroup; the softmax
// warpgroup takes 232 from the converters (160) and the issuing and loading
// warpgroup (112): 160 + 232 + 112 = 3 x 168, the launch budget exactly.
constexpr uint32_t kLaunchRegs = 168, kConvRegs = 160, kSoftRegs = 232, kAuxRegs = 112;
static_assert(kConvRegs + kSoftRegs + kAuxRegs == 3 * kLaunchRegs, "register split must equal the launch budget");
constexpr int kStages = 2;                             // V stages, K buffers, S and P buffers
constexpr int kHalfRows = 64;                          // raw tiles come in halves of 64 rows
constexpr int kRawStages = 3;
constexpr int kRowBytes = kDqk / 2;                    // 288 fp4x2 bytes a row
constexpr int kRowScales = kDqk / kMxBlock;            // 18 e8m0 bytes a row
constexpr int kRawBox = kHalfRows * 128;               // one 128-byte-wide box of 64 rows (8 KB)
constexpr int kRawOffTail = 2 * kRawBox;               // bytes 256-287 of the 64 rows (2 KB)
constexpr int kRawNibBytes = kHalfRows * kRowBytes;    // 18 KB per half, the TMA transaction
constexpr int kRawOffSc = kRawNibBytes;                // [64 rows][18] e8m0 bytes
constexpr int kRawStageBytes = 20 * 1024;
static_assert(kRawOffSc + kHalfRows * kRowScales <= kRawStageBytes, "raw stage");
// tensor-memory columns
constexpr uint32_t kTmS = 0;          // S: 2 buffers x 32
constexpr uint32_t kTmK = 64;         // K operand buffer b at kTmK + kTmKStride b, 144 columns
constexpr uint32_t kTmKStride = 160;
constexpr uint32_t kTmO = 384;        // O^T: 4 blocks x 32 columns
static_assert(kTmK + kTmKStride + kDqk / 4 <= kTmO && kTmO + 128 <= kTmemCols, "tensor memory");

struct L {
  static constexpr int kThreads = mx::kThreads;
  static constexpr int kOffKv = 0;                                       // V stages
  static constexpr int kOffRaw = kOffKv + kStages * kVBytes;             // raw halves
  static constexpr int kOffQ = kOffRaw + kRawStages * kRawStageBytes;
  static constexpr int kOffP = kOffQ + kQBytes;                          // 2 x 4 KB
  static constexpr int kOffRexp = kOffP + kStages * kPBytes;             // [2][128] u8: R of each row
  static constexpr int kOffRedMax = kOffRexp + kStages * kTileRows;      // [2][4][16] f32
  static constexpr int kOffRedMu = kOffRedMax + 2 * 4 * 16 * 4;          // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMu + 2 * 4 * 16 * 4;            // [4][16] f32
  static constexpr int kOffAmax = kOffRedL + 4 * 16 * 4;                 // [4] u32
  static constexpr int kOffMList = kOffAmax + 16;                        // MergeList (64 B)
  static constexpr int kOffScan = kOffMList + 64;                        // 16 x i64
  static constexpr int kOffMeta = kOffScan + 16 * 8;                     // [4] u32: tile i in slot i % 4
  static constexpr int kOffBars = kOffMeta + 16;
  enum {
    kKvFull = 0, kSFull = 2, kSEmpty = 4, kPFull = 6, kPvDone = 8, kQFull = 10, kQEmpty = 11, kOFull = 12,
    kOEmpty = 13, kGrp = 14, kRawFull = 16, kRawEmpty = 19, kDrain = 22, kMerge = 23, kNumBars = 24
  };
  static constexpr int kMergeBytes = kStages * kVBytes;  // the V stages hold partials for the end-of-CTA merge
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;
  template <class C>
  __device__ static void init_barriers(const C& cx) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(cx.bar(kKvFull + i), 4);  // the 4 converter warps
      mbar_init(cx.bar(kSFull + i), 1);
      mbar_init(cx.bar(kSEmpty + i), 4);
      mbar_init(cx.bar(kPFull + i), 4);
      mbar_init(cx.bar(kPvDone + i), 1);
      mbar_init(cx.bar(kGrp + i), 4);
    }
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(cx.bar(kRawFull + i), 1);   // the producer (TMA bytes + scales)
      mbar_init(cx.bar(kRawEmpty + i), 2);  // the 2 converter warps of that half
    }
    mbar_init(cx.bar(kQFull), 4);
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kOFull), 1);
    mbar_init(cx.bar(kOEmpty), 4);
    mbar_init(cx.bar(kDrain), 1);
  }
};
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffRaw % 1024 == 0 && kRawStageBytes % 1024 == 0 && L::kOffQ % 1024 == 0 &&
                  L::kOffP % 1024 == 0,
              "operand and swizzle alignment");
static_assert(L::kOffBars % 8 == 0, "barrier alignment");
using Cx = Ctx<L>;

// The two tensor maps over the fp4x2 rows [total_kv][288]: 128-byte boxes of
// 64 rows with 128-byte swizzle (bytes 0-127, 128-255) and 32-byte boxes with
// 32-byte swizzle (bytes 256-287).
struct RawMaps {
  CUtensorMap wide, tail;
};

__device__ __forceinline__ uint32_t ld_nc_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Warp 9: the raw halves of each tile into the ring, half j into stage j % 3
// once the converters of half j - 3 have read it.
__device__ void producer_role(const Stage1Params& p, const Cx& cx, const RawMaps* maps, PieceCursor cur, int lane) {
  const uint64_t pol = policy_evict_first();
  if (lane == 0) {
    prefetch_tensormap(&maps->wide);
    prefetch_tensormap(&maps->tail);
  }
  const uint8_t* scales = static_cast<const uint8_t*>(p.kv_scale);
  const int64_t sc_end = static_cast<int64_t>(p.total_kv) * kRowScales;
  TileWalker tw;
  tw.init(cur);
  uint32_t j = 0;
  int32_t row0 = 0;
  bool ok = true;
  while (ok && tw.next(row0)) {
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t s = j % kRawStages, rnd = j / kRawStages;
      const int32_t r0 = row0 + hh * kHalfRows;
      // the half's 64 x 18 e8m0 bytes as 16-bit words, 18 per lane (rows past
      // the end of the cache read as zero), loaded before the stage is free
      uint32_t w[18];
      const int64_t sb = static_cast<int64_t>(r0) * kRowScales;
#pragma unroll
      for (int k = 0; k < 18; ++k) {
        const int64_t off = sb + 2 * (32 * k + lane);
        w[k] = off + 2 <= sc_end ? ld_nc_u16(scales + off) : 0u;
      }
      if (rnd >= 1 && !cx.wait(L::kRawEmpty + s, (rnd - 1) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t dst = cx.s + L::kOffRaw + s * kRawStageBytes;
      if (lane == 0) {
        mbar_expect_tx(cx.bar(L::kRawFull + s), kRawNibBytes);
        tma_load_2d(dst, &maps->wide, 0, r0, cx.bar(L::kRawFull + s), pol);
        tma_load_2d(dst + kRawBox, &maps->wide, 128, r0, cx.bar(L::kRawFull + s), pol);
        tma_load_2d(dst + kRawOffTail, &maps->tail, 256, r0, cx.bar(L::kRawFull + s), pol);
      }
      uint8_t* scd = cx.g + L::kOffRaw + s * kRawStageBytes + kRawOffSc;
#pragma unroll
      for (int k = 0; k < 18; ++k) *reinterpret_cast<uint16_t*>(scd + 2 * (32 * k + lane)) = static_cast<uint16_t>(w[k]);
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kRawFull + s));
      ++j;
    }
  }
  // the last TMA issued on each raw stage must have landed before the CTA exits
  for (uint32_t s = 0; s < kRawStages && s < j; ++s) {
    const uint32_t last = ((j - 1 - s) / kRawStages) * kRawStages + s;
    mbar_wait_drain_tc(cx.bar(L::kRawFull + s), (last / kRawStages) & 1u);
  }
}

// ---------------------------------------------------------------------------
// Converters (warps 0-3; thread = tile row = tensor-memory lane).

// Row rr of the raw half at `raw` (tile row `row`): the rebased e5m2 bytes
// into tensor-memory columns tk.. (all 576) and into the V stage (dims 0-511,
// 128-byte-swizzled K-major rows); records R.
__device__ __forceinline__ void convert_row(const uint8_t* raw, int rr, uint8_t* vstage, int row, uint32_t tk,
                                            uint8_t* rexp) {
  const uint8_t* sc = raw + kRawOffSc + rr * kRowScales;
  uint32_t scw[9];
  uint32_t R = 0;
#pragma unroll
  for (int k = 0; k < 9; ++k) {
    scw[k] = *reinterpret_cast<const uint16_t*>(sc + 2 * k);
    R = max(R, max(scw[k] & 0xFFu, scw[k] >> 8));
  }
  const int sw = row & 7, swa = rr & 7, swt = (rr >> 2) & 1;
#pragma unroll 1
  for (int bp = 0; bp < 9; ++bp) {  // blocks 2 bp, 2 bp + 1: bytes 32 bp .. 32 bp + 31
    uint4 v0, v1;
    if (bp < 8) {
      const uint8_t* rb = raw + (bp >> 2) * kRawBox + rr * 128;
      const int u0 = 2 * (bp & 3);
      v0 = *reinterpret_cast<const uint4*>(rb + ((u0 ^ swa) << 4));
      v1 = *reinterpret_cast<const uint4*>(rb + (((u0 + 1) ^ swa) << 4));
    } else {
      const uint8_t* rb = raw + kRawOffTail + rr * 32;
      v0 = *reinterpret_cast<const uint4*>(rb + (swt << 4));
      v1 = *reinterpret_cast<const uint4*>(rb + ((swt ^ 1) << 4));
    }
    const uint32_t s2 = bp < 8 ? scw[bp] : scw[8];
    uint4 a0, a1, b0, b1;
    convert_block(v0, rebase_scale2(R - (s2 & 0xFFu)), a0, a1);
    convert_block(v1, rebase_scale2(R - (s2 >> 8)), b0, b1);
    if (bp < 8) {  // V dims 64 bp .. 64 bp + 63: chunk bp / 2, 16-byte units 4 (bp % 2) ..
      uint8_t* vb = vstage + (bp >> 1) * kChunkBytes + row * 128;
      const int u = 4 * (bp & 1);
      *reinterpret_cast<uint4*>(vb + ((u ^ sw) << 4)) = a0;
      *reinterpret_cast<uint4*>(vb + (((u + 1) ^ sw) << 4)) = a1;
      *reinterpret_cast<uint4*>(vb + (((u + 2) ^ sw) << 4)) = b0;
      *reinterpret_cast<uint4*>(vb + (((u + 3) ^ sw) << 4)) = b1;
    }
    const uint32_t w[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                            b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    tmem_st16(tk + 16 * bp, w);
  }
  rexp[row] = static_cast<uint8_t>(R);
}

__device__ void converter_role(const Cx& cx, PieceCursor cur, int warp, int lane) {
  const uint32_t ntiles = static_cast<uint32_t>(count_tiles(cur));
  volatile uint32_t* meta_slot = reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffMeta);
  MetaTileWalker rw;
  rw.init(cur);
  const int row = 32 * warp + lane, hh = warp >> 1, rr = 32 * (warp & 1) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
  for (uint32_t i = 0; i < ntiles; ++i) {
    int32_t row0 = 0;
    uint32_t meta = 0;
    rw.next(row0, meta);
    const uint32_t b = i & 1u;
    // stage b and K buffer b are free once the P.V of tile i - 2 is done
    if (i >= 2 && !cx.wait(L::kPvDone + b, ((i - 2) >> 1) & 1u)) return;
    const uint32_t j = 2 * i + static_cast<uint32_t>(hh), s = j % kRawStages;
    if (!cx.wait(L::kRawFull + s, (j / kRawStages) & 1u)) return;
    tc_fence_after();
    convert_row(cx.g + L::kOffRaw + s * kRawStageBytes, rr, cx.g + L::kOffKv + b * kVBytes, row,
                cx.tmem + lane_base + kTmK + b * kTmKStride, cx.g + L::kOffRexp + b * kTileRows);
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kRawEmpty + s));
    if (warp == 0 && lane == 0) meta_slot[i & 3u] = meta;
    // the stage's shared-memory bytes and the tensor-memory stores, visible to the tensor core
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kKvFull + b));
  }
}

// ---------------------------------------------------------------------------
// Warp 8, lane 0: issues Q.K^T of tile qi and P.V of tile pi as soon as each
// is ready (non-blocking tests, bounded overall), in tile order for each kind.
constexpr uint32_t kIdQK = umma_idesc(128, 32, 1, 0, false, false);  // A e5m2 from tensor memory, B e4m3
constexpr uint32_t kIdPV = umma_idesc(128, 32, 1, 0, true, true);    // A = V^T MN-major, B = P^T MN-major

__device__ __forceinline__ void issue_qk(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint32_t qbuf = cx.s + L::kOffQ, ka = cx.tmem + kTmK + b * kTmKStride;
  const uint32_t d = cx.tmem + kTmS + 32 * b;
#pragma unroll
  for (int ks = 0; ks < kDqk / 32; ++ks) umma_e4m3_ta(d, ka + 8 * ks, qk_desc_b(qbuf, ks), kIdQK, ks > 0 ? 1u : 0u);
  umma_commit(cx.bar(L::kSFull + b));
  if (t.last) umma_commit(cx.bar(L::kQEmpty));
}

__device__ __forceinline__ void issue_pv(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + b * kVBytes, pbuf = cx.s + L::kOffP + b * kPBytes;
  const uint32_t obuf = cx.tmem + kTmO;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_e4m3(obuf + 32 * mb, pv_desc_a(stage, mb, ks), pv_desc_b(pbuf, ks), kIdPV, (ks > 0 || !t.first) ? 1u : 0u);
  umma_commit(cx.bar(L::kPvDone + b));
  if (t.last) umma_commit(cx.bar(L::kOFull));
}

__device__ void issuer_role(const Cx& cx, PieceCursor cur) {
  const uint32_t n = static_cast<uint32_t>(count_tiles(cur));
  const volatile uint32_t* meta = reinterpret_cast<const volatile uint32_t*>(cx.g + L::kOffMeta);
  uint32_t qi = 0, pi = 0;
  long long t0 = clock64();
  while (pi < n) {
    bool progressed = false;
    if (pi < qi && mbar_test_wait(cx.bar(L::kPFull + (pi & 1u)), (pi >> 1) & 1u)) {
      const TileMeta t = TileMeta::unpack(meta[pi & 3u]);
      // the first P.V of piece k overwrites O: the epilogue of piece k - 1 has read it
      if (!t.first || t.k == 0 || mbar_test_wait(cx.bar(L::kOEmpty), (t.k - 1) & 1u)) {
        issue_pv(cx, pi, t);
        ++pi;
        progressed = true;
      }
    }
    if (qi < n && mbar_test_wait(cx.bar(L::kKvFull + (qi & 1u)), (qi >> 1) & 1u) &&
        (qi < 2 || mbar_test_wait(cx.bar(L::kSEmpty + (qi & 1u)), ((qi - 2) >> 1) & 1u))) {
      const TileMeta t = TileMeta::unpack(meta[qi & 3u]);
      if (!t.first || mbar_test_wait(cx.bar(L::kQFull), t.k & 1u)) {
        issue_qk(cx, qi, t);
        ++qi;
        progressed = true;
      }
    }
    if (progressed) {
      t0 = clock64();
    } else if (*cx.abort_word) {
      break;
    } else if (clock64() - t0 > kWaitLimitCycles) {
      *cx.abort_word = 1u;
      atomicOr(cx.flags, kFlagTimeout);
      break;
    }
  }
  // every issued tcgen05 operation completes before tensor memory is freed
  umma_commit(cx.bar(L::kDrain));
  mbar_wait_drain_tc(cx.bar(L::kDrain), 0);
}

// ---------------------------------------------------------------------------
// Softmax (warps 4-7).
template <int QF>
__device__ void softmax_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = warp - 4;
  sx.row = 32 * (warp & 3) + lane;
  sx.lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  sx.gcount = 0;
  float* red_max = reinterpret_cast<float*>(cx.g + L::kOffRedMax);
  float* red_mu = reinterpret_cast<float*>(cx.g + L::kOffRedMu);
  float* red_l = reinterpret_cast<float*>(cx.g + L::kOffRedL);
  PieceCursor ahead = cur;
  Piece pc, nxt;
  bool have = ahead.next(pc);
  if (!have) return;
  float c = setup_q<L, QF>(p, cx, sx, pc.token, 0, 1.0f);
  if (c < 0.f) return;
  uint32_t i = 0, k = 0;
  while (have) {
    const bool have_next = ahead.next(nxt);
    float m[16], mu[16], l[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      m[h] = -INFINITY;
      mu[h] = -INFINITY;
      l[h] = 0.f;
    }
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const int nr = min(kTileRows, pc.nrows - r0);
      const uint32_t b = i & 1u;
      const bool valid = sx.row < nr;
      if (!cx.wait(L::kSFull + b, (i >> 1) & 1u)) return;
      // the converters' row exponents of this stage (already complete: Q.K^T read the stage)
      if (!cx.wait(L::kKvFull + b, (i >> 1) & 1u)) return;
      const int r = row_exp(cx.g[L::kOffRexp + b * kTileRows + sx.row]);
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(cx.tmem + sx.lane_base + kTmS + 32 * b, sr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + b));
      const float cr = c * exp2i(r), rf = static_cast<float>(r);
      float x[16], z[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float v = (__uint_as_float(sr[h]) + __uint_as_float(sr[16 + h]) * (1.0f / kLoScale)) * cr;
        x[h] = valid ? v : -INFINITY;
        z[h] = x[h] + rf;
      }
      float* rm = red_max + b * 64;
      float* rz = red_mu + b * 64;
      {
        float wm[16], wz[16];
        warp_max16(x, wm);
        warp_max16(z, wz);
        store16(rm + sx.wi * 16, wm, lane);
        store16(rz + sx.wi * 16, wz, lane);
      }
      if (!group_sync(cx, sx)) return;
      bool grew = false;
      float alpha[16], alpha_o[16], tm[16], tz[16];
      {
        const float4* rm4 = reinterpret_cast<const float4*>(rm);  // [4 warps][16 heads]
        const float4* rz4 = reinterpret_cast<const float4*>(rz);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 a = rm4[q], b4 = rm4[4 + q], c4 = rm4[8 + q], d = rm4[12 + q];
          tm[4 * q] = fmaxf(fmaxf(a.x, b4.x), fmaxf(c4.x, d.x));
          tm[4 * q + 1] = fmaxf(fmaxf(a.y, b4.y), fmaxf(c4.y, d.y));
          tm[4 * q + 2] = fmaxf(fmaxf(a.z, b4.z), fmaxf(c4.z, d.z));
          tm[4 * q + 3] = fmaxf(fmaxf(a.w, b4.w), fmaxf(c4.w, d.w));
          const float4 e = rz4[q], f4 = rz4[4 + q], g4 = rz4[8 + q], k4 = rz4[12 + q];
          tz[4 * q] = fmaxf(fmaxf(e.x, f4.x), fmaxf(g4.x, k4.x));
          tz[4 * q + 1] = fmaxf(fmaxf(e.y, f4.y), fmaxf(g4.y, k4.y));
          tz[4 * q + 2] = fmaxf(fmaxf(e.z, f4.z), fmaxf(g4.z, k4.z));
          tz[4 * q + 3] = fmaxf(fmaxf(e.w, f4.w), fmaxf(g4.w, k4.w));
        }
      }
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float mn = fmaxf(m[h], tm[h]);
        const float un = fmaxf(mu[h], tz[h]);
        alpha[h] = fast_exp2(m[h] - mn);
        alpha_o[h] = fast_exp2(mu[h] - un);
        grew |= un > mu[h];
        m[h] = mn;
        mu[h] = un;
      }
      float pv[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) pv[h] = fast_exp2(z[h] - mu[h]) * kPScale;
      // P buffer b is free once the P.V of tile i - 2 is done
      if (i >= 2 && !cx.wait(L::kPvDone + b, ((i - 2) >> 1) & 1u)) return;
      put_p_row(cx.g + L::kOffP + b * kPBytes, sx.row, pv);
      if (grew && r0 > 0) {
        // O holds this piece up to tile i - 1: wait for that P.V, then rescale
        if (!cx.wait(L::kPvDone + (b ^ 1u), ((i - 1) >> 1) & 1u)) return;
        tc_fence_after();
        rescale_o(cx.tmem + sx.lane_base + kTmO, alpha_o);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull + b));
      // the row sums, off the P handoff
#pragma unroll
      for (int h = 0; h < 16; ++h) l[h] = l[h] * alpha[h] + fast_exp2(x[h] - m[h]);
      ++i;
    }
    // the next piece's q goes in while this piece's last P.V runs
    float c_next = c;
    if (have_next) {
      c_next = setup_q<L, QF>(p, cx, sx, nxt.token, k + 1, 1.0f);
      if (c_next < 0.f) return;
    }
    const float wl = warp_reduce16<false>(l, lane);
    if ((lane & 1) == 0) red_l[sx.wi * 16 + (lane >> 1)] = wl;
    if (!group_sync(cx, sx)) return;
    float f[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const float L = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
      f[h] = fast_exp2(mu[h] - m[h]) / (kPScale * L);
      if (!pc.direct && sx.row == h) p.part_lse[pc.slot * kHeads + h] = m[h] + fast_log2(L);
    }
    if (!cx.wait(L::kOFull, k & 1u)) return;
    tc_fence_after();
    store_o(p, pc, cx.tmem + sx.lane_base + kTmO, sx.row, f);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty));
    if (!pc.direct && !finish_partial(p, cx, sx, pc)) return;
    pc = nxt;
    have = have_next;
    c = c_next;
    ++k;
  }
}

template <int QF>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_mx_kernel(const Stage1Params p, const __grid_constant__ RawMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  Cx cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, kIssuerWarp, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < 4) {
    setmaxnreg_dec<kConvRegs>();
    converter_role(cx, cur, warp, lane);
  } else if (warp < 8) {
    setmaxnreg_inc<kSoftRegs>();  // granted once warpgroups 0 and 2 have made their decreases (unconditional)
    softmax_role<QF>(p, cx, cur, warp, lane);
    setmaxnreg_dec<kLaunchRegs>();
  } else {
    setmaxnreg_dec<kAuxRegs>();
    if (warp == kIssuerWarp) {
      if (lane == 0) issuer_role(cx, cur);
      __syncwarp();
    } else if (warp == kIssuerWarp + 1) {
      producer_role(p, cx, &maps, cur, lane);
    }
  }
  // Warpgroup 1 returned its extra registers before this barrier: the
  // increases below are always granted at once.
  __syncthreads();
  if (warp < 4 || warp >= 8) setmaxnreg_inc<kLaunchRegs>();
  cta_end(p, cx, kIssuerWarp);
}

template <int QF>
static cudaError_t launch_q(const Stage1Params& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    // the warpgroup register split adds up to the launch budget only at 168
    // registers per thread; with any other count the kernel is not launched
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, stage1_mx_kernel<QF>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(stage1_mx_kernel<QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  RawMaps maps;
  e = make_u8_map(&maps.wide, p.kv, kRowBytes, p.total_kv, kRowBytes, 128, kHalfRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_u8_map(&maps.tail, p.kv, kRowBytes, p.total_kv, kRowBytes, 32, kHalfRows, CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  return launch_dependent(stage1_mx_kernel<QF>, p.num_splits, kThreads, L::kAlloc, stream, p, maps);
}

}  // namespace mx
}  // namespace tc

cudaError_t launch_stage1_tc_mxfp4(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  return q_fmt == kQBf16 ? tc::mx::launch_q<kQBf16>(p, stream) : tc::mx::launch_q<kQFp8>(p, stream);
}

}  // namespace mla
