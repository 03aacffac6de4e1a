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
//        past the end of the cache read as zero. The halves' e8m0 bytes come
//        along as one bulk copy of the 16-byte units around them (a half's
//        1152 bytes need not start on a 16-byte boundary);
//      - two converter threads per tile row (the warps of one tensor-memory
//        lane quarter, 9 blocks each) read the row from the stage (the
//        swizzle makes the reads conflict-free) and write the e5m2 bytes
//        twice: all 576 into tensor memory, where Q.K^T reads its A operand
//        (144 columns a row), and the 512 V dims into a 64 KB shared-memory
//        stage in the 128-byte-swizzled layout that P.V reads as V^T. The K
//        operand therefore never crosses shared memory.
//  * Buffers: two V stages, two K buffers in tensor memory, two S and two P
//    buffers, one O accumulator (2 x 144 + 2 x 32 + 128 = 480 of the 512
//    tensor-memory columns). A tile's stage and K buffer are rewritten once
//    the P.V of the tile two back is done.
//  * Roles: warps 0-7 convert, warps 8-11 run the online softmax (thread =
//    row = tensor-memory lane), warp 12 issues both UMMA kinds from a
//    non-blocking loop (an issue blocks while the tensor pipe's queue is full,
//    so the issuer is neither a converter nor a softmax warp) and owns tensor
//    memory, warp 13 loads the raw tiles. Every mbarrier wait is bounded.
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

constexpr int kThreads = 512;                          // four warpgroups
constexpr int kConvWarps = 8;                          // two per tensor-memory lane quarter, half a row each
constexpr int kSoftWarp0 = 8;                          // warps 8-11 run the softmax
constexpr int kIssuerWarp = 12;                        // warp 13 loads the raw tiles, 14-15 only hold registers
// Registers per thread: the launch gives 128 to every warpgroup; the softmax
// warpgroup takes 232 from the two converting warpgroups (96 each) and the
// issuing and loading warpgroup (88): 96 + 96 + 232 + 88 = 4 x 128, the
// launch budget exactly.
constexpr uint32_t kLaunchRegs = 128, kConvRegs = 96, kSoftRegs = 232, kAuxRegs = 88;
static_assert(2 * kConvRegs + kSoftRegs + kAuxRegs == 4 * kLaunchRegs, "register split must equal the launch budget");
constexpr int kStages = 2;                             // V stages, K buffers, S and P buffers
constexpr int kHalfRows = 64;                          // raw tiles come in halves of 64 rows
constexpr int kRawStages = 3;
constexpr int kRowBytes = kDqk / 2;                    // 288 fp4x2 bytes a row
constexpr int kRowScales = kDqk / kMxBlock;            // 18 e8m0 bytes a row
constexpr int kRawBox = kHalfRows * 128;               // one 128-byte-wide box of 64 rows (8 KB)
constexpr int kRawOffTail = 2 * kRawBox;               // bytes 256-287 of the 64 rows (2 KB)
constexpr int kRawNibBytes = kHalfRows * kRowBytes;    // 18 KB per half, the TMA transaction
constexpr int kRawOffSc = kRawNibBytes;                // the 16-byte units holding the 64 rows' e8m0 bytes
constexpr int kRawStageBytes = 20 * 1024;
static_assert(kRawOffSc + kHalfRows * kRowScales + 30 <= kRawStageBytes && kRawOffSc % 16 == 0, "raw stage");
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
  static constexpr int kOffRexp = kOffP + kStages * kPBytes;             // [4][128] u8: R of each row
  static constexpr int kOffRedMax = kOffRexp + 4 * kTileRows;            // [2][4][16] f32
  static constexpr int kOffRedMu = kOffRedMax + 2 * 4 * 16 * 4;          // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMu + 2 * 4 * 16 * 4;            // [4][16] f32
  static constexpr int kOffAmax = kOffRedL + 4 * 16 * 4;                 // [4] u32
  static constexpr int kOffMList = kOffAmax + 16;                        // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                        // 24 x i64
  static constexpr int kOffMeta = kOffScan + 24 * 8;                     // [4] u32: tile i in slot i % 4
  static constexpr int kOffBars = kOffMeta + 16;
  // kKvFull and the row exponents have four slots (tile i in slot i % 4): the
  // converters run up to two tiles ahead of the softmax, which still reads
  // them, while K buffers and V stages have two (tile i in i % 2)
  enum {
    kKvFull = 0, kSFull = 4, kSEmpty = 6, kPFull = 8, kPvDone = 10, kQFull = 12, kQEmpty = 13, kOFull = 14,
    kOEmpty = 15, kGrp = 16, kRawFull = 18, kRawEmpty = 21, kDrain = 24, kMerge = 25, kVFull = 26, kNumBars = 28
  };
  static constexpr int kMergeBytes = kStages * kVBytes;  // the V stages hold partials for the end-of-CTA merge
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;
  template <class C>
  __device__ static void init_barriers(const C& cx) {
    for (int i = 0; i < 4; ++i) mbar_init(cx.bar(kKvFull + i), kConvWarps);  // K operand in tensor memory
    for (int i = 0; i < kStages; ++i) {
      mbar_init(cx.bar(kVFull + i), kConvWarps);  // V dims of the tile in the V stage
      mbar_init(cx.bar(kSFull + i), 1);
      mbar_init(cx.bar(kSEmpty + i), 4);
      mbar_init(cx.bar(kPFull + i), 4);
      mbar_init(cx.bar(kPvDone + i), 1);
      mbar_init(cx.bar(kGrp + i), 4);
    }
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(cx.bar(kRawFull + i), 1);   // the producer (TMA bytes + scales)
      mbar_init(cx.bar(kRawEmpty + i), 4);  // the 4 converter warps that read that half
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
// Warp 13: the raw halves of each tile into the ring, half j into stage j % 3
// once the converters of half j - 3 have read it.
__device__ void producer_role(const Stage1Params& p, const Cx& cx, const RawMaps* maps, PieceCursor cur, int lane) {
  const uint64_t pol = policy_evict_first();
  if (lane == 0) {
    prefetch_tensormap(&maps->wide);
    prefetch_tensormap(&maps->tail);
  }
  const uint8_t* scales = static_cast<const uint8_t*>(p.kv_scale);  // 16-byte aligned (checked by the host)
  const int64_t sc_end = static_cast<int64_t>(p.total_kv) * kRowScales;
  const int64_t sc_full = sc_end & ~int64_t{15};  // bytes readable in whole 16-byte units
  TileWalker tw;
  tw.init(cur);
  uint32_t j = 0;
  int32_t row0 = 0;
  bool ok = true;
  while (ok && tw.next(row0)) {
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t s = j % kRawStages, rnd = j / kRawStages;
      const int32_t r0 = row0 + hh * kHalfRows;
      // the half's e8m0 bytes [sb, se) come in as the 16-byte units [a, b)
      // around them; bytes of the cache's last partial unit by plain loads
      const int64_t sb = static_cast<int64_t>(r0) * kRowScales;
      const int64_t se = min(sb + kHalfRows * kRowScales, sc_end);
      const int64_t a = sb & ~int64_t{15};
      const int64_t b = min((se + 15) & ~int64_t{15}, sc_full);
      const uint32_t win = b > a ? static_cast<uint32_t>(b - a) : 0u;
      if (rnd >= 1 && !cx.wait(L::kRawEmpty + s, (rnd - 1) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t dst = cx.s + L::kOffRaw + s * kRawStageBytes;
      if (lane == 0) {
        mbar_expect_tx(cx.bar(L::kRawFull + s), kRawNibBytes + win);
        tma_load_2d(dst, &maps->wide, 0, r0, cx.bar(L::kRawFull + s), pol);
        tma_load_2d(dst + kRawBox, &maps->wide, 128, r0, cx.bar(L::kRawFull + s), pol);
        tma_load_2d(dst + kRawOffTail, &maps->tail, 256, r0, cx.bar(L::kRawFull + s), pol);
        if (win) bulk_g2s(dst + kRawOffSc, scales + a, win, cx.bar(L::kRawFull + s), pol);
      }
      uint8_t* scd = cx.g + L::kOffRaw + s * kRawStageBytes + kRawOffSc;
      for (int64_t off = max(b, sb) + 2 * lane; off < se; off += 64)
        *reinterpret_cast<uint16_t*>(scd + (off - a)) = static_cast<uint16_t>(ld_nc_u16(scales + off));
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
// Converters (warps 0-7; two threads per tile row, in its tensor-memory lane).

// Blocks [bl0, bl0 + 9) of row rr of the raw half at `raw` (the row's scale
// bytes start sc0 bytes into the stage's scale window): the rebased e5m2 bytes
// into tensor-memory columns tk + 8 bl. Returns R.
__device__ __forceinline__ uint32_t convert_half_row(const uint8_t* raw, int sc0, int rr, uint32_t tk, int bl0) {
  const uint8_t* sc = raw + kRawOffSc + sc0 + rr * kRowScales;
  uint32_t R = 0;
#pragma unroll
  for (int k = 0; k < 9; ++k) {
    const uint32_t h = *reinterpret_cast<const uint16_t*>(sc + 2 * k);
    R = max(R, max(h & 0xFFu, h >> 8));
  }
  const int swa = rr & 7, swt = (rr >> 2) & 1;
#pragma unroll 1
  for (int bl = bl0; bl < bl0 + 9; ++bl) {  // block bl: fp4x2 bytes 16 bl .. 16 bl + 15
    const uint8_t* src = bl < 16 ? raw + (bl >> 3) * kRawBox + rr * 128 + (((bl & 7) ^ swa) << 4)
                                 : raw + kRawOffTail + rr * 32 + (((bl - 16) ^ swt) << 4);
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    uint4 lo, hi;
    convert_block(v, rebase_scale2(R - sc[bl]), lo, hi);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    tmem_st8(tk + 8 * bl, w);
  }
  return R;
}

// V blocks [bl0, bl1) of tile row `row` (dims 32 bl .. 32 bl + 31), copied from
// the K operand in tensor memory (columns tk + 8 bl) into the V stage: 128-byte
// -swizzled K-major rows, 16 KB per 128 dims. Four blocks per tensor-memory
// wait.
__device__ __forceinline__ void copy_v_blocks(uint32_t tk, uint8_t* vstage, int row, int bl0, int bl1) {
  const int sw = row & 7;
  for (int g = bl0; g < bl1; g += 4) {
    const int n = min(4, bl1 - g);
    uint32_t w[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < n) tmem_ld8(tk + 8 * (g + k), w[k]);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < n) {
        const int bl = g + k, u = 2 * (bl & 3);
        uint8_t* vb = vstage + (bl >> 2) * kChunkBytes + row * 128;
        *reinterpret_cast<uint4*>(vb + ((u ^ sw) << 4)) = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
        *reinterpret_cast<uint4*>(vb + (((u + 1) ^ sw) << 4)) = make_uint4(w[k][4], w[k][5], w[k][6], w[k][7]);
      }
    }
  }
}

// Warps 0-7: warp w converts blocks 9 (w / 4) .. 9 (w / 4) + 8 of tile rows
// 32 (w % 4) .. + 31 (its tensor-memory lane quarter) into tensor memory, and
// once the V stage is free copies the V dims among them into it. The V stage
// is thus held only from that copy to the tile's P.V, not through the
// conversion, Q.K^T and softmax.
__device__ void converter_role(const Cx& cx, PieceCursor cur, int warp, int lane) {
  const uint32_t ntiles = static_cast<uint32_t>(count_tiles(cur));
  volatile uint32_t* meta_slot = reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffMeta);
  MetaTileWalker rw;
  rw.init(cur);
  const int q4 = warp & 3, part = warp >> 2;
  const int row = 32 * q4 + lane, hh = q4 >> 1, rr = 32 * (q4 & 1) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
  for (uint32_t i = 0; i < ntiles; ++i) {
    int32_t row0 = 0;
    uint32_t meta = 0;
    rw.next(row0, meta);
    const uint32_t b = i & 1u;
    const uint32_t tk = cx.tmem + lane_base + kTmK + b * kTmKStride;
    // K buffer b is free once the Q.K^T of tile i - 2 is done (this warp's
    // copy out of it came before, in program order)
    if (i >= 2 && !cx.wait(L::kSFull + b, ((i - 2) >> 1) & 1u)) return;
    const uint32_t j = 2 * i + static_cast<uint32_t>(hh), s = j % kRawStages;
    if (!cx.wait(L::kRawFull + s, (j / kRawStages) & 1u)) return;
    tc_fence_after();
    const int sc0 = static_cast<int>((static_cast<int64_t>(row0 + hh * kHalfRows) * kRowScales) & 15);
    const uint32_t R = convert_half_row(cx.g + L::kOffRaw + s * kRawStageBytes, sc0, rr, tk, 9 * part);
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kRawEmpty + s));
    if (part == 0) cx.g[L::kOffRexp + (i & 3u) * kTileRows + row] = static_cast<uint8_t>(R);
    if (warp == 0 && lane == 0) meta_slot[i & 3u] = meta;
    // the tensor-memory stores, visible to the tensor core
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kKvFull + (i & 3u)));
    // V stage b is free once the P.V of tile i - 2 is done
    if (i >= 2 && !cx.wait(L::kPvDone + b, ((i - 2) >> 1) & 1u)) return;
    tc_fence_after();
    copy_v_blocks(tk, cx.g + L::kOffKv + b * kVBytes, row, part == 0 ? 0 : 9, part == 0 ? 9 : 16);
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kVFull + b));
  }
}

// ---------------------------------------------------------------------------
// Warp 12, lane 0: issues Q.K^T of tile qi and P.V of tile pi as soon as each
// is ready (non-blocking tests, bounded overall), in tile order for each kind.
constexpr uint32_t kIdQK = umma_idesc(128, 32, 1, 0, false, false);  // A e5m2 from tensor memory, B e4m3
constexpr uint32_t kIdPV = umma_idesc(128, 32, 1, 0, true, true);    // A = V^T MN-major, B = P^T MN-major

__device__ __forceinline__ void issue_qk(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint32_t ka = cx.tmem + kTmK + b * kTmKStride, d = cx.tmem + kTmS + 32 * b;
  const uint64_t qb = qk_desc_b(cx.s + L::kOffQ, 0);
#pragma unroll
  for (int ks = 0; ks < kDqk / 32; ++ks)
    umma_e4m3_ta(d, ka + 8 * ks, desc_add(qb, (ks >> 2) * kQChunkBytes + (ks & 3) * 32), kIdQK, ks > 0 ? 1u : 0u);
  umma_commit(cx.bar(L::kSFull + b));
  if (t.last) umma_commit(cx.bar(L::kQEmpty));
}

__device__ __forceinline__ void issue_pv(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint64_t va = pv_desc_a(cx.s + L::kOffKv + b * kVBytes, 0, 0), pb = pv_desc_b(cx.s + L::kOffP + b * kPBytes, 0);
  const uint32_t obuf = cx.tmem + kTmO;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_e4m3(obuf + 32 * mb, desc_add(va, mb * kChunkBytes + ks * 4096), desc_add(pb, ks * 1024), kIdPV,
                (ks > 0 || !t.first) ? 1u : 0u);
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
    if (pi < qi && mbar_test_wait(cx.bar(L::kPFull + (pi & 1u)), (pi >> 1) & 1u) &&
        mbar_test_wait(cx.bar(L::kVFull + (pi & 1u)), (pi >> 1) & 1u)) {
      const TileMeta t = TileMeta::unpack(meta[pi & 3u]);
      // the first P.V of piece k overwrites O: the epilogue of piece k - 1 has read it
      if (!t.first || t.k == 0 || mbar_test_wait(cx.bar(L::kOEmpty), (t.k - 1) & 1u)) {
        issue_pv(cx, pi, t);
        ++pi;
        progressed = true;
      }
    }
    if (qi < n && mbar_test_wait(cx.bar(L::kKvFull + (qi & 3u)), (qi >> 2) & 1u) &&
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
// Softmax (warps 8-11).
template <int QF>
__device__ void softmax_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = warp - kSoftWarp0;
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
      // the converters' row exponents of this tile (already complete: Q.K^T read its K operand)
      if (!cx.wait(L::kKvFull + (i & 3u), (i >> 2) & 1u)) return;
      const int r = row_exp(cx.g[L::kOffRexp + (i & 3u) * kTileRows + sx.row]);
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
        const bool up = tz[h] > mu[h] + kMaxSlack;  // O's reference moves lazily
        alpha[h] = fast_exp2(m[h] - mn);
        alpha_o[h] = up ? fast_exp2(mu[h] - tz[h]) : 1.0f;
        grew |= up;
        m[h] = mn;
        mu[h] = up ? tz[h] : mu[h];
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
  if (warp < kSoftWarp0) {
    setmaxnreg_dec<kConvRegs>();
    converter_role(cx, cur, warp, lane);
  } else if (warp < kIssuerWarp) {
    setmaxnreg_inc<kSoftRegs>();  // granted once warpgroups 0, 1 and 3 have made their decreases (unconditional)
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
  // The softmax warpgroup returned its extra registers before this barrier:
  // the increases below are always granted at once.
  __syncthreads();
  if (warp < kSoftWarp0 || warp >= kIssuerWarp) setmaxnreg_inc<kLaunchRegs>();
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
