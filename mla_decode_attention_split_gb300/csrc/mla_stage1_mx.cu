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
//    e5m2 value rebased to the row's largest block exponent R,
//    e5m2 = e2m1 * 2^(scale - R). That is exact while scale >= R - 15 (e5m2
//    reaches down to 2^-16 with subnormals); blocks more than 15 binades below
//    the row's largest are flushed to zero: their elements are at most
//    6 * 2^(R - 143), under 2^-15 of the largest block's range.
//  * The row factor 2^r, r = R - 127, multiplies that row's scores, and enters
//    P.V through the weights: per head, the softmax keeps m = max x (for the
//    denominator l) and mu = max (x + r) (the reference of O), writes
//    P = 2^(x + r - mu) (<= 1, the largest term of O exactly 1), and the
//    epilogue multiplies O by 2^(mu - m) / l.
//  * Conversion is per tile row (one thread per row) from registers loaded
//    two tiles ahead into one of two 72 KB stages (V dims in the 128B-swizzled
//    K-major layout of a TMA box, rope dims in the no-swizzle rope layout).
//    With two stages, a stage is rewritten only once the P.V of the tile two
//    back is done, so tiles move in pairs: the converters fill both stages,
//    the tensor pipe runs Q.K^T of both tiles, then P.V of both, while the
//    softmax of the first tile overlaps the second Q.K^T and the next pair's
//    conversion overlaps the P.V.
//  * Warps 0-3 convert (warp 0, lane 0 also issues the UMMAs and owns tensor
//    memory), warps 4-7 run the online softmax (thread = row = TMEM lane).
//    Every mbarrier wait is bounded.
#include "mla_mx_convert.cuh"
#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace mx {

using mxcvt::convert_block;
using mxcvt::exp2i;
using mxcvt::rebase_scale2;

constexpr int kThreads = 384;  // warpgroup 0 converts, 1 runs the softmax, 2 issues the UMMAs (warp 8)
// Registers per thread: launched at 168 (384 threads), then the issuing
// warpgroup gives up 112 so the converting and softmax warpgroups get 224
// (128 x (224 + 224 + 56) = 384 x 168: the split uses exactly the launch budget).
constexpr uint32_t kLaunchRegs = 168, kWorkRegs = 224, kIssueRegs = 56;
static_assert(kWorkRegs * 2 + kIssueRegs == 3 * kLaunchRegs, "register split must equal the launch budget");
constexpr int kStages = 2;
constexpr int kStageBytes = kVBytes + kRopeBytes;  // 72 KB: V dims + rope dims (e5m2)

struct L {
  static constexpr int kThreads = mx::kThreads;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + kQBytes;                      // 2 x 4 KB
  static constexpr int kOffRexp = kOffP + 2 * kPBytes;               // [2][128] u8: R of each row
  static constexpr int kOffRedMax = kOffRexp + 2 * kTileRows;        // [2][4][16] f32
  static constexpr int kOffRedMu = kOffRedMax + 2 * 4 * 16 * 4;      // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMu + 2 * 4 * 16 * 4;        // [4][16] f32
  static constexpr int kOffAmax = kOffRedL + 4 * 16 * 4;             // [4] u32
  static constexpr int kOffMList = kOffAmax + 16;                    // MergeList (64 B)
  static constexpr int kOffScan = kOffMList + 64;                    // 16 x i64
  static constexpr int kOffMeta = kOffScan + 16 * 8;                 // [4] u32: bookkeeping of tile i in slot i % 4
  static constexpr int kOffRaw = kOffMeta + 16;                  // [4 warps][32 rows][288 B] fp4x2
  static constexpr int kOffRawSc = kOffRaw + 4 * 32 * (kDqk / 2);    // [4 warps][32 rows][18 B] e8m0
  static constexpr int kOffBars = kOffRawSc + 4 * 32 * (kDqk / kMxBlock);
  enum {
    kKvFull = 0, kSFull = 2, kSEmpty = 4, kPFull = 6, kPvDone = 8, kQFull = 10, kQEmpty = 11, kOFull = 12,
    kOEmpty = 14, kGrp = 16, kDrain = 18, kMerge = 19, kNumBars = 20
  };
  static constexpr int kMergeBytes = kStages * kStageBytes;  // the stages hold partials for the end-of-CTA merge
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;
  template <class C>
  __device__ static void init_barriers(const C& cx) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(kKvFull + i), 4);  // the 4 converter warps
      mbar_init(cx.bar(kSFull + i), 1);
      mbar_init(cx.bar(kSEmpty + i), 4);
      mbar_init(cx.bar(kPFull + i), 4);
      mbar_init(cx.bar(kPvDone + i), 1);
      mbar_init(cx.bar(kOFull + i), 1);
      mbar_init(cx.bar(kOEmpty + i), 4);
      mbar_init(cx.bar(kGrp + i), 4);
    }
    mbar_init(cx.bar(kQFull), 4);
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kDrain), 1);
  }
};
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(kStageBytes % 1024 == 0 && L::kOffQ % 1024 == 0 && L::kOffP % 1024 == 0, "operand alignment");
static_assert(L::kOffRaw % 16 == 0 && L::kOffBars % 8 == 0, "staging alignment");
using Cx = Ctx<L>;

// ---------------------------------------------------------------------------
// Converters (warps 0-3; thread = tile row).

// The raw rows of one warp's 32 tile rows, loaded coalesced: lane l holds
// 16-byte unit 32 j + l of the warp's 32 x 288 contiguous fp4x2 bytes and
// 2-byte word 32 k + l of its 32 x 18 scale bytes.
struct MxRaw {
  uint4 nib[18];
  uint32_t sc[9];
};

// Global loads that stay where they are written (issued two tiles ahead of
// their use; the compiler may not sink them next to the use).
__device__ __forceinline__ uint4 ld_pinned_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_pinned_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Loads the warp's rows of the next tile (rows past the end of the cache or of
// the CTA's tiles read as zero).
__device__ __forceinline__ void load_mx_raw(const Stage1Params& p, MetaTileWalker& rw, int warp, int lane, MxRaw& r,
                                            uint32_t& meta) {
  int32_t row0 = 0;
  meta = 0;
  const bool have = rw.next(row0, meta);
  const int64_t gb = static_cast<int64_t>(row0) + 32 * warp;
  const uint8_t* kvb = static_cast<const uint8_t*>(p.kv) + gb * (kDqk / 2) + 16 * lane;
  const uint8_t* scb = static_cast<const uint8_t*>(p.kv_scale) + gb * (kDqk / kMxBlock) + 2 * lane;
  if (have && gb + 32 <= p.total_kv) {
#pragma unroll
    for (int j = 0; j < 18; ++j) r.nib[j] = ld_pinned_v4(kvb + 512 * j);
#pragma unroll
    for (int k = 0; k < 9; ++k) r.sc[k] = ld_pinned_u16(scb + 64 * k);
  } else if (have && gb < p.total_kv) {
    // the warp's rows straddle the end of the cache: unit u belongs to row u / 18
    const int nvalid = static_cast<int>(p.total_kv - gb);
#pragma unroll
    for (int j = 0; j < 18; ++j)
      r.nib[j] = (32 * j + lane) / 18 < nvalid ? ld_pinned_v4(kvb + 512 * j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 9; ++k) r.sc[k] = (64 * k + 2 * lane) / 18 < nvalid ? ld_pinned_u16(scb + 64 * k) : 0u;
  } else {
#pragma unroll
    for (int j = 0; j < 18; ++j) r.nib[j] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 9; ++k) r.sc[k] = 0u;
  }
}

// Registers -> the warp's staging area, in memory order (conflict-free).
__device__ __forceinline__ void dump_raw(uint8_t* raw_w, uint8_t* sc_w, int lane, const MxRaw& r) {
#pragma unroll
  for (int j = 0; j < 18; ++j) *reinterpret_cast<uint4*>(raw_w + 16 * (32 * j + lane)) = r.nib[j];
#pragma unroll
  for (int k = 0; k < 9; ++k) *reinterpret_cast<uint16_t*>(sc_w + 2 * (32 * k + lane)) = static_cast<uint16_t>(r.sc[k]);
}

// Converts this thread's row (tile row tr, staged at srow / ssc) into the
// stage: V dims into the 128B-swizzled chunks, rope dims into the no-swizzle
// rope part; records R.
__device__ __forceinline__ void convert_row(uint8_t* stage, uint8_t* rexp, int tr, const uint8_t* srow,
                                            const uint8_t* ssc) {
  uint32_t R = 0;
#pragma unroll
  for (int k = 0; k < 9; ++k) {
    const uint32_t h = *reinterpret_cast<const uint16_t*>(ssc + 2 * k);
    R = max(R, max(h & 0xFFu, h >> 8));
  }
  const int sw = tr & 7;
  uint8_t* vrow = stage + tr * 128;
#pragma unroll 1
  for (int b = 0; b < 16; b += 2) {  // blocks b, b + 1 of V chunk b / 4
    const uint32_t sc = *reinterpret_cast<const uint16_t*>(ssc + b);
    const uint4 v0 = *reinterpret_cast<const uint4*>(srow + 16 * b);
    const uint4 v1 = *reinterpret_cast<const uint4*>(srow + 16 * (b + 1));
    uint8_t* rb = vrow + (b >> 2) * kChunkBytes;
    const int u0 = 2 * (b & 3);  // elements 32(b%4).. of the chunk: 16-byte units u0 .. u0+3, swizzled by row
    uint4 lo, hi;
    convert_block(v0, rebase_scale2(R - (sc & 0xFFu)), lo, hi);
    *reinterpret_cast<uint4*>(rb + ((u0 ^ sw) << 4)) = lo;
    *reinterpret_cast<uint4*>(rb + (((u0 + 1) ^ sw) << 4)) = hi;
    convert_block(v1, rebase_scale2(R - (sc >> 8)), lo, hi);
    *reinterpret_cast<uint4*>(rb + (((u0 + 2) ^ sw) << 4)) = lo;
    *reinterpret_cast<uint4*>(rb + (((u0 + 3) ^ sw) << 4)) = hi;
  }
  // rope dims: blocks 16, 17 -> 16-byte columns 0..3 of the no-swizzle operand
  uint8_t* rrow = stage + kVBytes + (tr >> 3) * 512 + (tr & 7) * 16;
  const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(ssc + 16);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(srow + 16 * (16 + q));
    uint4 lo, hi;
    convert_block(v, rebase_scale2(R - ((sc2 >> (8 * q)) & 0xFFu)), lo, hi);
    *reinterpret_cast<uint4*>(rrow + (2 * q) * 128) = lo;
    *reinterpret_cast<uint4*>(rrow + (2 * q + 1) * 128) = hi;
  }
  rexp[tr] = static_cast<uint8_t>(R);
}

// Stage i % 2 is free for tile i once the P.V of tile i - 2 is done.
__device__ __forceinline__ bool wait_stage(const Cx& cx, uint32_t i) {
  return i < 2 || cx.wait(L::kPvDone + (i & 1u), ((i - 2) >> 1) & 1u);
}

// Tile i (this warp's rows staged in raw_w / sc_w) into stage i % 2.
__device__ __forceinline__ void convert_tile(const Cx& cx, uint32_t i, int warp, int lane, const uint8_t* raw_w,
                                             const uint8_t* sc_w) {
  const uint32_t st = i & 1u;
  convert_row(cx.g + L::kOffKv + st * kStageBytes, cx.g + L::kOffRexp + st * kTileRows, 32 * warp + lane,
              raw_w + lane * (kDqk / 2), sc_w + lane * (kDqk / kMxBlock));
}

// Hands stage i % 2 to the UMMA issuer (generic-proxy writes made visible to
// the tensor core first).
__device__ __forceinline__ void publish_tile(const Cx& cx, uint32_t i, int warp, int lane, uint32_t meta) {
  if (warp == 0 && lane == 0) reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffMeta)[i & 3u] = meta;
  fence_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(cx.bar(L::kKvFull + (i & 1u)));
}

constexpr uint32_t kIdQK = umma_idesc(128, 32, 1, 0, false, false);  // A e5m2 K-major, B e4m3
constexpr uint32_t kIdPV = umma_idesc(128, 32, 1, 0, true, true);    // A = V^T MN-major, B = P^T MN-major

// Q.K^T of tile i into S[i % 2] (its stage, S buffer and q are ready).
__device__ __forceinline__ void issue_qk(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + b * kStageBytes, qbuf = cx.s + L::kOffQ;
  const uint32_t d = cx.tmem + kTmemS + 32 * b;
#pragma unroll
  for (int ks = 0; ks < 16; ++ks) umma_e4m3(d, qk_desc_a(stage, ks), qk_desc_b(qbuf, ks), kIdQK, ks > 0 ? 1u : 0u);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) umma_e4m3(d, rope_desc_a(stage + kVBytes, ks), qk_desc_b(qbuf, 16 + ks), kIdQK, 1u);
  umma_commit(cx.bar(L::kSFull + b));
  if (t.last) umma_commit(cx.bar(L::kQEmpty));
}

// P.V of tile i into O[piece % 2] (its P is written and O is free).
__device__ __forceinline__ void issue_pv(const Cx& cx, uint32_t i, const TileMeta& t) {
  const uint32_t b = i & 1u;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + b * kStageBytes, pbuf = cx.s + L::kOffP + b * kPBytes;
  const uint32_t obuf = cx.tmem + kTmemO + (t.k & 1u) * 128;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_e4m3(obuf + 32 * mb, pv_desc_a(stage, mb, ks), pv_desc_b(pbuf, ks), kIdPV, (ks > 0 || !t.first) ? 1u : 0u);
  umma_commit(cx.bar(L::kPvDone + b));
  if (t.last) umma_commit(cx.bar(L::kOFull + (t.k & 1u)));
}

__device__ void converter_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  const uint32_t ntiles = static_cast<uint32_t>(count_tiles(cur));
  uint8_t* raw_w = cx.g + L::kOffRaw + warp * 32 * (kDqk / 2);
  uint8_t* sc_w = cx.g + L::kOffRawSc + warp * 32 * (kDqk / kMxBlock);
  MetaTileWalker rw;
  rw.init(cur);
  // one tile ahead in registers (a second set measured slower: the register
  // pressure slowed the conversion more than the earlier loads gained)
  MxRaw ra;
  uint32_t ma;
  load_mx_raw(p, rw, warp, lane, ra, ma);
  for (uint32_t i = 0; i < ntiles; i += 2) {
    const bool two = i + 1 < ntiles;
    if (!wait_stage(cx, i)) break;
    dump_raw(raw_w, sc_w, lane, ra);
    __syncwarp();
    const uint32_t m0 = ma;
    load_mx_raw(p, rw, warp, lane, ra, ma);  // tile i + 1
    convert_tile(cx, i, warp, lane, raw_w, sc_w);
    publish_tile(cx, i, warp, lane, m0);
    if (!two) break;
    if (!wait_stage(cx, i + 1)) break;
    dump_raw(raw_w, sc_w, lane, ra);
    __syncwarp();
    const uint32_t m1 = ma;
    load_mx_raw(p, rw, warp, lane, ra, ma);  // tile i + 2
    convert_tile(cx, i + 1, warp, lane, raw_w, sc_w);
    publish_tile(cx, i + 1, warp, lane, m1);
  }
}

// Warp 8, lane 0: issues Q.K^T of tile qi and P.V of tile pi as soon as each
// is ready (non-blocking tests, bounded overall), in tile order for each kind.
__device__ void issuer_role(const Cx& cx, PieceCursor cur) {
  const uint32_t n = static_cast<uint32_t>(count_tiles(cur));
  const volatile uint32_t* meta = reinterpret_cast<const volatile uint32_t*>(cx.g + L::kOffMeta);
  uint32_t qi = 0, pi = 0;
  long long t0 = clock64();
  while (pi < n) {
    bool progressed = false;
    if (pi < qi && mbar_test_wait(cx.bar(L::kPFull + (pi & 1u)), (pi >> 1) & 1u)) {
      const TileMeta t = TileMeta::unpack(meta[pi & 3u]);
      if (!t.first || t.k < 2 || mbar_test_wait(cx.bar(L::kOEmpty + (t.k & 1u)), ((t.k >> 1) - 1) & 1u)) {
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
      const int r = static_cast<int>(cx.g[L::kOffRexp + b * kTileRows + sx.row]) - 127;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(cx.tmem + sx.lane_base + kTmemS + 32 * b, sr);
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
        rescale_o(cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128, alpha_o);
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
    if (!cx.wait(L::kOFull + (k & 1u), (k >> 1) & 1u)) return;
    tc_fence_after();
    store_o(p, pc, cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128, sx.row, f);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty + (k & 1u)));
    if (!pc.direct && !finish_partial(p, cx, sx, pc)) return;
    pc = nxt;
    have = have_next;
    c = c_next;
    ++k;
  }
}

template <int QF>
__global__ void __launch_bounds__(kThreads, 1) stage1_mx_kernel(const Stage1Params p) {
  extern __shared__ uint8_t smem_raw[];
  Cx cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, 8, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < 4) {
    setmaxnreg_inc<kWorkRegs>();
    converter_role(p, cx, cur, warp, lane);
    setmaxnreg_dec<kLaunchRegs>();
  } else if (warp < 8) {
    setmaxnreg_inc<kWorkRegs>();
    softmax_role<QF>(p, cx, cur, warp, lane);
    setmaxnreg_dec<kLaunchRegs>();
  } else {
    setmaxnreg_dec<kIssueRegs>();
    if (warp == 8 && lane == 0) issuer_role(cx, cur);
    __syncwarp();
  }
  // The issuing warpgroup takes its registers back only after warpgroups 0
  // and 1 have returned theirs (their dec comes before this barrier), so the
  // inc below can always be granted at once. Asking for them earlier could
  // leave warpgroups 0-1 waiting in their own inc for registers that the
  // issuing warpgroup holds while it waits at a barrier for them.
  __syncthreads();
  if (warp >= 8) setmaxnreg_inc<kLaunchRegs>();  // back to the launch budget for the common tail
  cta_end(p, cx, 8);
}

template <int QF>
static cudaError_t launch_q(const Stage1Params& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    // the warpgroup register split adds up to the launch budget only at 168
    // registers per thread; anything else would leave setmaxnreg waiting
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, stage1_mx_kernel<QF>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(stage1_mx_kernel<QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_dependent(stage1_mx_kernel<QF>, p.num_splits, kThreads, L::kAlloc, stream, p);
}

}  // namespace mx
}  // namespace tc

cudaError_t launch_stage1_tc_mxfp4(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  return q_fmt == kQBf16 ? tc::mx::launch_q<kQBf16>(p, stream) : tc::mx::launch_q<kQFp8>(p, stream);
}

}  // namespace mla
