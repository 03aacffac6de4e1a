// Stage 1 of split-K MLA decode for an fp8 (e4m3) KV cache on the 5th-generation
// tensor cores (tcgen05): TMA streams 128-row KV tiles, one thread issues the
// UMMAs, accumulators live in tensor memory, 4 warps run the online softmax.
//
// Method: split-K flash decoding as in kernelbot-amd-mixed-mla-753817
// (`mla_flash_decode_stage1`): the 16 query heads share the single latent KV
// head, scores use all 576 dims, values the first 512, the online softmax runs
// in the exp2 domain with sm_scale*log2(e) folded into the scores, and each
// split leaves a normalised partial output plus its LSE.
//
// GB300 design:
//  * Rows of KV are the MMA M dimension (M = 128), heads are N:
//      S^T[row, head]  = K[row, 0:576] . Q^T          (A = KV tile, K-major)
//      O^T[dim, head] += V^T[dim, rows] . P^T[rows, head]  (A = the same tile
//                         read MN-major, so V needs no transpose and no copy)
//  * The stored e4m3 codes are the MMA operands; there is no dequantisation
//    pass. The bf16 operand (q, or the softmax weights P) enters as two e4m3
//    values hi = e4m3(x), lo = e4m3(16 (x - hi)) stacked along N (N = 32:
//    16 hi columns + 16 lo columns): a UMMA with N = 32 costs the same as one
//    with N = 16, and hi + lo/16 carries x to 8 significant bits wherever hi is
//    a normal number. The per-tensor kv scale, 2^-shift of q and 1/256 of P are
//    applied to the fp32 results.
//  * Shared memory holds three 64 KB stages of the 512 V dims of 128-row tiles
//    (four 128B-swizzled 128x128 TMA boxes each), so two tiles stream in while
//    one is consumed. The 64 rope dims of each row (used by Q.K^T only) are
//    loaded by the softmax threads into registers two tiles ahead and written
//    into a single 8 KB slot as soon as the previous tile's Q.K^T is done.
//  * Warp 0 issues the TMA loads, warp 1 owns tensor memory and issues QK(n)
//    then PV(n-1) so the tensor core overlaps the softmax of tile n, warps 2-5
//    (one thread per tile row / tensor-memory lane) read S, reduce the per-head
//    max across the 128 rows, write P into shared memory, rescale O in tensor
//    memory only when some head's running max grew, and run the epilogue.
//  * Every mbarrier wait is bounded; on a timeout the CTA stops issuing work,
//    lets in-flight copies and MMAs finish, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_device.cuh"
#include "mla_internal.h"
#include "mla_partition.cuh"
#include "mla_tcgen05.cuh"

namespace mla {
namespace tc {

constexpr int kThreads = 192;                        // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kTileRows = 128;
constexpr int kVChunks = 4;                          // 128-byte column chunks of the 512 V dims
constexpr int kChunkBytes = kTileRows * 128;         // 16 KB (one TMA box)
constexpr int kStageBytes = kVChunks * kChunkBytes;  // 64 KB
constexpr int kStages = 3;
constexpr int kQChunkBytes = 32 * 128;               // 32 B-operand rows (hi, lo) x 128 B
constexpr int kQBytes = 5 * kQChunkBytes;            // 20 KB (chunk 4: rope dims, 64 B used)
constexpr int kRopeBytes = kTileRows * 64;           // [row group 16][16-B column 4][8 rows][16 B]
constexpr int kPBytes = kTileRows * 32;              // [row group][hi | lo][8 rows][16 heads]
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;                      // 2 buffers x 32 columns
constexpr uint32_t kTmemO = 64;                     // 2 buffers x (4 blocks x 32 columns)
constexpr float kLoScale = 16.0f;
constexpr float kPScale = 256.0f;
constexpr float kLog2e = 1.4426950408889634f;

struct L {
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffRope = kOffQ + kQBytes;
  static constexpr int kOffP = kOffRope + kRopeBytes;
  static constexpr int kOffRedMax = kOffP + kPBytes;              // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * 16 * 4;    // [4][16] f32
  static constexpr int kOffAmax = kOffRedL + 4 * 16 * 4;          // [4] u32
  static constexpr int kOffScan = kOffAmax + 16;                  // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  enum {
    kKvFull = 0, kKvEmpty = 3, kSFull = 6, kSEmpty = 8, kRopeFull = 10, kPFull = 11, kPEmpty = 12, kQFull = 13,
    kQEmpty = 14, kOFull = 15, kOEmpty = 17, kGrp = 19, kDrain = 21, kNumBars = 22
  };
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;  // slack: the base is aligned up to 1024 B
};
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffQ % 1024 == 0 && L::kOffRope % 1024 == 0, "operands need 1024-byte alignment");

// Optional phase timers (build with -DMLA_PHASE_TIMING): cycles per CTA, warp
// and phase, summed over the launch. Off by default.
#ifdef MLA_PHASE_TIMING
constexpr int kPhaseCtas = 1024;
__device__ unsigned long long g_tc_phase[kPhaseCtas * 8 * 8];
#define TC_PT_INIT long long tc_pt_ = clock64();
#define TC_PT(ph)                                                                                          \
  do {                                                                                                     \
    const long long now_ = clock64();                                                                      \
    if ((threadIdx.x & 31) == 0 && blockIdx.x < kPhaseCtas)                                                \
      atomicAdd(&g_tc_phase[(blockIdx.x * 8 + (threadIdx.x >> 5)) * 8 + (ph)],                             \
                static_cast<unsigned long long>(now_ - tc_pt_));                                           \
    tc_pt_ = now_;                                                                                         \
  } while (0)
#else
#define TC_PT_INIT
#define TC_PT(ph) \
  do {            \
  } while (0)
#endif

struct Ctx {
  uint8_t* g;        // generic pointer to the aligned base
  uint32_t s;        // shared address of the aligned base
  volatile uint32_t* abort_word;
  uint32_t* flags;
  uint32_t tmem;
  __device__ __forceinline__ uint32_t bar(int i) const { return s + L::kOffBars + 8u * i; }
  __device__ __forceinline__ bool wait(int i, uint32_t parity) const { return mbar_wait(bar(i), parity, abort_word, flags); }
};

__device__ __forceinline__ void mbar_wait_drain_tc(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// ---------------------------------------------------------------------------
// Walks the CTA's tiles in order (one 128-row tile at a time).
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
};

// Warp 0: the V dims of each tile, four 128-row x 128-byte boxes, into stage
// (tile % 3) once the tile three back has been released by its P.V.
__device__ void producer(const Ctx& cx, const CUtensorMap* map, PieceCursor cur, int lane) {
  const uint64_t pol = policy_evict_first();
  Piece pc;
  uint32_t n = 0;
  bool ok = true;
  TC_PT_INIT
  while (ok && cur.next(pc)) {
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n % kStages, rnd = n / kStages;
      TC_PT(1);
      if (rnd >= 1 && !cx.wait(L::kKvEmpty + s, (rnd - 1) & 1u)) {
        ok = false;
        break;
      }
      TC_PT(0);
      if (lane == 0) {
        mbar_arrive_expect_tx(cx.bar(L::kKvFull + s), kStageBytes);
        const uint32_t dst = cx.s + L::kOffKv + s * kStageBytes;
        for (int c = 0; c < kVChunks; ++c)
          tma_load_2d(dst + c * kChunkBytes, map, c * 128, pc.kv_row + r0, cx.bar(L::kKvFull + s), pol);
      }
      __syncwarp();
      ++n;
    }
  }
  // the last tile issued on each stage must have landed before the CTA exits
  for (uint32_t s = 0; s < kStages && s < n; ++s) {
    const uint32_t last = ((n - 1 - s) / kStages) * kStages + s;
    mbar_wait_drain_tc(cx.bar(L::kKvFull + s), (last / kStages) & 1u);
  }
}

// ---------------------------------------------------------------------------
// Warp 1 (one thread): QK(n) into S[n % 2], then PV(n-1) into O[piece % 2].
struct PendingPV {
  uint32_t n, k;
  bool first, last, valid;
};

__device__ bool issue_pv(const Ctx& cx, const PendingPV& t) {
  constexpr uint32_t id_pv = umma_idesc(128, 32, 0, 0, true, true);
  TC_PT_INIT
  if (!cx.wait(L::kPFull, t.n & 1u)) return false;
  if (t.first && t.k >= 2 && !cx.wait(L::kOEmpty + (t.k & 1u), ((t.k >> 1) - 1) & 1u)) return false;
  TC_PT(4);
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + (t.n % kStages) * kStageBytes;
  const uint32_t pbuf = cx.s + L::kOffP;
  const uint32_t obuf = cx.tmem + kTmemO + (t.k & 1u) * 128;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      // A = V^T: dims 128mb.. of rows 32ks..: MN-major, 8-row atoms 1024 B apart
      const uint64_t a = smem_desc(stage + mb * kChunkBytes + ks * 4096, kChunkBytes, 1024, kLayoutSw128);
      // B = P^T: N = 32 (hi heads, lo heads: core matrices 128 B apart), K = rows (8-row groups 256 B apart)
      const uint64_t b = smem_desc(pbuf + ks * 1024, 256, 128, kLayoutNone);
      umma_e4m3(obuf + 32 * mb, a, b, id_pv, (ks > 0 || !t.first) ? 1u : 0u);
    }
  umma_commit(cx.bar(L::kKvEmpty + (t.n % kStages)));
  umma_commit(cx.bar(L::kPEmpty));
  if (t.last) umma_commit(cx.bar(L::kOFull + (t.k & 1u)));
  TC_PT(5);
  return true;
}

__device__ void mma_issuer(const Ctx& cx, PieceCursor cur) {
  constexpr uint32_t id_qk = umma_idesc(128, 32, 0, 0, false, false);
  Piece pc;
  uint32_t n = 0, k = 0;
  PendingPV pend{0, 0, false, false, false};
  bool ok = true;
  TC_PT_INIT
  while (ok && cur.next(pc)) {
    TC_PT(7);
    if (!cx.wait(L::kQFull, k & 1u)) break;
    TC_PT(0);
    const uint32_t qbuf = cx.s + L::kOffQ;
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n & 1u, st = n % kStages;
      TC_PT(7);
      if (!cx.wait(L::kKvFull + st, (n / kStages) & 1u) || !cx.wait(L::kRopeFull, n & 1u)) {
        ok = false;
        break;
      }
      TC_PT(1);
      if (n >= 2 && !cx.wait(L::kSEmpty + s, ((n >> 1) - 1) & 1u)) {
        ok = false;
        break;
      }
      TC_PT(2);
      tc_fence_after();
      const uint32_t stage = cx.s + L::kOffKv + st * kStageBytes;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {  // the 512 V dims, from the stage
        const uint64_t a = smem_desc(stage + (ks >> 2) * kChunkBytes + (ks & 3) * 32, 16, 1024, kLayoutSw128);
        const uint64_t b = smem_desc(qbuf + (ks >> 2) * kQChunkBytes + (ks & 3) * 32, 16, 1024, kLayoutSw128);
        umma_e4m3(cx.tmem + kTmemS + 32 * s, a, b, id_qk, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {  // the 64 rope dims, from the rope slot (no swizzle)
        const uint64_t a = smem_desc(cx.s + L::kOffRope + ks * 256, 128, 512, kLayoutNone);
        const uint64_t b = smem_desc(qbuf + 4 * kQChunkBytes + ks * 32, 16, 1024, kLayoutSw128);
        umma_e4m3(cx.tmem + kTmemS + 32 * s, a, b, id_qk, 1u);
      }
      umma_commit(cx.bar(L::kSFull + s));
      const bool last = r0 + kTileRows >= pc.nrows;
      if (last) umma_commit(cx.bar(L::kQEmpty));
      TC_PT(3);
      if (pend.valid && !issue_pv(cx, pend)) {
        ok = false;
        break;
      }
      pend = PendingPV{n, k, r0 == 0, last, true};
#ifdef MLA_PHASE_TIMING
      tc_pt_ = clock64();
#endif
      ++n;
    }
    ++k;
  }
  if (ok && pend.valid) issue_pv(cx, pend);
  // every issued tcgen05 operation completes before tensor memory is freed
  umma_commit(cx.bar(L::kDrain));
  mbar_wait_drain_tc(cx.bar(L::kDrain), 0);
}

// ---------------------------------------------------------------------------
// Warps 2-5. Thread = tile row = tensor-memory lane (32 * (warp % 4) + lane).

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

struct SoftmaxCtx {
  int row, wi, lane;
  uint32_t lane_base;
  uint32_t gcount;
};

__device__ __forceinline__ bool group_sync(const Ctx& cx, SoftmaxCtx& sx) {
  const uint32_t k = sx.gcount & 1u, par = (sx.gcount >> 1) & 1u;
  ++sx.gcount;
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kGrp + k));
  return cx.wait(L::kGrp + k, par);
}

// q of one token -> Q buffer kk % 2 as the B operand (K-major, 128B swizzle,
// rows 0-15 = e4m3(q 2^shift), rows 16-31 = e4m3(16 (q 2^shift - hi))).
// Returns the score scale (exp2 domain) or a negative value on abort.
template <int QF>
__device__ float setup_q(const Stage1Params& p, const Ctx& cx, SoftmaxCtx& sx, int token, uint32_t kk, float kvsc) {
  // the single Q buffer is free once the previous piece's last Q.K^T is done
  if (kk >= 1 && !cx.wait(L::kQEmpty, (kk - 1) & 1u)) return -1.f;
  const int t = 32 * sx.wi + sx.lane;  // 0..127
  const int h = t >> 3, d0 = 72 * (t & 7);
  uint8_t* qb = cx.g + L::kOffQ;
  auto qaddr = [&](int row, int d) -> uint32_t* {
    const int unit = (d & 127) >> 4;
    return reinterpret_cast<uint32_t*>(qb + (d >> 7) * kQChunkBytes + (row >> 3) * 1024 + (row & 7) * 128 +
                                       ((unit ^ (row & 7)) << 4) + (d & 15));
  };
  float c;
  if (QF == kQBf16) {
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
    uint32_t* am = reinterpret_cast<uint32_t*>(cx.g + L::kOffAmax);
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
      *qaddr(16 + h, d0 + 8 * i) = 0u;
      *qaddr(16 + h, d0 + 8 * i + 4) = 0u;
    }
    c = p.sm_scale * kLog2e * kvsc * __ldg(p.q_scale);
  }
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kQFull));
  return c;
}

// Rope dims (bytes 512..575) of one tile row, from global memory into registers;
// rows past the end of the cache read as zero.
__device__ __forceinline__ void load_rope(const Stage1Params& p, TileWalker& rw, int row, uint4 (&r)[4]) {
  int32_t row0;
  const bool have = rw.next(row0);
  const int64_t g = static_cast<int64_t>(row0) + row;
  if (have && g < p.total_kv) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.kv) + g * kDqk + 512);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __ldg(src + i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Writes one row's rope bytes into the slot (no-swizzle K-major A operand:
// 8-row x 16-byte core matrices, 128 B apart along K, 512 B apart along rows)
// and hands the slot to the MMA warp.
__device__ __forceinline__ void store_rope(const Ctx& cx, const SoftmaxCtx& sx, const uint4 (&r)[4]) {
  uint8_t* base = cx.g + L::kOffRope + (sx.row >> 3) * 512 + (sx.row & 7) * 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(base + i * 128) = r[i];
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kRopeFull));
}

template <int QF>
__device__ void softmax_role(const Stage1Params& p, const Ctx& cx, PieceCursor cur, int warp, int lane) {
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = warp - 2;
  sx.row = 32 * (warp & 3) + lane;
  sx.lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  sx.gcount = 0;
  const float kvsc = __ldg(static_cast<const float*>(p.kv_scale));
  float* red_max = reinterpret_cast<float*>(cx.g + L::kOffRedMax);
  float* red_l = reinterpret_cast<float*>(cx.g + L::kOffRedL);

  PieceCursor ahead = cur;
  Piece pc, nxt;
  bool have = ahead.next(pc);
  if (!have) return;
  // rope of tiles 0 and 1 into registers; tile 0 into the slot; tile 2 loads
  TileWalker rw;
  rw.init(cur);
  uint4 rb0[4], rb1[4];  // rope of the even / odd tile in flight
  load_rope(p, rw, sx.row, rb0);
  load_rope(p, rw, sx.row, rb1);
  store_rope(cx, sx, rb0);
  load_rope(p, rw, sx.row, rb0);
  float c = setup_q<QF>(p, cx, sx, pc.token, 0, kvsc);
  if (c < 0.f) return;
  uint32_t n = 0, k = 0;
  int tiles_left = 0;  // tiles of the CTA after the current one (for the rope slot)
  {
    PieceCursor cnt = cur;
    Piece t;
    while (cnt.next(t)) tiles_left += (t.nrows + kTileRows - 1) / kTileRows;
    tiles_left -= 1;
  }
  TC_PT_INIT
  while (have) {
    const bool have_next = ahead.next(nxt);
    float m[16], l[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const int nr = min(kTileRows, pc.nrows - r0);
      const uint32_t s = n & 1u;
      TC_PT(7);
      if (!cx.wait(L::kSFull + s, (n >> 1) & 1u)) return;
      TC_PT(0);
      // Q.K^T(n) is done: the rope slot takes tile n+1, its registers tile n+3
      if (tiles_left > 0) {
        if (n & 1u) {
          store_rope(cx, sx, rb0);
          load_rope(p, rw, sx.row, rb0);
        } else {
          store_rope(cx, sx, rb1);
          load_rope(p, rw, sx.row, rb1);
        }
      }
      --tiles_left;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(cx.tmem + sx.lane_base + kTmemS + 32 * s, sr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + s));
      const bool valid = sx.row < nr;
      float x[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float v = (__uint_as_float(sr[h]) + __uint_as_float(sr[16 + h]) * (1.0f / kLoScale)) * c;
        x[h] = valid ? v : -INFINITY;
      }
      const float wm = warp_reduce16<true>(x, lane);
      float* rm = red_max + (n & 1u) * 64;
      if ((lane & 1) == 0) rm[sx.wi * 16 + (lane >> 1)] = wm;
      TC_PT(1);
      if (!group_sync(cx, sx)) return;
      TC_PT(2);
      bool grew = false;
      float alpha[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float tm = fmaxf(fmaxf(rm[h], rm[16 + h]), fmaxf(rm[32 + h], rm[48 + h]));
        const float mn = fmaxf(m[h], tm);
        alpha[h] = fast_exp2(m[h] - mn);
        grew |= mn > m[h];
        m[h] = mn;
      }
      const bool rescale = grew && r0 > 0;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 4 * q4 + e;
          pv[e] = fast_exp2(x[h] - m[h]);
          l[h] = l[h] * alpha[h] + pv[e];
          pv[e] *= kPScale;
        }
        const uint32_t h01 = f32x2_to_e4m3x2(pv[0], pv[1]), h23 = f32x2_to_e4m3x2(pv[2], pv[3]);
        const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
        hi[q4] = h01 | (h23 << 16);
        lo[q4] = f32x2_to_e4m3x2(kLoScale * (pv[0] - d01.x), kLoScale * (pv[1] - d01.y)) |
                 (f32x2_to_e4m3x2(kLoScale * (pv[2] - d23.x), kLoScale * (pv[3] - d23.y)) << 16);
      }
      TC_PT(3);
      // single P buffer: P.V(n-1) must be done
      if (n >= 1 && !cx.wait(L::kPEmpty, (n - 1) & 1u)) return;
      TC_PT(4);
      uint8_t* pb = cx.g + L::kOffP + (sx.row >> 3) * 256 + (sx.row & 7) * 16;
      *reinterpret_cast<uint4*>(pb) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(pb + 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (!valid) {
        // rows past the piece: zero their V bytes so P = 0 meets finite values
        uint8_t* vrow = cx.g + L::kOffKv + (n % kStages) * kStageBytes + sx.row * 128;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(vrow + ch * kChunkBytes + u * 16) = make_uint4(0, 0, 0, 0);
      }
      if (rescale) {
        // O of this piece is final for tile n-1: P.V(n-1) completed (waited above)
        tc_fence_after();
        const uint32_t ob = cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128;
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
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull));
      TC_PT(5);
      ++n;
    }

    // the next piece's q goes in while this piece's last PV runs
    float c_next = c;
    if (have_next) {
      c_next = setup_q<QF>(p, cx, sx, nxt.token, k + 1, kvsc);
      if (c_next < 0.f) return;
    }
    // l over the 128 rows, per head
    const float wl = warp_reduce16<false>(l, lane);
    if ((lane & 1) == 0) red_l[sx.wi * 16 + (lane >> 1)] = wl;
    if (!group_sync(cx, sx)) return;
    float f[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const float L = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
      f[h] = kvsc / (kPScale * L);
      if (!pc.direct && sx.row == h) p.part_lse[pc.slot * kHeads + h] = m[h] + fast_log2(L);
    }
    if (!cx.wait(L::kOFull + (k & 1u), (k >> 1) & 1u)) return;
    tc_fence_after();
    const uint32_t ob = cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128;
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
      uint32_t o[32];
      tmem_ld32(ob + 32 * mb, o);
      tmem_wait_ld();
      const int dim = 128 * mb + sx.row;
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
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty + (k & 1u)));
    TC_PT(6);
    pc = nxt;
    have = have_next;
    c = c_next;
    ++k;
  }
}

template <int QF>
__global__ void __launch_bounds__(kThreads, 1) stage1_tc_kernel(const Stage1Params p, const __grid_constant__ CUtensorMap kvmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  Ctx cx;
  cx.s = (raw + 1023u) & ~1023u;
  cx.g = smem_raw + (cx.s - raw);
  cx.abort_word = reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffAbort);
  cx.flags = p.dev_flags;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(cx.bar(L::kKvFull + i), 1);
      mbar_init(cx.bar(L::kKvEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(L::kSFull + i), 1);
      mbar_init(cx.bar(L::kSEmpty + i), 4);
      mbar_init(cx.bar(L::kOFull + i), 1);
      mbar_init(cx.bar(L::kOEmpty + i), 4);
      mbar_init(cx.bar(L::kGrp + i), 4);
    }
    mbar_init(cx.bar(L::kRopeFull), 4);
    mbar_init(cx.bar(L::kPFull), 4);
    mbar_init(cx.bar(L::kPEmpty), 1);
    mbar_init(cx.bar(L::kQFull), 4);
    mbar_init(cx.bar(L::kQEmpty), 1);
    mbar_init(cx.bar(L::kDrain), 1);
    *cx.abort_word = 0u;
    fence_mbar_init();
  }
  const int64_t parts = p.num_splits, c = blockIdx.x;
  int64_t* sh = reinterpret_cast<int64_t*>(cx.g + L::kOffScan);
  const SegLocate loc = block_locate<kThreads, 1>(
      p.qo_indptr, p.kv_indptr, p.batch, p.total_q, p.total_kv,
      [=](int64_t total) { return part_start(c, total, parts); }, 0, sh);
  if (!loc.ok) {
    if (threadIdx.x == 0) atomicOr(p.dev_flags, kFlagBadIndptr);
    return;
  }
  const int64_t x0 = part_start(c, loc.total, parts), x1 = part_start(c + 1, loc.total, parts);
  if (x0 >= x1 || loc.seg < 0) return;  // uniform across the block: nothing allocated yet
  if (warp == 1) tmem_alloc(cx.s + L::kOffSlot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffSlot);
  PieceCursor cur{p.qo_indptr, p.kv_indptr, p.batch, x0, x1, loc.seg, loc.seg_vs, c};
  if (warp == 0)
    producer(cx, &kvmap, cur, lane);
  else if (warp == 1) {
    if (lane == 0) mma_issuer(cx, cur);
    __syncwarp();
  } else
    softmax_role<QF>(p, cx, cur, warp, lane);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host: the KV tensor map (rows of 576 bytes, 128 x 128 boxes, 128B swizzle).
using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  }
  return fn;
}

static cudaError_t make_kv_map(CUtensorMap* map, const void* kv, int64_t total_kv) {
  EncodeFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(total_kv)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

#ifdef MLA_PHASE_TIMING
extern "C" int mla_debug_phase_cycles_tc(unsigned long long* host, int n, int reset) {
  if (n > kPhaseCtas * 64) n = kPhaseCtas * 64;
  if (cudaMemcpyFromSymbol(host, g_tc_phase, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
  if (reset) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_tc_phase) != cudaSuccess) return -1;
    if (cudaMemset(q, 0, sizeof(g_tc_phase)) != cudaSuccess) return -1;
  }
  return n;
}
#endif

template <int QF>
static cudaError_t launch_q(const Stage1Params& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(stage1_tc_kernel<QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap map;
  e = make_kv_map(&map, p.kv, p.total_kv);
  if (e != cudaSuccess) return e;
  stage1_tc_kernel<QF><<<p.num_splits, kThreads, L::kAlloc, stream>>>(p, map);
  return cudaGetLastError();
}

}  // namespace tc

cudaError_t launch_stage1_tc_fp8(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  return q_fmt == kQBf16 ? tc::launch_q<kQBf16>(p, stream) : tc::launch_q<kQFp8>(p, stream);
}

}  // namespace mla
