// Stage 1 for an fp8 (e4m3) KV cache and bf16 q with the query tokens of a
// segment taken in pairs that share one pass over the KV rows (multi-token
// decode). fp8 q has its own kernel (mla_stage1_duo.cu).
//
// Method: as the single-token tensor-core kernel (split-K flash decoding as in
// kernelbot-amd-mixed-mla-753817 `mla_flash_decode_stage1`, scores over all
// 576 dims, values the first 512, exp2-domain online softmax, normalised
// partials plus LSE). Each query token attends to all KV rows of its segment
// (the naive reference of kernelbot-amd-mixed-mla-675627), so two tokens of
// one segment read the same rows; here one tile of rows serves both:
//  * the B operands hold both tokens: Q is 64 rows (token A hi, lo; token B
//    hi, lo) and P is 64 columns, so every UMMA has N = 64. The tensor core
//    reads the 128-row KV tile (the A operand, which bounds a UMMA's time)
//    once for two tokens;
//  * tensor memory: S in 2 buffers x 64 columns, O in one buffer of
//    4 blocks x 64 columns (token A hi, lo, token B hi, lo);
//  * shared memory: two 64 KB V stages (a tile now carries two tokens' work,
//    which hides the TMA latency with one stage in flight), a 40 KB Q buffer,
//    the 8 KB rope slot and an 8 KB P buffer;
//  * a segment with an odd token count ends with a one-token group, which
//    loads that token into both halves and writes only the first;
//  * with two stages the MMA warp issues each product from a polling loop as
//    soon as its inputs are ready, so a P.V does not wait behind the landing
//    of the next tile.
// A token's arithmetic (tiles, maxima, weights, accumulation) is the same as
// in the single-token kernel, so with one partition per segment both give the
// same bits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace pair {

constexpr int kThreads = 256;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax, 6-7 only in the merge
constexpr int kStageBytes = kVBytes;
constexpr int kPBytes2 = kTileRows * 64;  // [row group][A hi | A lo | B hi | B lo][8 rows][16 heads]

// Q = 64 rows (both tokens hi + lo), two stages, rope in the shared-memory slot.
struct L {
  static constexpr int kThreads = pair::kThreads;
  static constexpr int kStages = 2;
  static constexpr int kQRows = 64;
  static constexpr int kQChunk = kQRows * 128;
  static constexpr uint32_t kSCols = kQRows;      // S columns per buffer (Q.K^T N)
  static constexpr uint32_t kTmemO = 2 * kSCols;  // O: 4 blocks x 64 columns
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffRope = kOffQ + 5 * kQChunk;
  static constexpr int kOffP = kOffRope + kRopeBytes;
  static constexpr int kOffRedMax = kOffP + kPBytes2;                // [2 buffers][2 tokens][4 warps][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 2 * 4 * 16 * 4;   // [2 tokens][4][16] f32
  static constexpr int kOffAmax = kOffRedL + 2 * 4 * 16 * 4;         // [2 tokens][4 warps] u32
  static constexpr int kOffMList = kOffAmax + 32;                    // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                    // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  enum {
    kKvFull = 0, kKvEmpty = 3, kSFull = 6, kSEmpty = 8, kRopeFull = 10, kPFull = 11, /* 12 unused */ kQFull = 13,
    kQEmpty = 14, kOFull = 15, kOEmpty = 16, kGrp = 17, kDrain = 19, kMerge = 20, kNumBars = 21
  };
  static constexpr int kMergeBytes = kStages * kStageBytes;  // the stages hold partials for the end-of-CTA merge
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;  // slack: the base is aligned up to 1024 B
  template <class C>
  __device__ static void init_barriers(const C& cx) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(cx.bar(kKvFull + i), 1);
      mbar_init(cx.bar(kKvEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(kSFull + i), 1);
      mbar_init(cx.bar(kSEmpty + i), 4);
      mbar_init(cx.bar(kGrp + i), 4);
    }
    mbar_init(cx.bar(kRopeFull), 4);
    mbar_init(cx.bar(kPFull), 4);
    mbar_init(cx.bar(kQFull), 4);
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kOFull), 1);
    mbar_init(cx.bar(kOEmpty), 4);
    mbar_init(cx.bar(kDrain), 1);
  }
};
using Cx = Ctx<L>;
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffQ % 1024 == 0 && L::kOffRope % 1024 == 0 && L::kOffP % 1024 == 0, "operand alignment");
static_assert(L::kOffScan % 8 == 0, "scratch alignment");
static_assert(L::kTmemO + 256 <= kTmemCols, "tensor memory");

// B operands.
//   Q.K^T k-step ks: the Q rows of chunk ks / 4 (K-major, 128B swizzle).
__device__ __forceinline__ uint64_t qk_desc_b2(uint32_t qbuf, int ks) {
  return smem_desc(qbuf + (ks >> 2) * L::kQChunk + (ks & 3) * 32, 16, 1024, kLayoutSw128);
}
//   P.V k-step ks (32 rows): P^T, 4 N-blocks of 16 columns 128 B apart, 8-row
//   groups 512 B apart.
__device__ __forceinline__ uint64_t pv_desc_b2(uint32_t pbuf, int ks) {
  return smem_desc(pbuf + ks * 2048, 512, 128, kLayoutNone);
}

// Warp 0: the V dims of each tile, four 128-row x 128-byte boxes, into stage
// (tile % stages) once the tile that used it last has been released by its P.V.
__device__ void producer(const Cx& cx, const CUtensorMap* map, PieceCursor cur, int lane) {
  constexpr int kStages = L::kStages;
  const uint64_t pol = policy_evict_first();
  Piece pc;
  uint32_t n = 0;
  bool ok = true;
  while (ok && cur.next(pc)) {
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n % kStages, rnd = n / kStages;
      if (rnd >= 1 && !cx.wait(L::kKvEmpty + s, (rnd - 1) & 1u)) {
        ok = false;
        break;
      }
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

// Warp 1 (one thread): QK(n) into S[n % 2], then PV(n-1) into O. O has one
// buffer: the first P.V of piece k waits until the epilogue of piece k-1 has
// read O.
struct PendingPV {
  uint32_t n, k;
  bool first, last, valid;
};

__device__ bool issue_pv(const Cx& cx, const PendingPV& t) {
  constexpr int kStages = L::kStages;
  constexpr uint32_t id_pv = umma_idesc(128, 64, 0, 0, true, true);
  if (!cx.wait(L::kPFull, t.n & 1u)) return false;
  if (t.first && t.k >= 1 && !cx.wait(L::kOEmpty, (t.k - 1) & 1u)) return false;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + (t.n % kStages) * kStageBytes;
  const uint32_t pbuf = cx.s + L::kOffP;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_e4m3(cx.tmem + L::kTmemO + 64 * mb, pv_desc_a(stage, mb, ks), pv_desc_b2(pbuf, ks), id_pv,
                (ks > 0 || !t.first) ? 1u : 0u);
  umma_commit(cx.bar(L::kKvEmpty + (t.n % kStages)));
  if (t.last) umma_commit(cx.bar(L::kOFull));
  return true;
}

// With two stages (bf16 q), Q.K^T(n) and P.V(n) are each issued as soon as
// their inputs are ready (a polling loop): a P.V must not wait behind the
// landing of the next tile, whose load starts only when the P.V before it has
// released its stage. The phases tested cannot run ahead by two: stage s is
// refilled only after the P.V of its tile, the P buffer only after its P.V,
// the S buffer only after the Q.K^T that read it back, the rope slot only
// after the Q.K^T that read it, and the next Q only after the last Q.K^T of
// the piece.
__device__ void issue_qk_at(const Cx& cx, uint32_t n, const TileMeta& t) {
  constexpr int kStages = L::kStages;
  constexpr uint32_t id_qk = umma_idesc(128, L::kSCols, 0, 0, false, false);
  const uint32_t s = n & 1u, st = n % kStages;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + st * kStageBytes;
  const uint32_t sbuf = cx.tmem + L::kSCols * s;
  const uint32_t qbuf = cx.s + L::kOffQ;
#pragma unroll
  for (int ks = 0; ks < 16; ++ks)  // the 512 V dims, from the stage
    umma_e4m3(sbuf, qk_desc_a(stage, ks), qk_desc_b2(qbuf, ks), id_qk, ks > 0 ? 1u : 0u);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks)  // the 64 rope dims, from the rope slot
    umma_e4m3(sbuf, rope_desc_a(cx.s + L::kOffRope, ks), qk_desc_b2(qbuf, 16 + ks), id_qk, 1u);
  umma_commit(cx.bar(L::kSFull + s));
  if (t.last) umma_commit(cx.bar(L::kQEmpty));
}

__device__ void mma_issuer_polling(const Cx& cx, PieceCursor cur) {
  constexpr int kStages = L::kStages;
  const uint32_t n = static_cast<uint32_t>(count_tiles(cur));
  MetaTileWalker wq, wp;
  wq.init(cur);
  wp.init(cur);
  int32_t row;
  uint32_t mq = 0, mp = 0;
  wq.next(row, mq);
  wp.next(row, mp);
  uint32_t qi = 0, pi = 0;
  long long t0 = clock64();
  while (pi < n) {
    bool progressed = false;
    if (pi < qi && mbar_test_wait(cx.bar(L::kPFull), pi & 1u)) {
      const TileMeta t = TileMeta::unpack(mp);
      if (!t.first || t.k == 0 || mbar_test_wait(cx.bar(L::kOEmpty), (t.k - 1) & 1u)) {
        // its own waits (P full, O free) pass at once
        if (!issue_pv(cx, PendingPV{pi, t.k, t.first, t.last, true})) break;
        ++pi;
        wp.next(row, mp);
        progressed = true;
      }
    }
    if (qi < n && mbar_test_wait(cx.bar(L::kKvFull + qi % kStages), (qi / kStages) & 1u) &&
        mbar_test_wait(cx.bar(L::kRopeFull), qi & 1u) &&
        (qi < 2 || mbar_test_wait(cx.bar(L::kSEmpty + (qi & 1u)), ((qi - 2) >> 1) & 1u))) {
      const TileMeta t = TileMeta::unpack(mq);
      if (!t.first || mbar_test_wait(cx.bar(L::kQFull), t.k & 1u)) {
        issue_qk_at(cx, qi, t);
        ++qi;
        wq.next(row, mq);
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
// Warps 2-5. Thread = tile row = tensor-memory lane (32 * (warp % 4) + lane).

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

// One row's rope bytes into the shared-memory rope slot and the hand-off to
// the MMA warp.
__device__ __forceinline__ void store_rope(const Cx& cx, const SoftmaxCtx& sx, const uint4 (&r)[4]) {
  put_rope_row(cx.g + L::kOffRope, sx.row, r);
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kRopeFull));
}

// The q of a piece's tokens: token A into Q rows 0-31 (hi, lo), token B into
// rows 32-63; a one-token group loads its token twice. Returns false on abort.
__device__ bool setup_q2(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, const Piece& pc, uint32_t kk,
                         float kvsc, float& ca, float& cb) {
  if (kk >= 1 && !cx.wait(L::kQEmpty, (kk - 1) & 1u)) return false;
  ca = fill_q<L, kQBf16, L::kQChunk, true>(p, cx, sx, pc.token, 0, kk, kvsc);
  if (ca < 0.f) return false;
  cb = fill_q<L, kQBf16, L::kQChunk, true>(p, cx, sx, pc.token + (pc.ntok > 1 ? 1 : 0), L::kQRows / 2, kk, kvsc);
  if (cb < 0.f) return false;
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kQFull));
  return true;
}

// One row of softmax weights of both tokens (16 heads each, already times
// kPScale) as hi/lo e4m3 into the P operand's four 16-column blocks.
__device__ __forceinline__ void put_p_row2(uint8_t* pbuf, int row, const float (&pa)[16], const float (&pb)[16]) {
  uint8_t* dst = pbuf + (row >> 3) * 512 + (row & 7) * 16;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float(&pv)[16] = t == 0 ? pa : pb;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint32_t h01 = f32x2_to_e4m3x2(pv[4 * q4], pv[4 * q4 + 1]);
      const uint32_t h23 = f32x2_to_e4m3x2(pv[4 * q4 + 2], pv[4 * q4 + 3]);
      const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
      hi[q4] = h01 | (h23 << 16);
      lo[q4] = f32x2_to_e4m3x2(kLoScale * (pv[4 * q4] - d01.x), kLoScale * (pv[4 * q4 + 1] - d01.y)) |
               (f32x2_to_e4m3x2(kLoScale * (pv[4 * q4 + 2] - d23.x), kLoScale * (pv[4 * q4 + 3] - d23.y)) << 16);
    }
    *reinterpret_cast<uint4*>(dst + 256 * t) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + 256 * t + 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Multiplies one token's 4 x 32 O columns of this thread's lane by alpha[head].
__device__ __forceinline__ void rescale_o_tok(uint32_t ob, int t, const float (&alpha)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[32];
    tmem_ld32(ob + 64 * mb + 32 * t, o);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j & 15]);
    tmem_st32(ob + 64 * mb + 32 * t, o);
  }
  tmem_wait_st();
}

// Epilogue of one token t of a piece: O (hi + lo/16) times f[head] to the bf16
// output or the token's fp32 partial slot.
__device__ __forceinline__ void store_o_tok(const Stage1Params& p, const Piece& pc, int t, uint32_t ob, int row,
                                            const float (&f)[16]) {
  const int64_t token = pc.token + t;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[32];
    tmem_ld32(ob + 64 * mb + 32 * t, o);
    tmem_wait_ld();
    const int dim = 128 * mb + row;
    if (pc.direct) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + token * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        dst[h * kDv] = __float2bfloat16_rn((__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h]);
    } else {
      float* dst = p.part_o + (pc.slot + t) * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        dst[h * kDv] = (__uint_as_float(o[h]) + __uint_as_float(o[16 + h]) * (1.0f / kLoScale)) * f[h];
    }
  }
}

// Reference max (lazy, see kMaxSlack), weights and row sums of one token for
// one tile; returns whether some head's reference moved.
__device__ __forceinline__ bool softmax_tok(const float* rm, const float (&x)[16], float (&m)[16], float (&l)[16],
                                            float (&alpha)[16], float (&pv)[16]) {
  bool grew = false;
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const float tm = fmaxf(fmaxf(rm[h], rm[16 + h]), fmaxf(rm[32 + h], rm[48 + h]));
    const bool up = tm > m[h] + kMaxSlack;
    alpha[h] = up ? fast_exp2(m[h] - tm) : 1.0f;
    grew |= up;
    m[h] = up ? tm : m[h];
  }
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    pv[h] = fast_exp2(x[h] - m[h]);
    l[h] = l[h] * alpha[h] + pv[h];
    pv[h] *= kPScale;
  }
  return grew;
}

__device__ void softmax_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  constexpr int kStages = L::kStages;
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = warp - 2;
  sx.row = 32 * (warp & 3) + lane;
  sx.lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  sx.gcount = 0;
  const float kvsc = __ldg(static_cast<const float*>(p.kv_scale));
  float* red_max = reinterpret_cast<float*>(cx.g + L::kOffRedMax);
  float* red_l = reinterpret_cast<float*>(cx.g + L::kOffRedL);
  const uint32_t obase = cx.tmem + sx.lane_base + L::kTmemO;

  PieceCursor ahead = cur;
  Piece pc, nxt;
  bool have = ahead.next(pc);
  if (!have) return;
  // rope of tiles 0 and 1 into registers, the first Q, tile 0 into the slot, tile 2 loads
  TileWalker rw;
  rw.init(cur);
  uint4 rb0[4], rb1[4];  // rope of the even / odd tile in flight
  load_rope(p, rw, sx.row, rb0);
  load_rope(p, rw, sx.row, rb1);
  float ca, cb;  // the first Q operand while those rope rows are in flight
  if (!setup_q2(p, cx, sx, pc, 0, kvsc, ca, cb)) return;
  store_rope(cx, sx, rb0);
  load_rope(p, rw, sx.row, rb0);
  uint32_t n = 0, k = 0;
  int tiles_left = count_tiles(cur) - 1;  // tiles of the CTA after the current one (for the rope slot)
  while (have) {
    const bool have_next = ahead.next(nxt);
    float ma[16], la[16], mb[16], lb[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      ma[h] = mb[h] = -INFINITY;
      la[h] = lb[h] = 0.f;
    }
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const int nr = min(kTileRows, pc.nrows - r0);
      const uint32_t s = n & 1u;
      if (!cx.wait(L::kSFull + s, (n >> 1) & 1u)) return;
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
      const bool valid = sx.row < nr && (r0 > 0 || sx.row >= pc.lead);
      float xa[16], xb[16];
      tc_fence_after();
      {
        uint32_t sr[32];
        tmem_ld32(cx.tmem + sx.lane_base + L::kSCols * s, sr);
        tmem_wait_ld();
        // columns 0-31: token A hi, lo; 32-63: token B hi, lo
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float v = (__uint_as_float(sr[h]) + __uint_as_float(sr[16 + h]) * (1.0f / kLoScale)) * ca;
          xa[h] = valid ? v : -INFINITY;
        }
        tmem_ld32(cx.tmem + sx.lane_base + L::kSCols * s + 32, sr);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float v = (__uint_as_float(sr[h]) + __uint_as_float(sr[16 + h]) * (1.0f / kLoScale)) * cb;
          xb[h] = valid ? v : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + s));
      float* rm = red_max + (n & 1u) * 128;  // [token][warp][head]
      {
        float wm[16];
        warp_max16(xa, wm);
        store16(rm + sx.wi * 16, wm, lane);
        warp_max16(xb, wm);
        store16(rm + 64 + sx.wi * 16, wm, lane);
      }
      if (!group_sync(cx, sx)) return;
      float alpha_a[16], pa[16], alpha_b[16], pb[16];
      const bool grew_a = softmax_tok(rm, xa, ma, la, alpha_a, pa);
      const bool grew_b = softmax_tok(rm + 64, xb, mb, lb, alpha_b, pb);
      // single P buffer: P.V(n-1) must be done (the commit that releases its stage)
      if (n >= 1 && !cx.wait(L::kKvEmpty + (n - 1) % L::kStages, ((n - 1) / L::kStages) & 1u)) return;
      put_p_row2(cx.g + L::kOffP, sx.row, pa, pb);
      if (!valid) {
        // rows outside the piece: zero their V bytes so P = 0 meets finite values
        uint8_t* vrow = cx.g + L::kOffKv + (n % kStages) * kStageBytes + sx.row * 128;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(vrow + ch * kChunkBytes + u * 16) = make_uint4(0, 0, 0, 0);
      }
      if (r0 > 0 && (grew_a || grew_b)) {
        // O of this piece is final for tile n-1: P.V(n-1) completed (waited above)
        tc_fence_after();
        if (grew_a) rescale_o_tok(obase, 0, alpha_a);
        if (grew_b) rescale_o_tok(obase, 1, alpha_b);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull));
      ++n;
    }

    // the next piece's q goes in while this piece's last PV runs
    float ca_next = ca, cb_next = cb;
    if (have_next && !setup_q2(p, cx, sx, nxt, k + 1, kvsc, ca_next, cb_next)) return;
    // l over the 128 rows, per head and token
    {
      const float wa = warp_reduce16<false>(la, lane);
      const float wb = warp_reduce16<false>(lb, lane);
      if ((lane & 1) == 0) {
        red_l[sx.wi * 16 + (lane >> 1)] = wa;
        red_l[64 + sx.wi * 16 + (lane >> 1)] = wb;
      }
    }
    if (!group_sync(cx, sx)) return;
    float fa[16], fb[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const float La = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
      const float Lb = red_l[64 + h] + red_l[80 + h] + red_l[96 + h] + red_l[112 + h];
      fa[h] = kvsc / (kPScale * La);
      fb[h] = kvsc / (kPScale * Lb);
      if (!pc.direct && sx.row == h) p.part_lse[pc.slot * kHeads + h] = ma[h] + fast_log2(La);
      if (!pc.direct && pc.ntok > 1 && sx.row == 16 + h) p.part_lse[(pc.slot + 1) * kHeads + h] = mb[h] + fast_log2(Lb);
    }
    if (!cx.wait(L::kOFull, k & 1u)) return;
    tc_fence_after();
    store_o_tok(p, pc, 0, obase, sx.row, fa);
    if (pc.ntok > 1) store_o_tok(p, pc, 1, obase, sx.row, fb);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty));
    if (!pc.direct && !finish_partial(p, cx, sx, pc)) return;
    pc = nxt;
    have = have_next;
    ca = ca_next;
    cb = cb_next;
    ++k;
  }
}

__global__ void __launch_bounds__(kThreads, 1) stage1_pair_kernel(const Stage1Params p,
                                                                  const __grid_constant__ CUtensorMap kvmap) {
  extern __shared__ uint8_t smem_raw[];
  Cx cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, 1, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cur.align8 = 1;  // the tiles of the single-token kernel
  if (warp == 0) {
    producer(cx, &kvmap, cur, lane);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer_polling(cx, cur);
    __syncwarp();
  } else if (warp < 6) {
    softmax_role(p, cx, cur, warp, lane);
  }
  cta_end(p, cx, 1);
}

static cudaError_t launch(const Stage1Params& p, cudaStream_t stream) {
  constexpr int kAlloc = L::kAlloc;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(stage1_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap map;
  e = make_kv_map(&map, p.kv, p.total_kv, kTileRows);
  if (e != cudaSuccess) return e;
  return launch_dependent(stage1_pair_kernel, p.num_splits, kThreads, kAlloc, stream, p, map);
}

}  // namespace pair
}  // namespace tc

cudaError_t launch_stage1_pair(const Stage1Params& p, cudaStream_t stream) {
  return tc::pair::launch(p, stream);
}

}  // namespace mla
