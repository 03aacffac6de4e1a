// Stage 1 for an fp8 (e4m3) KV cache and fp8 q (a8w8, or q quantised in the
// call) with the query tokens of a segment taken in groups of up to four that
// share one pass over the KV rows (multi-token decode, q_len > 2).
//
// Method: as the single-token tensor-core kernel (split-K flash decoding as in
// kernelbot-amd-mixed-mla-753817 `mla_flash_decode_stage1`, scores over all
// 576 dims, values the first 512, exp2-domain online softmax, normalised
// partials plus LSE). kernelbot-amd-mixed-mla-586148 `_flash_splitk` groups
// the q_len x 16 query rows of a segment against one pass over its KV rows;
// here a group holds four tokens:
//  * Q holds the four tokens' e4m3 codes (64 rows: token t, head h at row
//    16 t + h), so Q.K^T runs at N = 64 and P.V at N = 64: the tensor core
//    reads each 128-row KV tile once for four tokens;
//  * a tile comes in as five TMA boxes (the four 128-byte chunks of the V
//    dims and the rope bytes, the latter's box reaching past the 576-byte row
//    and filled with zeros there), into one of two 80 KB stages;
//  * tensor memory: S in 2 buffers x 64 columns, O in 4 blocks x 64 columns.
//    Four tokens' O with separate hi and lo accumulators would need all 512
//    columns, so the weights' lo part (P - hi, e4m3) goes into the same
//    accumulator as hi: two P.V UMMAs per k-step, one per part;
//  * eight softmax warps: warps 4-7 take tokens 0 and 1, warps 8-11 tokens
//    2 and 3, each with its own maxima, sums and barriers; a thread is a tile
//    row (its warp's tensor-memory lane quarter);
//  * registers: warpgroup 0 (TMA, MMA, two idle warps) gives registers to the
//    two softmax warpgroups (setmaxnreg), and all take the launch count back
//    before the end-of-CTA merge.
// A group with fewer than four tokens (the last of a segment) fills the
// missing ones with its first token and writes only its own.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace quad {

constexpr int kThreads = 384;
constexpr int kSoftWarp0 = 4;                    // warps 4-11: two softmax halves
constexpr int kBoxes = 5;                        // V chunks 0-3 and the rope box
constexpr int kStageBytes = kBoxes * kChunkBytes;  // 80 KB
constexpr int kStages = 2;
constexpr int kQRows = 64;
constexpr int kQChunk = kQRows * 128;            // 8 KB per 128-dim chunk
constexpr int kPPart = kTileRows * 64;           // 8 KB: one part (hi or lo) of P
constexpr uint32_t kSCols = 64;
constexpr uint32_t kTmO = 2 * kSCols;            // O: 4 blocks x 64 columns
constexpr uint32_t kLaunchRegs = 168, kAuxRegs = 88, kSoftRegs = 208;
static_assert(kAuxRegs * 128 + kSoftRegs * 256 == kLaunchRegs * kThreads, "register split");

struct L {
  static constexpr int kThreads = quad::kThreads;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + 5 * kQChunk;                  // [hi | lo], 8 KB each
  static constexpr int kOffRedMax = kOffP + 2 * kPPart;              // [2 buffers][4 tokens][4 warps][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * 4 * 16 * 4;   // [4 tokens][4 warps][16] f32
  static constexpr int kOffAmax = kOffRedL + 4 * 4 * 16 * 4;         // (bf16 q only; unused here)
  static constexpr int kOffMList = kOffAmax + 32;                    // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                   // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  enum {
    kKvFull = 0, kKvEmpty = 2, kSFull = 4, kSEmpty = 6, kPFull = 8, kPEmpty = 9, kQFull = 10, kQEmpty = 11,
    kOFull = 12, kOEmpty = 13, kGrp = 14 /* [half][2] */, kDrain = 18, kMerge = 19, kNumBars = 20
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
      mbar_init(cx.bar(kSEmpty + i), 8);
    }
    for (int i = 0; i < 4; ++i) mbar_init(cx.bar(kGrp + i), 4);
    mbar_init(cx.bar(kPFull), 8);
    mbar_init(cx.bar(kPEmpty), 1);
    mbar_init(cx.bar(kQFull), 8);
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kOFull), 1);
    mbar_init(cx.bar(kOEmpty), 8);
    mbar_init(cx.bar(kDrain), 1);
  }
};
using Cx = Ctx<L>;
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffQ % 1024 == 0 && L::kOffP % 1024 == 0 && kStageBytes % 1024 == 0, "operand alignment");
static_assert(L::kOffScan % 8 == 0 && L::kOffRedMax % 16 == 0, "scratch alignment");
static_assert(kTmO + 4 * 64 <= kTmemCols, "tensor memory");

// B operands. Q.K^T k-step ks: the Q rows of chunk ks / 4 (K-major, 128B
// swizzle). P.V k-step ks (32 rows): one part of P^T, 4 N-blocks of 16 columns
// (the tokens) 128 B apart, 8-row groups 512 B apart.
__device__ __forceinline__ uint64_t qk_desc_b4(uint32_t qbuf, int ks) {
  return smem_desc(qbuf + (ks >> 2) * kQChunk + (ks & 3) * 32, 16, 1024, kLayoutSw128);
}
__device__ __forceinline__ uint64_t pv_desc_b4(uint32_t ppart, int ks) {
  return smem_desc(ppart + ks * 2048, 512, 128, kLayoutNone);
}

// Warp 0 (one lane issues): the five boxes of each tile into stage
// (tile % 2) once the tile that used it last has been released by its P.V.
__device__ void producer(const Cx& cx, const CUtensorMap* map, PieceCursor cur, int lane) {
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
        for (int c = 0; c < kBoxes; ++c)
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

// Warp 1 (one thread): QK(n) into S[n % 2] and PV(n) into O, each issued as
// soon as its inputs are ready (a polling loop, not a fixed order): with two
// stages, a P.V must not wait behind the landing of the next tile, whose load
// starts only when the P.V before it has released its stage. O has one
// buffer: the first P.V of piece k waits until the epilogue of piece k-1 has
// read O.
__device__ void issue_qk(const Cx& cx, uint32_t n, const TileMeta& t) {
  constexpr uint32_t id_qk = umma_idesc(128, kSCols, 0, 0, false, false);
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + (n % kStages) * kStageBytes;
  const uint32_t sbuf = cx.tmem + kSCols * (n & 1u);
  const uint32_t qbuf = cx.s + L::kOffQ;
#pragma unroll
  for (int ks = 0; ks < 18; ++ks)  // the 512 V dims, then the 64 rope dims (box 4)
    umma_e4m3(sbuf, qk_desc_a(stage, ks), qk_desc_b4(qbuf, ks), id_qk, ks > 0 ? 1u : 0u);
  umma_commit(cx.bar(L::kSFull + (n & 1u)));
  if (t.last) umma_commit(cx.bar(L::kQEmpty));
}

__device__ void issue_pv(const Cx& cx, uint32_t n, const TileMeta& t) {
  constexpr uint32_t id_pv = umma_idesc(128, 64, 0, 0, true, true);
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + (n % kStages) * kStageBytes;
  const uint32_t phi = cx.s + L::kOffP, plo = phi + kPPart;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t a = pv_desc_a(stage, mb, ks);
      umma_e4m3(cx.tmem + kTmO + 64 * mb, a, pv_desc_b4(phi, ks), id_pv, (ks > 0 || !t.first) ? 1u : 0u);
      umma_e4m3(cx.tmem + kTmO + 64 * mb, a, pv_desc_b4(plo, ks), id_pv, 1u);
    }
  umma_commit(cx.bar(L::kKvEmpty + (n % kStages)));
  umma_commit(cx.bar(L::kPEmpty));
  if (t.last) umma_commit(cx.bar(L::kOFull));
}

// Phases tested below cannot run ahead by two: stage s is refilled only after
// the P.V of its tile, the P buffer only after its P.V, the S buffer only
// after the Q.K^T that read it back, and the next Q only after the last Q.K^T
// of the piece.
__device__ void mma_issuer(const Cx& cx, PieceCursor cur) {
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
        issue_pv(cx, pi, t);
        ++pi;
        wp.next(row, mp);
        progressed = true;
      }
    }
    if (qi < n && mbar_test_wait(cx.bar(L::kKvFull + qi % kStages), (qi / kStages) & 1u) &&
        (qi < 2 || mbar_test_wait(cx.bar(L::kSEmpty + (qi & 1u)), ((qi - 2) >> 1) & 1u))) {
      const TileMeta t = TileMeta::unpack(mq);
      if (!t.first || mbar_test_wait(cx.bar(L::kQFull), t.k & 1u)) {
        issue_qk(cx, qi, t);
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
// Warps 4-11: half hf = (warp - 4) / 4 takes tokens 2 hf and 2 hf + 1 of the
// group. Thread = tile row = tensor-memory lane (32 * (warp % 4) + lane).

// Barrier among the four warps of one half (two alternating mbarriers each).
__device__ __forceinline__ bool half_sync(const Cx& cx, SoftmaxCtx& sx, int hf) {
  const uint32_t k = sx.gcount & 1u, par = (sx.gcount >> 1) & 1u;
  ++sx.gcount;
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kGrp + 2 * hf + k));
  return cx.wait(L::kGrp + 2 * hf + k, par);
}

// The q codes of this half's two tokens into Q rows 16 j.. (j = 2 hf + t); a
// token past the group's count repeats its first token. Both halves arrive on
// kQFull. Returns false on abort.
template <int QF>
__device__ bool setup_q4(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, int hf, const Piece& pc, uint32_t kk,
                         float kvsc, float (&c)[2]) {
  if (kk >= 1 && !cx.wait(L::kQEmpty, (kk - 1) & 1u)) return false;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int j = 2 * hf + t;
    c[t] = fill_q<L, QF, kQChunk, false>(p, cx, sx, pc.token + (j < pc.ntok ? j : 0), 16 * j, kk, kvsc);
    if (c[t] < 0.f) return false;
  }
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kQFull));
  return true;
}

// Reference max (lazy, see kMaxSlack), weights and row sums of one token for
// one tile; rm = the token's [4 warps][16 heads] tile maxima. Returns whether
// some head's reference moved.
__device__ __forceinline__ bool softmax_tok(const float* rm, const float (&x)[16], float (&m)[16], float (&l)[16],
                                            float (&alpha)[16], float (&pv)[16]) {
  bool grew = false;
  const float4* rm4 = reinterpret_cast<const float4*>(rm);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 a = rm4[q], b = rm4[4 + q], c = rm4[8 + q], d = rm4[12 + q];
    const float t4[4] = {fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x)), fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y)),
                         fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z)), fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w))};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = 4 * q + e;
      const bool up = t4[e] > m[h] + kMaxSlack;
      alpha[h] = up ? fast_exp2(m[h] - t4[e]) : 1.0f;
      grew |= up;
      m[h] = up ? t4[e] : m[h];
    }
  }
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    pv[h] = fast_exp2(x[h] - m[h]);
    l[h] = l[h] * alpha[h] + pv[h];
    pv[h] *= kPScale;
  }
  return grew;
}

// One row's weights of token j (16 heads, times kPScale) as e4m3 hi into the
// hi part of P and the unscaled e4m3 remainder into the lo part (both parts
// go into the same O accumulator).
__device__ __forceinline__ void put_p_tok(uint8_t* pbuf, int row, int j, const float (&pv)[16]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t h01 = f32x2_to_e4m3x2(pv[4 * q4], pv[4 * q4 + 1]);
    const uint32_t h23 = f32x2_to_e4m3x2(pv[4 * q4 + 2], pv[4 * q4 + 3]);
    const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
    hi[q4] = h01 | (h23 << 16);
    lo[q4] = f32x2_to_e4m3x2(pv[4 * q4] - d01.x, pv[4 * q4 + 1] - d01.y) |
             (f32x2_to_e4m3x2(pv[4 * q4 + 2] - d23.x, pv[4 * q4 + 3] - d23.y) << 16);
  }
  uint8_t* d = pbuf + (row >> 3) * 512 + j * 128 + (row & 7) * 16;
  *reinterpret_cast<uint4*>(d) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(d + kPPart) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Multiplies this half's O columns (tokens 2 hf, 2 hf + 1) of this thread's
// lane by alpha[token][head]; ob = lane base + kTmO + 32 hf.
__device__ __forceinline__ void rescale_o_half(uint32_t ob, const float (&a0)[16], const float (&a1)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[32];
    tmem_ld32(ob + 64 * mb, o);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j] = __float_as_uint(__uint_as_float(o[j]) * a0[j]);
      o[16 + j] = __float_as_uint(__uint_as_float(o[16 + j]) * a1[j]);
    }
    tmem_st32(ob + 64 * mb, o);
  }
  tmem_wait_st();
}

// Epilogue of token j of a piece: O times f[head] to the bf16 output or the
// token's fp32 partial slot; ob = lane base + kTmO.
__device__ __forceinline__ void store_o_tok(const Stage1Params& p, const Piece& pc, int j, uint32_t ob, int row,
                                            const float (&f)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[16];
    tmem_ld16(ob + 64 * mb + 16 * j, o);
    tmem_wait_ld();
    const int dim = 128 * mb + row;
    if (pc.direct) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(pc.token + j) * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h) dst[h * kDv] = __float2bfloat16_rn(__uint_as_float(o[h]) * f[h]);
    } else {
      float* dst = p.part_o + (pc.slot + j) * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h) dst[h * kDv] = __uint_as_float(o[h]) * f[h];
    }
  }
}

// After a half wrote its tokens' partials of a split group: publish and count
// them; a token whose count completes goes on the end-of-CTA merge list (the
// two halves append to it with a shared-memory atomic). The half barrier
// orders its 128 threads' writes before the leader's gpu-scope fence, which is
// cumulative. Returns false on abort.
__device__ __forceinline__ bool finish_half(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, int hf,
                                            const Piece& pc) {
  if (!half_sync(cx, sx, hf)) return false;
  if (sx.wi == 0 && sx.lane == 0) {
    __threadfence();
    const int64_t P = cx.parts;
    const int64_t c0 = part_of_row(pc.tok_vs, cx.total, P), c1 = part_of_row(pc.tok_vs + pc.kvlen - 1, cx.total, P);
    MergeList* ml = reinterpret_cast<MergeList*>(cx.g + L::kOffMList);
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * hf + t;
      if (j >= pc.ntok) break;
      const uint32_t arrived = atomicAdd(p.tok_cnt + pc.token + j, 1u) + 1u;
      // cooperative merge: every CTA of the token lists it; otherwise the one that completes its count
      if (p.coop_merge || arrived == static_cast<uint32_t>(c1 - c0 + 1)) {
        const uint32_t e = atomicAdd(&ml->n, 1u);
        if (e < kMergeMax) {
          ml->token[e] = pc.token + j;
          ml->c0[e] = static_cast<int32_t>(c0);
          ml->c1[e] = static_cast<int32_t>(c1);
        }
      }
    }
  }
  return true;
}

template <int QF>
__device__ void softmax_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  const int hf = (warp - kSoftWarp0) >> 2;
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = (warp - kSoftWarp0) & 3;
  sx.row = 32 * (warp & 3) + lane;
  sx.lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  sx.gcount = 0;
  const float kvsc = __ldg(static_cast<const float*>(p.kv_scale));
  float* red_max = reinterpret_cast<float*>(cx.g + L::kOffRedMax);
  float* red_l = reinterpret_cast<float*>(cx.g + L::kOffRedL);
  const uint32_t obase = cx.tmem + sx.lane_base + kTmO;

  PieceCursor ahead = cur;
  Piece pc, nxt;
  bool have = ahead.next(pc);
  if (!have) return;
  float c[2];
  if (!setup_q4<QF>(p, cx, sx, hf, pc, 0, kvsc, c)) return;
  uint32_t n = 0, k = 0;
  while (have) {
    const bool have_next = ahead.next(nxt);
    float m[2][16], l[2][16];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m[t][h] = -INFINITY;
        l[t][h] = 0.f;
      }
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const int nr = min(kTileRows, pc.nrows - r0);
      const uint32_t s = n & 1u;
      if (!cx.wait(L::kSFull + s, (n >> 1) & 1u)) return;
      const bool valid = sx.row < nr && (r0 > 0 || sx.row >= pc.lead);
      float x[2][16];
      tc_fence_after();
      {
        uint32_t sr[32];  // columns 32 hf..: this half's two tokens
        tmem_ld32(cx.tmem + sx.lane_base + kSCols * s + 32 * hf, sr);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          x[0][h] = valid ? __uint_as_float(sr[h]) * c[0] : -INFINITY;
          x[1][h] = valid ? __uint_as_float(sr[16 + h]) * c[1] : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + s));
      float* rm = red_max + (n & 1u) * 256;  // [token][warp][head]
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float wm[16];
        warp_max16(x[t], wm);
        store16(rm + (2 * hf + t) * 64 + sx.wi * 16, wm, lane);
      }
      if (!half_sync(cx, sx, hf)) return;
      // single P buffer: P.V(n-1) must be done
      if (n >= 1 && !cx.wait(L::kPEmpty, (n - 1) & 1u)) return;
      float alpha[2][16];
      bool grew = false;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float pv[16];
        grew |= softmax_tok(rm + (2 * hf + t) * 64, x[t], m[t], l[t], alpha[t], pv);
        put_p_tok(cx.g + L::kOffP, sx.row, 2 * hf + t, pv);
      }
      if (!valid && hf == 0) {
        // rows outside the piece: zero their V bytes so P = 0 meets finite values
        uint8_t* vrow = cx.g + L::kOffKv + (n % kStages) * kStageBytes + sx.row * 128;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(vrow + ch * kChunkBytes + u * 16) = make_uint4(0, 0, 0, 0);
      }
      if (r0 > 0 && grew) {
        // O of this piece is final for tile n-1: P.V(n-1) completed (waited above)
        tc_fence_after();
        rescale_o_half(obase + 32 * hf, alpha[0], alpha[1]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull));
      ++n;
    }

    // the next piece's q goes in while this piece's last P.V runs
    float c_next[2] = {c[0], c[1]};
    if (have_next && !setup_q4<QF>(p, cx, sx, hf, nxt, k + 1, kvsc, c_next)) return;
    // l over the 128 rows, per head and token
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float w = warp_reduce16<false>(l[t], lane);
      if ((lane & 1) == 0) red_l[(2 * hf + t) * 64 + sx.wi * 16 + (lane >> 1)] = w;
    }
    if (!half_sync(cx, sx, hf)) return;
    float f[2][16];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * hf + t;
      const float* rl = red_l + j * 64;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float Lh = rl[h] + rl[16 + h] + rl[32 + h] + rl[48 + h];
        f[t][h] = kvsc / (kPScale * Lh);
        if (!pc.direct && j < pc.ntok && sx.row == 16 * t + h)
          p.part_lse[(pc.slot + j) * kHeads + h] = m[t][h] + fast_log2(Lh);
      }
    }
    if (!cx.wait(L::kOFull, k & 1u)) return;
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (2 * hf + t < pc.ntok) store_o_tok(p, pc, 2 * hf + t, obase, sx.row, f[t]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty));
    if (!pc.direct && !finish_half(p, cx, sx, hf, pc)) return;
    pc = nxt;
    have = have_next;
    c[0] = c_next[0];
    c[1] = c_next[1];
    ++k;
  }
}

template <int QF>
__global__ void __launch_bounds__(kThreads, 1) stage1_quad_kernel(const Stage1Params p,
                                                                  const __grid_constant__ CUtensorMap kvmap) {
  extern __shared__ uint8_t smem_raw[];
  Cx cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, 1, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cur.align8 = 1;  // the tiles of the single-token kernel
  if (warp < kSoftWarp0) {
    setmaxnreg_dec<kAuxRegs>();
    if (warp == 0) {
      producer(cx, &kvmap, cur, lane);
    } else if (warp == 1) {
      if (lane == 0) mma_issuer(cx, cur);
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kSoftRegs>();  // granted once warpgroup 0 has made its decrease (unconditional)
    softmax_role<QF>(p, cx, cur, warp, lane);
    setmaxnreg_dec<kLaunchRegs>();
  }
  // Both softmax warpgroups returned their extra registers before this
  // barrier: the increase below is always granted at once.
  __syncthreads();
  if (warp < kSoftWarp0) setmaxnreg_inc<kLaunchRegs>();
  cta_end(p, cx, 1);
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
    e = cudaFuncGetAttributes(&fa, stage1_quad_kernel<QF>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(stage1_quad_kernel<QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap map;
  e = make_kv_map(&map, p.kv, p.total_kv, kTileRows);
  if (e != cudaSuccess) return e;
  return launch_dependent(stage1_quad_kernel<QF>, p.num_splits, kThreads, L::kAlloc, stream, p, map);
}

}  // namespace quad
}  // namespace tc

cudaError_t launch_stage1_quad(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (q_fmt == kQBf16Quant) return tc::quad::launch_q<kQBf16Quant>(p, stream);
  if (q_fmt == kQFp8) return tc::quad::launch_q<kQFp8>(p, stream);
  return cudaErrorInvalidValue;  // bf16 q needs hi + lo rows: not in a group of four
}

}  // namespace mla
