// Stage 1 for an fp8 (e4m3) KV cache and fp8 q (a8w8, or q quantised in the
// call) with the query tokens of a segment taken in pairs that share one pass
// over the KV rows, the softmax of the two tokens run by two groups of warps.
//
// Method: as the single-token tensor-core kernel (split-K flash decoding as in
// kernelbot-amd-mixed-mla-753817 `mla_flash_decode_stage1`, scores over all
// 576 dims, values the first 512, exp2-domain online softmax, normalised
// partials plus LSE), two tokens of a segment against one pass over its rows
// as the q_len x 16 query rows of kernelbot-amd-mixed-mla-586148
// `_flash_splitk` share one. The operands are those of the token-pair kernel
// with fp8 q:
//  * Q is 32 rows (token A codes, token B codes; no lo rows), so Q.K^T runs at
//    N = 32; P holds both tokens' hi and lo weights, so P.V runs at N = 64;
//  * three 64 KB V stages; the rope operand sits in tensor memory, written by
//    the softmax threads of token A and read as A by the rope UMMAs;
//  * tensor memory: S 2 x 32 columns, O 4 blocks x 64 columns (A hi, A lo,
//    B hi, B lo), rope 16 columns.
// The softmax, which bounds the token-pair kernel (one warp per sub-partition
// doing both tokens' maxima, weights and rescales), is split: warps 4-7 take
// token A and warps 8-11 token B, each group with its own maxima, sums and
// barriers, two warps per sub-partition. Warpgroup 0 (TMA, MMA, two warps
// that join only the merge) gives registers to the two softmax warpgroups
// (setmaxnreg). A token's arithmetic is the token-pair kernel's, step by step;
// the compiled code may still round an operation differently (a contraction
// into a fused multiply-add), so the two can differ by one bf16 step on a few
// outputs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace duo {

constexpr int kThreads = 384;
constexpr int kSoftWarp0 = 4;                     // warps 4-7: token A, warps 8-11: token B
constexpr int kStages = 3;
constexpr int kStageBytes = kVBytes;              // 64 KB: the 512 V dims of a tile
constexpr int kQRows = 32;
constexpr int kQChunk = kQRows * 128;             // 4 KB per 128-dim chunk
constexpr int kPBytes2 = kTileRows * 64;          // [row group][A hi | A lo | B hi | B lo][8 rows][16 heads]
constexpr uint32_t kSCols = kQRows;
constexpr uint32_t kTmO = 2 * kSCols;             // O: 4 blocks x 64 columns
constexpr uint32_t kTmRope = kTmO + 256;          // rope operand, 16 columns
constexpr uint32_t kLaunchRegs = 168, kAuxRegs = 88, kSoftRegs = 208;
static_assert(kAuxRegs * 128 + kSoftRegs * 256 == kLaunchRegs * kThreads, "register split");

struct L {
  static constexpr int kThreads = duo::kThreads;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + 5 * kQChunk;
  static constexpr int kOffRedMax = kOffP + kPBytes2;                // [2 buffers][2 tokens][4 warps][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 2 * 4 * 16 * 4;   // [2 tokens][4 warps][16] f32
  static constexpr int kOffAmax = kOffRedL + 2 * 4 * 16 * 4;         // (bf16 q only; unused here)
  static constexpr int kOffMList = kOffAmax + 32;                    // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                   // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  enum {
    kKvFull = 0, kKvEmpty = 3, kSFull = 6, kSEmpty = 8, kRopeFull = 10, kPFull = 11, /* 12 unused */ kQFull = 13,
    kQEmpty = 14, kOFull = 15, kOEmpty = 16, kGrp = 17 /* [half][2] */, kDrain = 21, kMerge = 22, kNumBars = 23
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
    mbar_init(cx.bar(kRopeFull), 4);  // token A's warps write the rope operand
    mbar_init(cx.bar(kPFull), 8);
    mbar_init(cx.bar(kQFull), 8);
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kOFull), 1);
    mbar_init(cx.bar(kOEmpty), 8);
    mbar_init(cx.bar(kDrain), 1);
  }
};
using Cx = Ctx<L>;
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffQ % 1024 == 0 && L::kOffP % 1024 == 0, "operand alignment");
static_assert(L::kOffScan % 8 == 0 && L::kOffRedMax % 16 == 0, "scratch alignment");
static_assert(kTmRope + 16 <= kTmemCols, "tensor memory");

// B operands. Q.K^T k-step ks: the Q rows of chunk ks / 4 (K-major, 128B
// swizzle). P.V k-step ks (32 rows): P^T, 4 N-blocks of 16 columns 128 B apart,
// 8-row groups 512 B apart.
__device__ __forceinline__ uint64_t qk_desc_b_duo(uint32_t qbuf, int ks) {
  return smem_desc(qbuf + (ks >> 2) * kQChunk + (ks & 3) * 32, 16, 1024, kLayoutSw128);
}
__device__ __forceinline__ uint64_t pv_desc_b_duo(uint32_t pbuf, int ks) {
  return smem_desc(pbuf + ks * 2048, 512, 128, kLayoutNone);
}

// Warp 0: the V dims of each tile, four 128-row x 128-byte boxes, into stage
// (tile % 3) once the tile three back has been released by its P.V.
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
      umma_e4m3(cx.tmem + kTmO + 64 * mb, pv_desc_a(stage, mb, ks), pv_desc_b_duo(pbuf, ks), id_pv,
                (ks > 0 || !t.first) ? 1u : 0u);
  umma_commit(cx.bar(L::kKvEmpty + (t.n % kStages)));
  if (t.last) umma_commit(cx.bar(L::kOFull));
  return true;
}

__device__ void mma_issuer(const Cx& cx, PieceCursor cur) {
  constexpr uint32_t id_qk = umma_idesc(128, kSCols, 0, 0, false, false);
  Piece pc;
  uint32_t n = 0, k = 0;
  PendingPV pend{0, 0, false, false, false};
  bool ok = true;
  while (ok && cur.next(pc)) {
    if (!cx.wait(L::kQFull, k & 1u)) break;
    const uint32_t qbuf = cx.s + L::kOffQ;
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n & 1u, st = n % kStages;
      if (!cx.wait(L::kKvFull + st, (n / kStages) & 1u) || !cx.wait(L::kRopeFull, n & 1u) ||
          (n >= 2 && !cx.wait(L::kSEmpty + s, ((n >> 1) - 1) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t stage = cx.s + L::kOffKv + st * kStageBytes;
      const uint32_t sbuf = cx.tmem + kSCols * s;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)  // the 512 V dims, from the stage
        umma_e4m3(sbuf, qk_desc_a(stage, ks), qk_desc_b_duo(qbuf, ks), id_qk, ks > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)  // the 64 rope dims, A from tensor memory
        umma_e4m3_ta(sbuf, cx.tmem + kTmRope + 8 * ks, qk_desc_b_duo(qbuf, 16 + ks), id_qk, 1u);
      umma_commit(cx.bar(L::kSFull + s));
      const bool last = r0 + kTileRows >= pc.nrows;
      if (last) umma_commit(cx.bar(L::kQEmpty));
      if (pend.valid && !issue_pv(cx, pend)) {
        ok = false;
        break;
      }
      pend = PendingPV{n, k, r0 == 0, last, true};
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
// Warps 4-11: group hf = (warp - 4) / 4 takes token hf of the pair. Thread =
// tile row = tensor-memory lane (32 * (warp % 4) + lane).

__device__ __forceinline__ bool half_sync(const Cx& cx, SoftmaxCtx& sx, int hf) {
  const uint32_t k = sx.gcount & 1u, par = (sx.gcount >> 1) & 1u;
  ++sx.gcount;
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kGrp + 2 * hf + k));
  return cx.wait(L::kGrp + 2 * hf + k, par);
}

// Rope dims (bytes 512..575) of one tile row into registers; rows past the
// end of the cache read as zero.
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

// One row's rope bytes into its 16 tensor-memory columns, handed to the MMA warp.
__device__ __forceinline__ void store_rope(const Cx& cx, const SoftmaxCtx& sx, const uint4 (&r)[4]) {
  const uint32_t w[16] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w,
                          r[2].x, r[2].y, r[2].z, r[2].w, r[3].x, r[3].y, r[3].z, r[3].w};
  tmem_st16(cx.tmem + sx.lane_base + kTmRope, w);
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kRopeFull));
}

// The q codes of token hf of the pair into Q rows 16 hf..; a one-token pair
// loads its token into both halves. Returns false on abort.
template <int QF>
__device__ bool setup_q1(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, int hf, const Piece& pc, uint32_t kk,
                         float kvsc, float& c) {
  if (kk >= 1 && !cx.wait(L::kQEmpty, (kk - 1) & 1u)) return false;
  c = fill_q<L, QF, kQChunk, false>(p, cx, sx, pc.token + (hf < pc.ntok ? hf : 0), 16 * hf, kk, kvsc);
  if (c < 0.f) return false;
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kQFull));
  return true;
}

// Reference max (lazy, see kMaxSlack), weights and row sums of the token for
// one tile; rm = its [4 warps][16 heads] tile maxima. Returns whether some
// head's reference moved.
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

// One row of token t's weights (16 heads, times kPScale) as hi/lo e4m3 into
// the P operand's blocks 2t (hi) and 2t + 1 (lo, times kLoScale).
__device__ __forceinline__ void put_p_tok(uint8_t* pbuf, int row, int t, const float (&pv)[16]) {
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
  uint8_t* dst = pbuf + (row >> 3) * 512 + (row & 7) * 16 + 256 * t;
  *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(dst + 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Multiplies token t's 4 x 32 O columns of this thread's lane by alpha[head].
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

// Epilogue of token t of a piece: O (hi + lo / kLoScale) times f[head] to the
// bf16 output or the token's fp32 partial slot.
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

// After a group wrote its token's partial of a split pair: publish it and
// count it; with the cooperative merge every CTA of the token lists it, else
// the one that completes the count (the two groups append with a
// shared-memory atomic). Returns false on abort.
__device__ __forceinline__ bool finish_half(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, int hf,
                                            const Piece& pc) {
  if (!half_sync(cx, sx, hf)) return false;
  if (sx.wi == 0 && sx.lane == 0 && hf < pc.ntok) {
    __threadfence();
    const int64_t P = cx.parts;
    const int64_t c0 = part_of_row(pc.tok_vs, cx.total, P), c1 = part_of_row(pc.tok_vs + pc.kvlen - 1, cx.total, P);
    MergeList* ml = reinterpret_cast<MergeList*>(cx.g + L::kOffMList);
    const uint32_t arrived = atomicAdd(p.tok_cnt + pc.token + hf, 1u) + 1u;
    if (p.coop_merge || arrived == static_cast<uint32_t>(c1 - c0 + 1)) {
      const uint32_t e = atomicAdd(&ml->n, 1u);
      if (e < kMergeMax) {
        ml->token[e] = pc.token + hf;
        ml->c0[e] = static_cast<int32_t>(c0);
        ml->c1[e] = static_cast<int32_t>(c1);
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
  // token A's group: rope of tiles 0 and 1 into registers, the first Q, tile 0
  // into tensor memory, tile 2 loads
  TileWalker rw;
  rw.init(cur);
  uint4 rb0[4], rb1[4];  // rope of the even / odd tile in flight
  if (hf == 0) {
    load_rope(p, rw, sx.row, rb0);
    load_rope(p, rw, sx.row, rb1);
  }
  float c;
  if (!setup_q1<QF>(p, cx, sx, hf, pc, 0, kvsc, c)) return;
  if (hf == 0) {
    store_rope(cx, sx, rb0);
    load_rope(p, rw, sx.row, rb0);
  }
  uint32_t n = 0, k = 0;
  int tiles_left = count_tiles(cur) - 1;  // tiles of the CTA after the current one (for the rope operand)
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
      if (!cx.wait(L::kSFull + s, (n >> 1) & 1u)) return;
      // Q.K^T(n) is done: the rope operand takes tile n+1, its registers tile n+3
      if (hf == 0 && tiles_left > 0) {
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
      float x[16];
      tc_fence_after();
      {
        uint32_t sr[16];  // columns 16 hf..: this group's token
        tmem_ld16(cx.tmem + sx.lane_base + kSCols * s + 16 * hf, sr);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) x[h] = valid ? __uint_as_float(sr[h]) * c : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + s));
      float* rm = red_max + (n & 1u) * 128 + 64 * hf;  // [warp][head] of this token
      {
        float wm[16];
        warp_max16(x, wm);
        store16(rm + sx.wi * 16, wm, lane);
      }
      if (!half_sync(cx, sx, hf)) return;
      float alpha[16], pv[16];
      const bool grew = softmax_tok(rm, x, m, l, alpha, pv);
      // single P buffer: P.V(n-1) must be done (the commit that releases its stage)
      if (n >= 1 && !cx.wait(L::kKvEmpty + (n - 1) % kStages, ((n - 1) / kStages) & 1u)) return;
      put_p_tok(cx.g + L::kOffP, sx.row, hf, pv);
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
        rescale_o_tok(obase, hf, alpha);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull));
      ++n;
    }

    // the next piece's q goes in while this piece's last P.V runs
    float c_next = c;
    if (have_next && !setup_q1<QF>(p, cx, sx, hf, nxt, k + 1, kvsc, c_next)) return;
    // l over the 128 rows, per head
    {
      const float w = warp_reduce16<false>(l, lane);
      if ((lane & 1) == 0) red_l[64 * hf + sx.wi * 16 + (lane >> 1)] = w;
    }
    if (!half_sync(cx, sx, hf)) return;
    float f[16];
    {
      const float* rl = red_l + 64 * hf;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float Lh = rl[h] + rl[16 + h] + rl[32 + h] + rl[48 + h];
        f[h] = kvsc / (kPScale * Lh);
        if (!pc.direct && hf < pc.ntok && sx.row == h) p.part_lse[(pc.slot + hf) * kHeads + h] = m[h] + fast_log2(Lh);
      }
    }
    if (!cx.wait(L::kOFull, k & 1u)) return;
    tc_fence_after();
    if (hf < pc.ntok) store_o_tok(p, pc, hf, obase, sx.row, f);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty));
    if (!pc.direct && !finish_half(p, cx, sx, hf, pc)) return;
    pc = nxt;
    have = have_next;
    c = c_next;
    ++k;
  }
}

template <int QF>
__global__ void __launch_bounds__(kThreads, 1) stage1_duo_kernel(const Stage1Params p,
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
    e = cudaFuncGetAttributes(&fa, stage1_duo_kernel<QF>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(stage1_duo_kernel<QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap map;
  e = make_kv_map(&map, p.kv, p.total_kv, kTileRows);
  if (e != cudaSuccess) return e;
  return launch_dependent(stage1_duo_kernel<QF>, p.num_splits, kThreads, L::kAlloc, stream, p, map);
}

}  // namespace duo
}  // namespace tc

cudaError_t launch_stage1_duo(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (q_fmt == kQBf16Quant) return tc::duo::launch_q<kQBf16Quant>(p, stream);
  if (q_fmt == kQFp8) return tc::duo::launch_q<kQFp8>(p, stream);
  return cudaErrorInvalidValue;  // bf16 q takes the token-pair kernel
}

}  // namespace mla
