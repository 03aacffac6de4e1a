// Stage 1 of split-K MLA decode for a bf16 KV cache on the tcgen05 tensor
// cores (kind::f16, bf16 x bf16 -> fp32).
//
// Method: split-K flash decoding as in kernelbot-amd-mixed-mla-753817
// (`mla_flash_decode_stage1`), with the arithmetic of the bf16 baseline of
// kernelbot-amd-mixed-mla-675627 ("Baseline: bf16 Q + bf16 KV"): scores over
// all 576 dims, values the first 512, online softmax in the exp2 domain,
// normalised partial output plus LSE per split.
//
// GB300 design:
//  * Rows of KV are the MMA M dimension (M = 128), the 16 heads are N = 16:
//      S^T[row, head]  = K[row, 0:576] . Q^T         (A = KV tile, K-major)
//      O^T[dim, head] += V^T[dim, rows] . P^T       (A = the same tile read
//                                                    MN-major, no transpose)
//    bf16 needs no hi/lo split: q, K, V and the softmax weights P are all
//    bf16 operands (P rounded to bf16, 8 significant bits).
//  * A 128-row tile is nine 128-row x 128-byte TMA boxes (64 dims each, 128B
//    swizzle): 144 KB, one buffer. Each box has its own full/empty barriers:
//    the rope box is released once the four Q.K^T UMMAs that read it are
//    done, the V boxes two at a time as P.V finishes each 128-dim block, so
//    the next tile's boxes stream in behind them; Q.K^T takes each box as it
//    lands (rope box first).
//  * Warp 0 issues the TMA loads, warp 1 (one thread) the UMMAs and owns
//    tensor memory, warps 2-5 (thread = tile row = tensor-memory lane) stage
//    q into the B operand, run the online softmax and the epilogue.
//  * G query tokens of a segment (multi-token decode, G = 1 or 2) share each
//    pass over its KV rows: Q holds 16 G rows (token t's heads at rows
//    16 t ..), so Q.K^T and P.V run at N = 16 G and the tile is read once for
//    the G tokens. Each token's arithmetic is that of G = 1.
//  * Every mbarrier wait is bounded; on a timeout the CTA stops issuing work,
//    lets in-flight copies and MMAs finish, frees tensor memory and returns.
#include <cuda.h>

#include "mla_tc_common.cuh"

namespace mla {
namespace tc {
namespace bf {

constexpr int kThreads = 192;               // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kBoxes = 9;                   // 64-dim boxes of a tile: 8 V + 1 rope
constexpr int kRopeBox = 8;
constexpr int kBoxBytes = kTileRows * 128;  // 16 KB
constexpr int kTileBytes = kBoxes * kBoxBytes;  // 144 KB
// Lazy rescaling: a head's reference max moves only when a tile's max exceeds
// it by more than this (log2 units), so bf16 weights stay below 2^8.
constexpr float kMaxSlackBf = 8.0f;

// Layout for G tokens per pass.
template <int G>
struct LB {
  static constexpr int kThreads = bf::kThreads;
  static constexpr int kN = 16 * G;                      // UMMA N: the heads of the G tokens
  static constexpr int kQBoxBytes = kN * 128;            // q of one 64-dim box: kN rows x 128 B
  static constexpr int kQBytes = kBoxes * kQBoxBytes;
  static constexpr int kPBytes = kTileRows * 32 * G;     // [row group 16][token][head half 2][8 rows][16 B]
  // tensor-memory columns: S in 2 x kN, O^T in 2 pieces x (4 blocks x kN)
  static constexpr uint32_t kTmS = 0, kTmO = 2 * kN;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kTileBytes;
  static constexpr int kOffP = kOffQ + kQBytes;                    // 2 buffers
  static constexpr int kOffRedMax = kOffP + 2 * kPBytes;           // [2 buffers][G tokens][4 warps][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * G * 4 * 16 * 4; // [G][4][16] f32
  static constexpr int kOffAmax = kOffRedL + G * 4 * 16 * 4;       // [4] u32 (unused by bf16 q)
  static constexpr int kOffMList = kOffAmax + 16;                  // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                  // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  enum {
    kKvFull = 0, kKvEmpty = 9, kSFull = 18, kSEmpty = 20, kPFull = 22, kPvDone = 24, kQFull = 26, kQEmpty = 27,
    kOFull = 28, kOEmpty = 30, kGrp = 32, kDrain = 34, kMerge = 35, kNumBars = 36
  };
  static constexpr int kMergeBytes = kTileBytes;  // the tile buffer holds partials for the end-of-CTA merge
  static constexpr int kOffSlot = kOffBars + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 8;
  static constexpr int kBytes = kOffAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;
  template <class C>
  __device__ static void init_barriers(const C& cx) {
    for (int i = 0; i < kBoxes; ++i) {
      mbar_init(cx.bar(kKvFull + i), 1);
      mbar_init(cx.bar(kKvEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
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
  static_assert(kTmO + 2 * 4 * kN <= kTmemCols, "tensor memory");
};
static_assert(LB<1>::kAlloc <= 227 * 1024 && LB<2>::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(LB<1>::kOffQ % 1024 == 0 && LB<1>::kOffP % 1024 == 0 && LB<2>::kOffP % 1024 == 0 &&
                  LB<1>::kOffBars % 8 == 0 && LB<2>::kOffBars % 8 == 0,
              "operand alignment");
template <int G>
using CxB = Ctx<LB<G>>;

// Box order of a tile: the rope box first (its slot frees earliest).
__device__ __forceinline__ int box_at(int j) { return j == 0 ? kRopeBox : j - 1; }

// ---------------------------------------------------------------------------
// Warp 0: box c of tile n into its slot once box c of tile n - 1 is released.
template <int G>
__device__ void producer(const CxB<G>& cx, const CUtensorMap* map, PieceCursor cur, int lane) {
  using L = LB<G>;
  const uint64_t pol = policy_evict_first();
  if (lane == 0) prefetch_tensormap(map);
  TileWalker tw;
  tw.init(cur);
  int32_t row0 = 0;
  uint32_t n = 0;  // tiles whose boxes were all issued
  int partial = 0;  // boxes of tile n issued before an abort (in box_at order)
  bool ok = true;
  while (ok && tw.next(row0)) {
    for (int j = 0; j < kBoxes; ++j) {
      const int c = box_at(j);
      if (n >= 1 && !cx.wait(L::kKvEmpty + c, (n - 1) & 1u)) {
        ok = false;
        partial = j;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(cx.bar(L::kKvFull + c), kBoxBytes);
        tma_load_2d(cx.s + L::kOffKv + c * kBoxBytes, map, 128 * c, row0, cx.bar(L::kKvFull + c), pol);
      }
      __syncwarp();
    }
    if (ok) ++n;
  }
  // the last box issued into each slot lands before the CTA exits: tile n for
  // the first `partial` boxes of an aborted tile, tile n - 1 for the others
  for (int j = 0; j < kBoxes; ++j) {
    const int c = box_at(j);
    if (j < partial)
      mbar_wait_drain_tc(cx.bar(L::kKvFull + c), n & 1u);
    else if (n >= 1)
      mbar_wait_drain_tc(cx.bar(L::kKvFull + c), (n - 1) & 1u);
  }
}

// ---------------------------------------------------------------------------
// Warp 1 (one thread): per tile, Q.K^T box by box, then (once P is written)
// P.V block by block.
template <int G>
__device__ void mma_issuer(const CxB<G>& cx, PieceCursor cur) {
  using L = LB<G>;
  constexpr uint32_t kIdQK = umma_idesc(128, L::kN, 1, 1, false, false);  // bf16 x bf16, both K-major
  constexpr uint32_t kIdPV = umma_idesc(128, L::kN, 1, 1, true, true);    // A = V^T MN-major, B = P^T MN-major
  Piece pc;
  uint32_t n = 0, k = 0;
  bool ok = true;
  const uint64_t qb = smem_desc(cx.s + L::kOffQ, 16, 1024, kLayoutSw128);
  const uint64_t ka = smem_desc(cx.s + L::kOffKv, 16, 1024, kLayoutSw128);
  const uint64_t va = smem_desc(cx.s + L::kOffKv, kBoxBytes, 1024, kLayoutSw128);
  while (ok && cur.next(pc)) {
    if (!cx.wait(L::kQFull, k & 1u)) break;
    for (int r0 = 0; r0 < pc.nrows && ok; r0 += kTileRows) {
      const uint32_t s = n & 1u;
      const bool first = r0 == 0, last = r0 + kTileRows >= pc.nrows;
      if (n >= 2 && !cx.wait(L::kSEmpty + s, ((n >> 1) - 1) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t d = cx.tmem + L::kTmS + L::kN * s;
      for (int j = 0; j < kBoxes; ++j) {  // Q.K^T: four k-steps of 16 dims per box
        const int c = box_at(j);
        if (!cx.wait(L::kKvFull + c, n & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(d, desc_add(ka, c * kBoxBytes + ks * 32), desc_add(qb, c * L::kQBoxBytes + ks * 32), kIdQK,
                   (j > 0 || ks > 0) ? 1u : 0u);
        if (c == kRopeBox) umma_commit(cx.bar(L::kKvEmpty + kRopeBox));
      }
      if (!ok) break;
      umma_commit(cx.bar(L::kSFull + s));
      if (last) umma_commit(cx.bar(L::kQEmpty));
      // P.V of this tile, once its P is written (and, for a piece's first
      // tile, O buffer k % 2 has been read by the epilogue of piece k - 2)
      if (!cx.wait(L::kPFull + s, (n >> 1) & 1u) ||
          (first && k >= 2 && !cx.wait(L::kOEmpty + (k & 1u), ((k >> 1) - 1) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T: core matrices of 8 rows x 8 heads, 128 B apart along N, 8-row
      // groups 256 G B apart along K
      const uint64_t pb = smem_desc(cx.s + L::kOffP + s * L::kPBytes, 256 * G, 128, kLayoutNone);
      const uint32_t ob = cx.tmem + L::kTmO + (k & 1u) * 4 * L::kN;
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {  // dims 128 mb .. : boxes 2 mb, 2 mb + 1
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // rows 16 ks ..: two 8-row atoms of 1024 B
          umma_f16(ob + L::kN * mb, desc_add(va, 2 * mb * kBoxBytes + ks * 2048), desc_add(pb, ks * 512 * G), kIdPV,
                   (ks > 0 || !first) ? 1u : 0u);
        umma_commit(cx.bar(L::kKvEmpty + 2 * mb));
        umma_commit(cx.bar(L::kKvEmpty + 2 * mb + 1));
      }
      umma_commit(cx.bar(L::kPvDone + s));
      if (last) umma_commit(cx.bar(L::kOFull + (k & 1u)));
      ++n;
    }
    ++k;
  }
  // every issued tcgen05 operation completes before tensor memory is freed
  umma_commit(cx.bar(L::kDrain));
  mbar_wait_drain_tc(cx.bar(L::kDrain), 0);
}

// ---------------------------------------------------------------------------
// Warps 2-5.

// q of the group's tokens into the B operand (bf16, K-major, 128B swizzle: box
// c holds dims 64 c .. 64 c + 63 of the kN rows; row 16 t + h = head h of
// token t). A group with fewer than G tokens repeats its last token. Thread t
// (0..127) copies head t / 8, dims 72 (t % 8) .. + 71 (nine 16-byte units) of
// each token. Returns the score scale (exp2 domain) or a negative value on
// abort. Piece kk >= 1 waits until the previous piece's last Q.K^T is done.
template <int G, int QF>
__device__ float setup_q_bf(const Stage1Params& p, const CxB<G>& cx, SoftmaxCtx& sx, const Piece& pc, uint32_t kk) {
  using L = LB<G>;
  if (kk >= 1 && !cx.wait(L::kQEmpty, (kk - 1) & 1u)) return -1.f;
  const int t = 32 * sx.wi + sx.lane;
  const int h = t >> 3, d0 = 72 * (t & 7);
  uint8_t* qb = cx.g + L::kOffQ;
  float c = p.sm_scale * kLog2e;
  if (QF != kQBf16) c *= __ldg(p.q_scale);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int64_t token = pc.token + min(g, pc.ntok - 1);
    const int r = 16 * g + h;  // row of the B operand
    uint4 v[9];
    if (QF == kQBf16) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + (token * kHeads + h) * kDqk + d0);
#pragma unroll
      for (int i = 0; i < 9; ++i) v[i] = __ldg(src + i);
    } else {  // e4m3 codes: exact in bf16; the per-tensor scale is in the score scale
      const uint2* src = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.q) + (token * kHeads + h) * kDqk + d0);
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const uint2 w = __ldg(src + i);
        const float2 a = e4m3x2_to_f32x2(w.x & 0xFFFFu), b = e4m3x2_to_f32x2(w.x >> 16);
        const float2 e = e4m3x2_to_f32x2(w.y & 0xFFFFu), f = e4m3x2_to_f32x2(w.y >> 16);
        v[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(b.x, b.y), pack_bf16x2(e.x, e.y), pack_bf16x2(f.x, f.y));
      }
    }
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int d = d0 + 8 * i, box = d >> 6, u = (d & 63) >> 3;
      *reinterpret_cast<uint4*>(qb + box * L::kQBoxBytes + (r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4)) =
          v[i];
    }
  }
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kQFull));
  return c;
}

// One row of softmax weights of token g (16 heads) as bf16 into the P
// operand: row r, token g, heads 8 hh .. 8 hh + 7 at
// (r / 8) 256 G + (2 g + hh) 128 + (r % 8) 16.
template <int G>
__device__ __forceinline__ void put_p_row_bf(uint8_t* pbuf, int row, int g, const float (&pv)[16]) {
  uint8_t* pb = pbuf + (row >> 3) * 256 * G + 2 * g * 128 + (row & 7) * 16;
  *reinterpret_cast<uint4*>(pb) = make_uint4(pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]),
                                             pack_bf16x2(pv[4], pv[5]), pack_bf16x2(pv[6], pv[7]));
  *reinterpret_cast<uint4*>(pb + 128) = make_uint4(pack_bf16x2(pv[8], pv[9]), pack_bf16x2(pv[10], pv[11]),
                                                   pack_bf16x2(pv[12], pv[13]), pack_bf16x2(pv[14], pv[15]));
}

// Multiplies token g's 4 x 16 O columns of this thread's lane by alpha[head].
template <int G>
__device__ __forceinline__ void rescale_o_bf(uint32_t ob, int g, const float (&alpha)[16]) {
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[16];
    tmem_ld16(ob + 16 * G * mb + 16 * g, o);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
    tmem_st16(ob + 16 * G * mb + 16 * g, o);
  }
  tmem_wait_st();
}

// Epilogue of token g of a piece: O times f[head] to the bf16 output (a
// whole-run piece) or the token's fp32 partial slot.
template <int G>
__device__ __forceinline__ void store_o_bf(const Stage1Params& p, const Piece& pc, int g, uint32_t ob, int row,
                                           const float (&f)[16]) {
  const int64_t token = pc.token + g;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[16];
    tmem_ld16(ob + 16 * G * mb + 16 * g, o);
    tmem_wait_ld();
    const int dim = 128 * mb + row;
    if (pc.direct) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + token * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h) dst[h * kDv] = __float2bfloat16_rn(__uint_as_float(o[h]) * f[h]);
    } else {
      float* dst = p.part_o + (pc.slot + g) * kHeads * kDv + dim;
#pragma unroll
      for (int h = 0; h < 16; ++h) dst[h * kDv] = __uint_as_float(o[h]) * f[h];
    }
  }
}

template <int G, int QF>
__device__ void softmax_role(const Stage1Params& p, const CxB<G>& cx, PieceCursor cur, int warp, int lane) {
  using L = LB<G>;
  SoftmaxCtx sx;
  sx.lane = lane;
  sx.wi = warp - 2;
  sx.row = 32 * (warp & 3) + lane;
  sx.lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  sx.gcount = 0;
  float* red_max = reinterpret_cast<float*>(cx.g + L::kOffRedMax);
  float* red_l = reinterpret_cast<float*>(cx.g + L::kOffRedL);
  PieceCursor ahead = cur;
  Piece pc, nxt;
  bool have = ahead.next(pc);
  if (!have) return;
  float c = setup_q_bf<G, QF>(p, cx, sx, pc, 0);
  if (c < 0.f) return;
  uint32_t i = 0, k = 0;
  while (have) {
    const bool have_next = ahead.next(nxt);
    float m[G][16], l[G][16];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m[g][h] = -INFINITY;
        l[g][h] = 0.f;
      }
    const uint32_t ob = cx.tmem + sx.lane_base + L::kTmO + (k & 1u) * 4 * L::kN;
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const int nr = min(kTileRows, pc.nrows - r0);
      const uint32_t b = i & 1u;
      const bool valid = sx.row < nr;
      if (!cx.wait(L::kSFull + b, (i >> 1) & 1u)) return;
      tc_fence_after();
      float x[G][16];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint32_t sr[16];
        tmem_ld16(cx.tmem + sx.lane_base + L::kTmS + L::kN * b + 16 * g, sr);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) x[g][h] = valid ? __uint_as_float(sr[h]) * c : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kSEmpty + b));
      float* rm = red_max + b * 64 * G;  // [token][warp][head]
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float wm[16];
        warp_max16(x[g], wm);
        store16(rm + 64 * g + sx.wi * 16, wm, lane);
      }
      if (!group_sync(cx, sx)) return;
      // P buffer b is free once the P.V of tile i - 2 is done
      if (i >= 2 && !cx.wait(L::kPvDone + b, ((i - 2) >> 1) & 1u)) return;
      bool grew_any = false;
      float alpha[G][16];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4* rm4 = reinterpret_cast<const float4*>(rm + 64 * g);  // [4 warps][16 heads]
        float pv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 a = rm4[q], b4 = rm4[4 + q], c4 = rm4[8 + q], d = rm4[12 + q];
          const float t4[4] = {fmaxf(fmaxf(a.x, b4.x), fmaxf(c4.x, d.x)), fmaxf(fmaxf(a.y, b4.y), fmaxf(c4.y, d.y)),
                               fmaxf(fmaxf(a.z, b4.z), fmaxf(c4.z, d.z)), fmaxf(fmaxf(a.w, b4.w), fmaxf(c4.w, d.w))};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = 4 * q + e;
            const bool up = t4[e] > m[g][h] + kMaxSlackBf;
            alpha[g][h] = up ? fast_exp2(m[g][h] - t4[e]) : 1.0f;
            grew_any |= up;
            m[g][h] = up ? t4[e] : m[g][h];
          }
        }
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          pv[h] = fast_exp2(x[g][h] - m[g][h]);
          l[g][h] = l[g][h] * alpha[g][h] + pv[h];
        }
        put_p_row_bf<G>(cx.g + L::kOffP + b * L::kPBytes, sx.row, g, pv);
      }
      if (grew_any && r0 > 0) {
        // O holds this piece up to tile i - 1: wait for that P.V, then rescale
        if (!cx.wait(L::kPvDone + (b ^ 1u), ((i - 1) >> 1) & 1u)) return;
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < G; ++g) rescale_o_bf<G>(ob, g, alpha[g]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull + b));
      ++i;
    }
    // the next piece's q goes in while this piece's last P.V runs
    float c_next = c;
    if (have_next) {
      c_next = setup_q_bf<G, QF>(p, cx, sx, nxt, k + 1);
      if (c_next < 0.f) return;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float wl = warp_reduce16<false>(l[g], lane);
      if ((lane & 1) == 0) red_l[64 * g + sx.wi * 16 + (lane >> 1)] = wl;
    }
    if (!group_sync(cx, sx)) return;
    if (!cx.wait(L::kOFull + (k & 1u), (k >> 1) & 1u)) return;
    tc_fence_after();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g < pc.ntok) {
        float f[16];
        const float* rl = red_l + 64 * g;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float Lh = rl[h] + rl[16 + h] + rl[32 + h] + rl[48 + h];
          f[h] = 1.0f / Lh;
          if (!pc.direct && sx.row == 16 * g + h) p.part_lse[(pc.slot + g) * kHeads + h] = m[g][h] + fast_log2(Lh);
        }
        store_o_bf<G>(p, pc, g, ob, sx.row, f);
      }
    }
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

template <int G, int QF>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_bf_kernel(const Stage1Params p, const __grid_constant__ CUtensorMap kvmap) {
  extern __shared__ uint8_t smem_raw[];
  CxB<G> cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, 1, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    producer<G>(cx, &kvmap, cur, lane);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<G>(cx, cur);
    __syncwarp();
  } else {
    softmax_role<G, QF>(p, cx, cur, warp, lane);
  }
  cta_end(p, cx, 1);
}

template <int G, int QF>
static cudaError_t launch_q(const Stage1Params& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(stage1_bf_kernel<G, QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, LB<G>::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap map;  // rows of 1152 bytes (576 bf16), boxes of 128 bytes x 128 rows
  e = make_u8_map(&map, p.kv, 2 * kDqk, p.total_kv, 2 * kDqk, 128, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return launch_dependent(stage1_bf_kernel<G, QF>, p.num_splits, kThreads, LB<G>::kAlloc, stream, p, map);
}

}  // namespace bf
}  // namespace tc

cudaError_t launch_stage1_tc_bf16(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (p.group == 2)
    return q_fmt == kQBf16 ? tc::bf::launch_q<2, kQBf16>(p, stream) : tc::bf::launch_q<2, kQFp8>(p, stream);
  return q_fmt == kQBf16 ? tc::bf::launch_q<1, kQBf16>(p, stream) : tc::bf::launch_q<1, kQFp8>(p, stream);
}

}  // namespace mla
