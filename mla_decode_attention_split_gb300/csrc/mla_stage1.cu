// Stage 1 of split-K MLA decode: for each piece of a token's KV run, the fused
// Q.K^T -> online softmax -> P.V over KV tiles streamed once from HBM, leaving
// a normalised partial output and its LSE (or, when the piece is the token's
// whole run, the final bf16 output).
//
// The method is the split-K flash-decoding stage 1 of kernelbot-amd-mixed-mla
// -753817 (`mla_flash_decode_stage1`: 16 heads packed against the single KV
// head, K = all 576 dims, V = the first 512, online softmax in the exp2 domain
// with the sm_scale*log2(e) factor folded into the scores) and -586148
// (`_flash_splitk`). The GB300 design differs from those MI355X kernels:
//
//  * One CTA per SM, 8 warps with fixed roles: 4 "score" warps (Q.K^T, softmax)
//    and 4 "output" warps (P.V, each owning 128 of the 512 V dims). Output
//    warp 0 also streams 64-row KV tiles into a 5-stage (fp8) shared-memory
//    ring with bulk asynchronous copies (one per row, padded row stride so both
//    operand access patterns are bank-conflict free), issuing tile n + S as
//    soon as tile n's stage is released. Stages, P handoff and piece summaries
//    are mbarrier-synchronised; every wait is bounded.
//  * fp8 KV: both contractions run on the e4m3 tensor-core MMA
//    (m16n8k32) directly on the stored codes -- no dequantisation pass. The
//    bf16 operand (the query, or the softmax weights P) enters as an exact
//    pair of e4m3 values hi + lo (hi = e4m3(x), lo = e4m3(x - hi)), so the
//    products are those of the full-precision operand; the per-tensor kv scale
//    is folded into the score scale and the output scale.
//  * bf16 KV: bf16 MMA (m16n8k16), P in bf16.
//  * The contraction index is permuted (consistently on both operands) so each
//    lane feeds the MMA from 16-byte shared-memory loads; the V operand is
//    transposed in registers with byte/halfword permutes.
#include "mla_device.cuh"
#include "mla_internal.h"
#include "mla_merge.cuh"
#include "mla_partition.cuh"

namespace mla {

constexpr int kThreads1 = 256;
constexpr int kTile = 64;
constexpr float kLog2e = 1.4426950408889634f;

template <int KV>
struct KvTraits;
template <>
struct KvTraits<kKvFp8> {
  static constexpr int kRowBytes = 576;
  static constexpr int kStride = 592;  // 37 x 16 B: rows land on distinct 16-B bank groups
  static constexpr int kStages = 5;
};
template <>
struct KvTraits<kKvBf16> {
  static constexpr int kRowBytes = 1152;
  static constexpr int kStride = 1168;  // 73 x 16 B
  static constexpr int kStages = 2;
};

template <int KV>
struct Smem {
  static constexpr int kStages = KvTraits<KV>::kStages;
  static constexpr int kStageBytes = kTile * KvTraits<KV>::kStride;
  static constexpr int kPBytes = 2048;  // one P slot
  static constexpr int kOffP = kStages * kStageBytes;
  static constexpr int kOffAlpha = kOffP + 2 * kPBytes;      // [2][16] f32
  static constexpr int kOffRedMax = kOffAlpha + 2 * 16 * 4;  // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * 16 * 4;  // [4][16] f32
  static constexpr int kOffSum = kOffRedL + 4 * 16 * 4;      // m[16], l[16]
  static constexpr int kOffScan = kOffSum + 32 * 4;          // 16 x i64
  static constexpr int kOffBars = kOffScan + 16 * 8;
  // full[S], empty[S], pfull[2], pempty[2], sfull, sempty, grp[2]
  static constexpr int kNumBars = 2 * kStages + 8;
  static constexpr int kOffAbort = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffAbort + 16;

  __host__ __device__ static constexpr int full(int s) { return s; }
  __host__ __device__ static constexpr int empty(int s) { return kStages + s; }
  __host__ __device__ static constexpr int pfull(int k) { return 2 * kStages + k; }
  __host__ __device__ static constexpr int pempty(int k) { return 2 * kStages + 2 + k; }
  __host__ __device__ static constexpr int sfull() { return 2 * kStages + 4; }
  __host__ __device__ static constexpr int sempty() { return 2 * kStages + 5; }
  __host__ __device__ static constexpr int grp(int k) { return 2 * kStages + 6 + k; }
};

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  volatile uint32_t* abort_word;
  uint32_t* flags;
  __device__ __forceinline__ uint32_t bar(int off_bars, int i) const { return sbase + off_bars + 8u * i; }
};

// Drain-wait: bounded by time only (used to let in-flight copies land before
// the CTA exits, even after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// ---------------------------------------------------------------------------
// KV tile producer (run by all lanes of output warp 0): walks its own copy of
// the piece cursor and issues tiles strictly in consumption order, one bulk
// copy per KV row into stage (tile % S).
template <int KV>
struct TileProducer {
  using S = Smem<KV>;
  static constexpr int RB = KvTraits<KV>::kRowBytes, ST = KvTraits<KV>::kStride;
  PieceCursor cur;
  Piece pc;
  int r0 = 0;
  bool have = false;
  uint32_t issued = 0;
  uint64_t pol;

  __device__ void init(const PieceCursor& c) {
    cur = c;
    have = cur.next(pc);
    r0 = 0;
    pol = policy_evict_first();
  }
  __device__ bool done() const { return !have; }

  // Issues the next tile into its stage. The caller has made sure the stage is
  // free (its previous tile was released by all eight warps).
  __device__ void issue(const Stage1Params& p, const Ctx& cx, int lane) {
    const int nr = min(kTile, pc.nrows - r0);
    const uint32_t s = issued % S::kStages;
    const uint32_t fb = cx.bar(S::kOffBars, S::full(s));
    if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nr * RB));
    __syncwarp();
    const uint8_t* src = static_cast<const uint8_t*>(p.kv) + static_cast<int64_t>(pc.kv_row + r0) * RB;
    const uint32_t dst = cx.sbase + s * S::kStageBytes;
    for (int r = lane; r < nr; r += 32) bulk_g2s(dst + r * ST, src + static_cast<int64_t>(r) * RB, RB, fb, pol);
    ++issued;
    r0 += kTile;
    if (r0 >= pc.nrows) {
      have = cur.next(pc);
      r0 = 0;
    }
  }

  // Lets every issued copy land (bounded by time), so the CTA never exits with
  // a copy still writing into its shared memory.
  __device__ void drain(const Ctx& cx) const {
    for (uint32_t s = 0; s < S::kStages && s < issued; ++s) {
      const uint32_t last = ((issued - 1 - s) / S::kStages) * S::kStages + s;
      mbar_wait_drain(cx.bar(S::kOffBars, S::full(s)), (last / S::kStages) & 1u);
    }
  }
};

// ---------------------------------------------------------------------------
// Query fragments. fp8 KV: 18 k-steps of 32 dims, hi/lo e4m3 pairs.
// Lane (g, t) holds, for heads g and g+8, the dims d = 128W + 32t + 8k + [0,8)
// of window W < 4 (k-steps 4W + k) and d = 512 + 16t + 8k + [0,8) of the last
// half window (k-steps 16 + k). Bytes [0,4) of such an 8-dim group are MMA
// rows/cols 4t..4t+3 of the k-step, bytes [4,8) are 16+4t..16+4t+3.
struct QFragsFp8 {
  uint32_t hi[18][4];
  uint32_t lo[18][4];
};

__device__ __forceinline__ int fp8_chunk_dim(int ks, int t) {
  return ks < 16 ? 128 * (ks >> 2) + 32 * t + 8 * (ks & 3) : 512 + 16 * t + 8 * (ks - 16);
}

// bf16 query -> exact hi/lo e4m3 pairs after scaling by 2^shift (shift puts the
// token's max |q| in [128, 256)). Returns the factor 2^-shift.
__device__ float load_q_fp8pair(const uint16_t* __restrict__ qtok, int g, int t, QFragsFp8& f) {
  uint4 raw[2][18];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint16_t* qh = qtok + (g + 8 * hh) * kDqk;
#pragma unroll
    for (int ks = 0; ks < 18; ++ks) raw[hh][ks] = __ldg(reinterpret_cast<const uint4*>(qh + fp8_chunk_dim(ks, t)));
  }
  uint32_t mx = 0;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int ks = 0; ks < 18; ++ks) {
      mx = __vmaxu2(mx, raw[hh][ks].x & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, raw[hh][ks].y & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, raw[hh][ks].z & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, raw[hh][ks].w & 0x7FFF7FFFu);
    }
  mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int e = static_cast<int>((mx >> 7) & 0xFF);  // biased exponent of max |q|
  int shift = (mx == 0) ? 0 : 134 - e;
  shift = max(-126, min(126, shift));
  const float up = __uint_as_float(static_cast<uint32_t>(shift + 127) << 23);
  const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int ks = 0; ks < 18; ++ks) {
      const uint32_t w[4] = {raw[hh][ks].x, raw[hh][ks].y, raw[hh][ks].z, raw[hh][ks].w};
      uint32_t hic[2], loc[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float x[4];
        x[0] = bf16_bits_to_f32(w[2 * half] & 0xFFFFu) * up;
        x[1] = bf16_bits_to_f32(w[2 * half] >> 16) * up;
        x[2] = bf16_bits_to_f32(w[2 * half + 1] & 0xFFFFu) * up;
        x[3] = bf16_bits_to_f32(w[2 * half + 1] >> 16) * up;
        const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
        const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
        const uint32_t l01 = f32x2_to_e4m3x2(x[0] - d01.x, x[1] - d01.y);
        const uint32_t l23 = f32x2_to_e4m3x2(x[2] - d23.x, x[3] - d23.y);
        hic[half] = h01 | (h23 << 16);
        loc[half] = l01 | (l23 << 16);
      }
      // hic[0] = dims [0,4) of the group (a0/a1), hic[1] = dims [4,8) (a2/a3)
      f.hi[ks][hh] = hic[0];
      f.hi[ks][2 + hh] = hic[1];
      f.lo[ks][hh] = loc[0];
      f.lo[ks][2 + hh] = loc[1];
    }
  return down;
}

__device__ void load_q_fp8codes(const uint8_t* __restrict__ qtok, int g, int t, QFragsFp8& f) {
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint8_t* qh = qtok + (g + 8 * hh) * kDqk;
#pragma unroll
    for (int ks = 0; ks < 18; ++ks) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(qh + fp8_chunk_dim(ks, t)));
      f.hi[ks][hh] = v.x;
      f.hi[ks][2 + hh] = v.y;
      f.lo[ks][hh] = 0;
      f.lo[ks][2 + hh] = 0;
    }
  }
}

// bf16 KV: 36 k-steps of 16 dims. Lane (g, t) holds, for heads g and g+8, the
// dims d = 64W + 16t + 4s + [0,4) (k-step 4W + s); [0,2) are MMA indices
// 2t, 2t+1 and [2,4) are 8+2t, 9+2t.
struct QFragsBf16 {
  uint32_t a[36][4];
};

template <int QF>
__device__ void load_q_bf16frag(const void* qtok_v, int g, int t, QFragsBf16& f) {
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
    for (int W = 0; W < 9; ++W) {
      uint32_t w[8];
      if (QF == kQBf16) {
        const uint16_t* qh = static_cast<const uint16_t*>(qtok_v) + (g + 8 * hh) * kDqk + 64 * W + 16 * t;
        const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(qh));
        const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(qh + 8));
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
      } else {  // e4m3 codes -> exact bf16
        const uint8_t* qh = static_cast<const uint8_t*>(qtok_v) + (g + 8 * hh) * kDqk + 64 * W + 16 * t;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh));
        const uint32_t c[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 lo = e4m3x2_to_f32x2(c[i] & 0xFFFFu), hi = e4m3x2_to_f32x2(c[i] >> 16);
          w[2 * i] = pack_bf16x2(lo.x, lo.y);
          w[2 * i + 1] = pack_bf16x2(hi.x, hi.y);
        }
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        f.a[4 * W + s][hh] = w[2 * s];
        f.a[4 * W + s][2 + hh] = w[2 * s + 1];
      }
    }
  }
}

__device__ __forceinline__ uint32_t u4w(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------
// Score warps: S = Q.K^T for 16 rows of the tile (warp w: rows 16w..16w+15),
// online softmax across the 4 score warps, P to the output warps.
template <int KV, int QF>
__device__ void score_role(const Stage1Params& p, const Ctx& cx, PieceCursor cur, int w, int lane) {
  using S = Smem<KV>;
  constexpr int ST = KvTraits<KV>::kStride;
  const int g = lane >> 2, t = lane & 3;
  float* red_max = reinterpret_cast<float*>(cx.smem + S::kOffRedMax);
  float* red_l = reinterpret_cast<float*>(cx.smem + S::kOffRedL);
  float* alpha_sm = reinterpret_cast<float*>(cx.smem + S::kOffAlpha);
  float* sum_m = reinterpret_cast<float*>(cx.smem + S::kOffSum);
  float* sum_l = sum_m + 16;
  const float qsc = (QF == kQFp8) ? __ldg(p.q_scale) : 1.0f;
  const float kvsc = (KV == kKvFp8) ? __ldg(static_cast<const float*>(p.kv_scale)) : 1.0f;

  uint32_t n = 0, gcount = 0, pm = 0;
  auto group_sync = [&]() -> bool {
    const uint32_t k = gcount & 1u, par = (gcount >> 1) & 1u;
    ++gcount;
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::grp(k)));
    return mbar_wait(cx.bar(S::kOffBars, S::grp(k)), par, cx.abort_word, cx.flags);
  };

  QFragsFp8 qf8;
  QFragsBf16 qfb;
  Piece pc;
  while (cur.next(pc)) {
    float c;  // score scale (exp2 domain)
    if constexpr (KV == kKvFp8) {
      if constexpr (QF == kQBf16) {
        const float down = load_q_fp8pair(static_cast<const uint16_t*>(p.q) + static_cast<int64_t>(pc.token) * kHeads * kDqk,
                                          g, t, qf8);
        c = p.sm_scale * kLog2e * kvsc * down;
      } else {
        load_q_fp8codes(static_cast<const uint8_t*>(p.q) + static_cast<int64_t>(pc.token) * kHeads * kDqk, g, t, qf8);
        c = p.sm_scale * kLog2e * kvsc * qsc;
      }
    } else {
      const size_t esz = (QF == kQBf16) ? 2 : 1;
      load_q_bf16frag<QF>(static_cast<const uint8_t*>(p.q) + static_cast<int64_t>(pc.token) * kHeads * kDqk * esz, g, t,
                          qfb);
      c = p.sm_scale * kLog2e * qsc;
    }
    float m_g = -INFINITY, m_g8 = -INFINITY, l_g = 0.f, l_g8 = 0.f;

    for (int r0 = 0; r0 < pc.nrows; r0 += kTile) {
      const int nr = min(kTile, pc.nrows - r0);
      const uint32_t s = n % S::kStages, rnd = n / S::kStages;
      if (!mbar_wait(cx.bar(S::kOffBars, S::full(s)), rnd & 1u, cx.abort_word, cx.flags)) return;
      const uint32_t sb = cx.sbase + s * S::kStageBytes;
      float s0[2][4], s1[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s0[j][e] = s1[j][e] = 0.f;

      if constexpr (KV == kKvFp8) {
#pragma unroll
        for (int W = 0; W < 5; ++W) {
          uint4 kb[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t row = 16 * w + 8 * j + g;
            const uint32_t a = sb + row * ST + (W < 4 ? 128 * W + 32 * t : 512 + 16 * t);
            kb[j][0] = lds128(a);
            if (W < 4) kb[j][1] = lds128(a + 16);
          }
#pragma unroll
          for (int k = 0; k < (W < 4 ? 4 : 2); ++k) {
            const int ks = (W < 4) ? 4 * W + k : 16 + k;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t b0 = u4w(kb[j][k >> 1], (2 * k) & 3), b1 = u4w(kb[j][k >> 1], (2 * k + 1) & 3);
              mma_e4m3(s0[j], qf8.hi[ks], b0, b1);
              if (QF == kQBf16) mma_e4m3(s1[j], qf8.lo[ks], b0, b1);
            }
          }
        }
      } else {
#pragma unroll
        for (int W = 0; W < 9; ++W) {
          uint4 kb[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t row = 16 * w + 8 * j + g;
            const uint32_t a = sb + row * ST + 128 * W + 32 * t;
            kb[j][0] = lds128(a);
            kb[j][1] = lds128(a + 16);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t b0 = u4w(kb[j][k >> 1], (2 * k) & 3), b1 = u4w(kb[j][k >> 1], (2 * k + 1) & 3);
              if (k & 1) mma_bf16(s1[j], qfb.a[4 * W + k], b0, b1);
              else mma_bf16(s0[j], qfb.a[4 * W + k], b0, b1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::empty(s)));

      // scale, mask, tile max over the 64 rows (this warp's 16, then across warps)
      float sc[2][4];
      float mx_g = -INFINITY, mx_g8 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = 16 * w + 8 * j + 2 * t + (e & 1);
          const float v = (s0[j][e] + s1[j][e]) * c;
          sc[j][e] = (row < nr) ? v : -INFINITY;
          if (e < 2) mx_g = fmaxf(mx_g, sc[j][e]);
          else mx_g8 = fmaxf(mx_g8, sc[j][e]);
        }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mx_g = fmaxf(mx_g, __shfl_xor_sync(0xffffffffu, mx_g, o));
        mx_g8 = fmaxf(mx_g8, __shfl_xor_sync(0xffffffffu, mx_g8, o));
      }
      float* rm = red_max + (n & 1u) * 64;
      if (t == 0) {
        rm[w * 16 + g] = mx_g;
        rm[w * 16 + g + 8] = mx_g8;
      }
      if (!group_sync()) return;
      float tm_g = rm[g], tm_g8 = rm[g + 8];
#pragma unroll
      for (int ww = 1; ww < 4; ++ww) {
        tm_g = fmaxf(tm_g, rm[ww * 16 + g]);
        tm_g8 = fmaxf(tm_g8, rm[ww * 16 + g + 8]);
      }
      const float mn_g = fmaxf(m_g, tm_g), mn_g8 = fmaxf(m_g8, tm_g8);
      const float al_g = fast_exp2(m_g - mn_g), al_g8 = fast_exp2(m_g8 - mn_g8);
      m_g = mn_g;
      m_g8 = mn_g8;
      float pv[2][4];
      float ps_g = 0.f, ps_g8 = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[j][e] = fast_exp2(sc[j][e] - (e < 2 ? mn_g : mn_g8));
          if (e < 2) ps_g += pv[j][e];
          else ps_g8 += pv[j][e];
        }
      l_g = l_g * al_g + ps_g;
      l_g8 = l_g8 * al_g8 + ps_g8;

      // hand P to the output warps through slot n & 1
      const uint32_t slot = n & 1u;
      if (n >= 2 && !mbar_wait(cx.bar(S::kOffBars, S::pempty(slot)), ((n >> 1) - 1) & 1u, cx.abort_word, cx.flags))
        return;
      uint8_t* pbuf = cx.smem + S::kOffP + slot * S::kPBytes;
      if constexpr (KV == kKvFp8) {
        // P' = 256 P as hi + lo e4m3; byte layout [ks][hl][khalf][head][16]
        const int ks = w >> 1, kin = 4 * t + 2 * (w & 1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float x0 = 256.f * pv[0][2 * hh + e], x1 = 256.f * pv[1][2 * hh + e];
            const uint32_t hic = f32x2_to_e4m3x2(x0, x1);
            const float2 hd = e4m3x2_to_f32x2(hic);
            const uint32_t loc = f32x2_to_e4m3x2(x0 - hd.x, x1 - hd.y);
            const int head = g + 8 * hh;
            uint8_t* b = pbuf + ((ks * 2 + 0) * 2 + e) * 256 + head * 16 + kin;
            *reinterpret_cast<uint16_t*>(b) = static_cast<uint16_t>(hic);
            *reinterpret_cast<uint16_t*>(b + 2 * 256) = static_cast<uint16_t>(loc);
          }
      } else {
        // P in bf16; layout [ks][khalf][head][8]; rows 8j + (2t + e) of k-step w
        // map to MMA index 8j + (bit-swapped 2t + e) (see the output warps).
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int k8 = ((t & 2) << 1) | (e << 1) | (t & 1);
              const int head = g + 8 * hh;
              const __nv_bfloat16 v = __float2bfloat16_rn(pv[j][2 * hh + e]);
              *reinterpret_cast<__nv_bfloat16*>(pbuf + ((w * 2 + j) * 16 + head) * 16 + k8 * 2) = v;
            }
      }
      if (w == 0 && t == 0) {
        alpha_sm[slot * 16 + g] = al_g;
        alpha_sm[slot * 16 + g + 8] = al_g8;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::pfull(slot)));
      ++n;
    }

    // piece summary: l over the 64 rows of every tile (lanes, then warps)
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      l_g += __shfl_xor_sync(0xffffffffu, l_g, o);
      l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, o);
    }
    if (t == 0) {
      red_l[w * 16 + g] = l_g;
      red_l[w * 16 + g + 8] = l_g8;
    }
    if (!group_sync()) return;
    if (w == 0) {
      float L_g = 0.f, L_g8 = 0.f;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        L_g += red_l[ww * 16 + g];
        L_g8 += red_l[ww * 16 + g + 8];
      }
      if (pm >= 1 && !mbar_wait(cx.bar(S::kOffBars, S::sempty()), (pm - 1) & 1u, cx.abort_word, cx.flags)) return;
      if (t == 0) {
        sum_m[g] = m_g;
        sum_m[g + 8] = m_g8;
        sum_l[g] = L_g;
        sum_l[g + 8] = L_g8;
        if (!pc.direct) {
          p.part_lse[pc.slot * kHeads + g] = m_g + fast_log2(L_g);
          p.part_lse[pc.slot * kHeads + g + 8] = m_g8 + fast_log2(L_g8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::sfull()));
    }
    ++pm;
  }
}

// ---------------------------------------------------------------------------
// Output warps: acc[16 heads][128 dims] += P.V for warp v's dims 128v..128v+127.
// V operand: n-tile j, column g <-> dim 128v + 16g + j, so each lane reads 16
// contiguous dims of a row; accumulator lane (g, t) ends with heads g, g+8 x
// dims 128v + 32t + [0, 32).
template <int KV, int QF>
__device__ void output_role(const Stage1Params& p, const Ctx& cx, PieceCursor cur, int v, int lane) {
  using S = Smem<KV>;
  constexpr int ST = KvTraits<KV>::kStride;
  const int g = lane >> 2, t = lane & 3;
  const float* alpha_sm = reinterpret_cast<const float*>(cx.smem + S::kOffAlpha);
  const float* sum_l = reinterpret_cast<const float*>(cx.smem + S::kOffSum) + 16;
  const float kvsc = (KV == kKvFp8) ? __ldg(static_cast<const float*>(p.kv_scale)) : 1.0f;
  const float pscale = (KV == kKvFp8) ? (1.0f / 256.0f) : 1.0f;

  TileProducer<KV> prod;
  if (v == 0) {
    prod.init(cur);
    for (int i = 0; i < S::kStages && !prod.done(); ++i) prod.issue(p, cx, lane);
  }
  uint32_t n = 0, pm = 0;
  Piece pc;
  bool ok = true;
  while (ok && cur.next(pc)) {
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    for (int r0 = 0; r0 < pc.nrows; r0 += kTile) {
      const int nr = min(kTile, pc.nrows - r0);
      const uint32_t slot = n & 1u;
      if (!mbar_wait(cx.bar(S::kOffBars, S::pfull(slot)), (n >> 1) & 1u, cx.abort_word, cx.flags)) {
        ok = false;
        break;
      }
      const float al_g = alpha_sm[slot * 16 + g], al_g8 = alpha_sm[slot * 16 + g + 8];
      const uint32_t pb = cx.sbase + S::kOffP + slot * S::kPBytes;
      uint32_t pa[4][4];  // fp8: [ks*2 + hl]; bf16: [ks]
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t base = pb + i * 512;
        pa[i][0] = lds32(base + g * 16 + 4 * t);
        pa[i][1] = lds32(base + (g + 8) * 16 + 4 * t);
        pa[i][2] = lds32(base + 256 + g * 16 + 4 * t);
        pa[i][3] = lds32(base + 256 + (g + 8) * 16 + 4 * t);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::pempty(slot)));
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        acc[j][0] *= al_g;
        acc[j][1] *= al_g;
        acc[j][2] *= al_g8;
        acc[j][3] *= al_g8;
      }
      const uint32_t s = n % S::kStages, rnd = n / S::kStages;
      if (!mbar_wait(cx.bar(S::kOffBars, S::full(s)), rnd & 1u, cx.abort_word, cx.flags)) {
        ok = false;
        break;
      }
      const uint32_t sb = cx.sbase + s * S::kStageBytes;

      if constexpr (KV == kKvFp8) {
        // k-step ks covers tile rows 32ks..32ks+31; MMA index 4t+i <-> row
        // 2t + 8i, 16+4t+i <-> row 2t + 8i + 1.
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t bw[2][16];  // [e][j]
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint4 r[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int row = 32 * ks + 2 * t + 8 * i + e;
              r[i] = lds128(sb + row * ST + 128 * v + 16 * g);
              if (row >= nr) r[i] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
              transpose4x4_bytes(u4w(r[0], q), u4w(r[1], q), u4w(r[2], q), u4w(r[3], q), bw[e][4 * q + 0],
                                 bw[e][4 * q + 1], bw[e][4 * q + 2], bw[e][4 * q + 3]);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            mma_e4m3(acc[j], pa[ks * 2 + 0], bw[0][j], bw[1][j]);
            mma_e4m3(acc[j], pa[ks * 2 + 1], bw[0][j], bw[1][j]);
          }
        }
      } else {
        // k-step ks covers tile rows 16ks..16ks+15; MMA index 2t+e <-> row
        // tau(t) + 2e, 8+2t+e <-> row 8 + tau(t) + 2e, tau = {0,1,4,5}.
        const int tau = (t & 1) | ((t & 2) << 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint4 r[4][2];
          const int rows[4] = {16 * ks + tau, 16 * ks + tau + 2, 16 * ks + tau + 8, 16 * ks + tau + 10};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t a = sb + rows[i] * ST + 256 * v + 32 * g;
            r[i][0] = lds128(a);
            r[i][1] = lds128(a + 16);
            if (rows[i] >= nr) r[i][0] = r[i][1] = make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t ra = u4w(r[0][k >> 2], k & 3), rb = u4w(r[1][k >> 2], k & 3);
            const uint32_t rc = u4w(r[2][k >> 2], k & 3), rd = u4w(r[3][k >> 2], k & 3);
            mma_bf16(acc[2 * k], pa[ks], prmt(ra, rb, 0x5410), prmt(rc, rd, 0x5410));
            mma_bf16(acc[2 * k + 1], pa[ks], prmt(ra, rb, 0x7632), prmt(rc, rd, 0x7632));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::empty(s)));
      if (v == 0 && !prod.done()) {
        // tile n + S goes into stage s once all eight warps released tile n
        if (!mbar_wait(cx.bar(S::kOffBars, S::empty(s)), rnd & 1u, cx.abort_word, cx.flags)) {
          ok = false;
          break;
        }
        prod.issue(p, cx, lane);
      }
      ++n;
    }
    if (!ok) break;

    if (!mbar_wait(cx.bar(S::kOffBars, S::sfull()), pm & 1u, cx.abort_word, cx.flags)) break;
    const float L_g = sum_l[g], L_g8 = sum_l[g + 8];
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(S::kOffBars, S::sempty()));
    ++pm;
    const float f_g = kvsc * pscale / L_g, f_g8 = kvsc * pscale / L_g8;
    const int d0 = 128 * v + 32 * t;
    if (pc.direct) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(pc.token) * kHeads * kDv;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float f = hh ? f_g8 : f_g;
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w[k] = pack_bf16x2(acc[2 * k][2 * hh] * f, acc[2 * k + 1][2 * hh] * f);          // dims d0 + 0..15
          w[8 + k] = pack_bf16x2(acc[2 * k][2 * hh + 1] * f, acc[2 * k + 1][2 * hh + 1] * f);  // d0 + 16..31
        }
        uint4* dst = reinterpret_cast<uint4*>(o + (g + 8 * hh) * kDv + d0);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      }
    } else {
      float* o = p.part_o + pc.slot * kHeads * kDv;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float f = hh ? f_g8 : f_g;
        float4* dst = reinterpret_cast<float4*>(o + (g + 8 * hh) * kDv + d0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          dst[k] = make_float4(acc[4 * k][2 * hh] * f, acc[4 * k + 1][2 * hh] * f, acc[4 * k + 2][2 * hh] * f,
                               acc[4 * k + 3][2 * hh] * f);
          dst[4 + k] = make_float4(acc[4 * k][2 * hh + 1] * f, acc[4 * k + 1][2 * hh + 1] * f,
                                   acc[4 * k + 2][2 * hh + 1] * f, acc[4 * k + 3][2 * hh + 1] * f);
        }
      }
    }
  }
  if (v == 0) prod.drain(cx);
}

template <int KV, int QF>
__global__ void __launch_bounds__(kThreads1, 1) mla_stage1_kernel(const Stage1Params p) {
  using S = Smem<KV>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.smem = smem;
  cx.sbase = smem_addr(smem);
  cx.abort_word = reinterpret_cast<volatile uint32_t*>(smem + S::kOffAbort);
  cx.flags = p.dev_flags;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(cx.bar(S::kOffBars, S::full(s)), 1);
      mbar_init(cx.bar(S::kOffBars, S::empty(s)), 8);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(cx.bar(S::kOffBars, S::pfull(k)), 4);
      mbar_init(cx.bar(S::kOffBars, S::pempty(k)), 4);
      mbar_init(cx.bar(S::kOffBars, S::grp(k)), 4);
    }
    mbar_init(cx.bar(S::kOffBars, S::sfull()), 1);
    mbar_init(cx.bar(S::kOffBars, S::sempty()), 4);
    *cx.abort_word = 0u;
    fence_mbar_init();
  }
  // launched as a programmatic dependent: wait for the kernel before in the
  // stream before touching global memory
  griddep_launch_dependents();
  griddep_wait();
  const int64_t parts = p.num_splits, c = blockIdx.x;
  int64_t* sh = reinterpret_cast<int64_t*>(smem + S::kOffScan);
  const SegLocate loc = block_locate<kThreads1, 1>(
      p.qo_indptr, p.kv_indptr, p.batch, p.total_q, p.total_kv, p.group,
      [=](int64_t total) { return part_start(c, total, parts); }, 0, sh);
  if (!loc.ok) {
    if (threadIdx.x == 0) atomicOr(p.dev_flags, kFlagBadIndptr);
    return;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) p.dev_flags[1] = static_cast<uint32_t>(p.total_q);  // counters in use
  zero_empty_tokens<kThreads1>(p);
  const int64_t x0 = part_start(c, loc.total, parts), x1 = part_start(c + 1, loc.total, parts);
  if (x0 >= x1 || loc.seg < 0) return;
  PieceCursor cur{p.qo_indptr, p.kv_indptr, p.batch, x0, x1, loc.seg, loc.seg_vs, c};
  cur.group = p.group;
  if (warp < 4)
    score_role<KV, QF>(p, cx, cur, warp, lane);
  else
    output_role<KV, QF>(p, cx, cur, warp - 4, lane);
  // split tokens: the CTA that completes a token's partials merges it
  __syncthreads();
  if (!*cx.abort_word) merge_split_tokens_at_end<kThreads1>(p, cur, loc.total, sh);
}

template <int KV, int QF>
static cudaError_t launch_t(const Stage1Params& p, cudaStream_t stream) {
  constexpr int bytes = Smem<KV>::kBytes;
  static_assert(bytes <= 227 * 1024, "shared memory budget");
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(mla_stage1_kernel<KV, QF>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_dependent(mla_stage1_kernel<KV, QF>, p.num_splits, kThreads1, bytes, stream, p);
}

bool stage1_supported(int kv_fmt, int q_fmt) {
  if (q_fmt == kQBf16Quant) return kv_fmt == kKvFp8;  // the in-call a8w8 mode
  return (kv_fmt == kKvFp8 || kv_fmt == kKvBf16 || kv_fmt == kKvMxfp4) && (q_fmt == kQBf16 || q_fmt == kQFp8);
}

cudaError_t launch_stage1(int kv_fmt, int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (kv_fmt == kKvFp8) return launch_stage1_tc_fp8(q_fmt, p, stream);
  if (kv_fmt == kKvMxfp4) return launch_stage1_tc_mxfp4(q_fmt, p, stream);
  if (kv_fmt == kKvBf16) return launch_stage1_tc_bf16(q_fmt, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mla
