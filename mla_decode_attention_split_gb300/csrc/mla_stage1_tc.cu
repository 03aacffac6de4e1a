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
//    a normal number. The per-tensor kv scale, 2^-shift of q and 1/kPScale of P
//    are applied to the fp32 results.
//  * Shared memory holds three 64 KB stages of the 512 V dims of 128-row tiles
//    (four 128B-swizzled 128x128 TMA boxes each), so two tiles stream in while
//    one is consumed. The 64 rope dims of each row (used by Q.K^T only) are
//    loaded by the softmax threads into registers two tiles ahead and written
//    into a single 8 KB slot as soon as the previous tile's Q.K^T is done.
//  * Warp 0 issues the TMA loads (a paged cache: runs of consecutive pool
//    rows by TMA, other rows by cp.async), warp 1 owns tensor memory and
//    issues QK(n) then PV(n-1) so the tensor core overlaps the softmax of tile
//    n; one commit after PV(n-1) frees its stage and the P buffer. Warps 2-5
//    (one thread per tile row / tensor-memory lane) read S, reduce the per-head
//    max across the 128 rows, write P into shared memory, rescale O in tensor
//    memory only when some head's reference max moved (lazily, see kMaxSlack),
//    and store each token run's output (a contiguous cache: one 128-dim block
//    per tile of the next run). Warps 6-7 prepare the Q operand of later runs.
//  * Every mbarrier wait is bounded; on a timeout the CTA stops issuing work,
//    lets in-flight copies and MMAs finish, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "mla_tc_common.cuh"

namespace mla {
namespace tc {

constexpr int kThreads = 256;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax, 6-7 the Q operand of pieces >= 1
constexpr uint32_t kBarQprep = 2;  // named barrier of the two q-prep warps (0 is __syncthreads)
constexpr int kStages = 3;
constexpr int kStageBytes = kVBytes;  // 64 KB: the 512 V dims of a tile

struct L {
  static constexpr int kThreads = tc::kThreads;
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kStages * kStageBytes;
  static constexpr int kOffRope = kOffQ + kQBytes;
  static constexpr int kOffP = kOffRope + kRopeBytes;
  static constexpr int kOffRedMax = kOffP + kPBytes;              // [2][4][16] f32
  static constexpr int kOffRedL = kOffRedMax + 2 * 4 * 16 * 4;    // [4][16] f32
  static constexpr int kOffFac = kOffRedL + 4 * 16 * 4;           // [piece % 2][16] f32: output factors
  static constexpr int kOffAmax = kOffFac + 2 * 16 * 4;           // [4] u32
  static constexpr int kOffMList = kOffAmax + 16;                 // MergeList (128 B)
  static constexpr int kOffScan = kOffMList + 128;                 // 16 x i64
  static constexpr int kOffCRing = kOffScan + 16 * 8;             // score scale of piece k: f32 [4] + tag u32 [4]
  static constexpr int kOffQpAmax = kOffCRing + 32;               // [2] u32: the q-prep warps' maxima
  static constexpr int kOffBars = kOffQpAmax + 16;
  enum {
    kKvFull = 0, kKvEmpty = 3, kSFull = 6, kSEmpty = 8, kRopeFull = 10, kPFull = 11, /* 12 unused */ kQFull = 13,
    kQEmpty = 14, kOFull = 15, kOEmpty = 17, kGrp = 19, kDrain = 21, kMerge = 22, kQ0 = 23, kNumBars = 24
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
      mbar_init(cx.bar(kOFull + i), 1);
      mbar_init(cx.bar(kOEmpty + i), 4);
      mbar_init(cx.bar(kGrp + i), 4);
    }
    mbar_init(cx.bar(kRopeFull), 4);
    mbar_init(cx.bar(kPFull), 4);
    mbar_init(cx.bar(kQFull), 4);  // piece 0: the 4 softmax warps; later pieces: the 2 q-prep warps, 2 each
    mbar_init(cx.bar(kQEmpty), 1);
    mbar_init(cx.bar(kDrain), 1);
    mbar_init(cx.bar(kQ0), 4);  // the CTA's first Q operand is in (one phase)
    for (int i = 0; i < 4; ++i) reinterpret_cast<volatile uint32_t*>(cx.g + kOffCRing + 16)[i] = 0u;
  }
};
static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
static_assert(L::kOffQ % 1024 == 0 && L::kOffRope % 1024 == 0, "operands need 1024-byte alignment");
static_assert(L::kOffFac % 16 == 0, "factor buffer alignment");
using Cx = Ctx<L>;

// Warp 0: the V dims of each tile, four 128-row x 128-byte boxes, into stage
// (tile % 3) once the tile three back has been released by its P.V. Tiles
// after the first wait until the CTA's first Q operand is in: the q (and rope)
// loads of the call's start then do not queue behind every CTA's full ring.
__device__ void producer(const Cx& cx, const CUtensorMap* map, PieceCursor cur, int lane) {
  const uint64_t pol = policy_evict_first();
  Piece pc;
  uint32_t n = 0;
  bool ok = true;
  while (ok && cur.next(pc)) {
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n % kStages, rnd = n / kStages;
      if ((n == 1 && !cx.wait(L::kQ0, 0)) || (rnd >= 1 && !cx.wait(L::kKvEmpty + s, (rnd - 1) & 1u))) {
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

// Warp 0 with a paged cache. Rows of a tile that are consecutive rows of the
// pool (a run inside one page, or pages laid out in order) come in by TMA:
// each maximal run of whole 8-row groups is one box per 128-byte chunk, 8 to
// 128 rows high (one tensor map per height), landing in the same
// 128B-swizzled layout as the contiguous path's 128-row boxes. The rows of the
// other groups are gathered with 16-byte cp.async copies (lane l copies bytes
// 16l..16l+15 of each row) into that layout; once they have landed every lane
// makes them visible to the tensor core (async proxy) before the warp's
// arrival on kv_full. The page ids of a tile are loaded two tiles ahead and
// its runs are worked out before its stage is free. Rows past the piece, and rows whose page id is
// outside the pool, are not copied.
struct PagedMaps {
  CUtensorMap box[16];  // box[h]: 128 bytes x 8 (h + 1) rows of the pool
};

struct PagedDrain {
  uint32_t issued, tma_hist, n_last;  // tiles issued, which of the last ones used TMA, the last tile
};

__device__ PagedDrain producer_paged(const Stage1Params& p, const Cx& cx, const PagedMaps* maps, PieceCursor cur,
                                     int lane) {
  const uint64_t pol = policy_evict_first();
  const uint8_t* kv = static_cast<const uint8_t*>(p.kv) + lane * 16;
  const uint32_t unit = lane & 7, chunk_off = (lane >> 3) * kChunkBytes;
  if (lane < 16) prefetch_tensormap(&maps->box[lane]);
  TileWalker tw;
  tw.init(cur);
  PagedRow id[4], id_next[4];  // page ids of this tile and the next (loaded two tiles ahead)
  bool have = paged_tile_ids(p, tw, lane, id);
  bool have_next = have && paged_tile_ids(p, tw, lane, id_next);
  PagedDrain d{0u, 0u, 0u};
  for (uint32_t n = 0; have; ++n) {
    const uint32_t s = n % kStages, rnd = n / kStages;
    // the tile's rows and runs are worked out before its stage is free
    int32_t phys[4];  // tile rows lane + 32 j
#pragma unroll
    for (int j = 0; j < 4; ++j) phys[j] = phys_row(p, id[j]);
    uint32_t contig = 0;  // bit g: rows 8g..8g+7 are consecutive rows of the pool
    uint32_t linked = 0;  // bit g: row 8g follows row 8g-1 in the pool
    int32_t run_y = 0, run_len = 0;
    // the whole tile one run of the pool (pages laid out in order, or pages of
    // 128 rows and more): one box per chunk
    const int32_t phys0 = __shfl_sync(0xffffffffu, phys[0], 0);
    const bool whole = __all_sync(0xffffffffu, phys0 >= 0 && phys[0] == phys0 + lane && phys[1] == phys0 + 32 + lane &&
                                                   phys[2] == phys0 + 64 + lane && phys[3] == phys0 + 96 + lane);
    if (whole) {
      contig = 0xFFFFu;
      linked = 0xFFFEu;
      run_y = phys0;
      run_len = lane == 0 ? 16 : 0;
    } else {
      int32_t last_prev = -1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int32_t prev = __shfl_up_sync(0xffffffffu, phys[j], 1);
        if (lane == 0) prev = last_prev;
        last_prev = __shfl_sync(0xffffffffu, phys[j], 31);
        const bool follows = phys[j] >= 0 && prev >= 0 && phys[j] == prev + 1;
        const uint32_t b = __ballot_sync(0xffffffffu, phys[j] >= 0 && ((lane & 7) == 0 || follows));
        const uint32_t l = __ballot_sync(0xffffffffu, follows);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (((b >> (8 * q)) & 0xFFu) == 0xFFu) contig |= 1u << (4 * j + q);
          if ((l >> (8 * q)) & 1u) linked |= 1u << (4 * j + q);
        }
      }
      // runs: a contiguous group starts one unless it continues the previous
      // contiguous group; lane g < 16 holds the first pool row and the length
      // (in groups) of the run that starts at group g
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int32_t v = __shfl_sync(0xffffffffu, phys[j], (lane & 3) * 8);
        if ((lane >> 2) == j) run_y = v;
      }
      const uint32_t starts0 = contig & ~((contig << 1) & linked);
      if (lane < 16 && ((starts0 >> lane) & 1u)) {
        // groups lane + 1.. that continue the run: the trailing ones of (contig & linked) >> (lane + 1)
        const uint32_t cont = (contig & linked) >> (lane + 1);
        run_len = min(__ffs(~cont), 16 - lane);
      }
    }
    const uint32_t starts = contig & ~((contig << 1) & linked);
    if (rnd >= 1 && !cx.wait(L::kKvEmpty + s, (rnd - 1) & 1u)) break;
    const uint32_t bar = cx.bar(L::kKvFull + s);
    const uint32_t stage = cx.s + L::kOffKv + s * kStageBytes;
    if (contig) {
      if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(__popc(contig)) * kVChunks * 1024u);
      __syncwarp();
      uint32_t left = starts;
      while (left) {
        const int g0 = __ffs(left) - 1;
        left &= left - 1;
        const int32_t y = __shfl_sync(0xffffffffu, run_y, g0);
        const int32_t len = __shfl_sync(0xffffffffu, run_len, g0);
        if (lane < kVChunks)
          tma_load_2d(stage + lane * kChunkBytes + g0 * 1024, &maps->box[len - 1], lane * 128, y, bar, pol);
      }
    }
    if (contig != 0xFFFFu) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll 8
        for (int rr = 0; rr < 32; ++rr) {
          const int32_t g = __shfl_sync(0xffffffffu, phys[j], rr);
          const uint32_t r = 32 * j + rr;
          if (g >= 0 && !((contig >> (r >> 3)) & 1u))
            cp_async16(stage + chunk_off + r * 128 + ((unit ^ (r & 7u)) << 4), kv + static_cast<int64_t>(g) * kDqk,
                       pol);
        }
      }
      // each lane's copies complete its own (pending-count neutral) arrival
      // on the barrier; the producer does not wait for them
      cp_async_mbar_arrive(bar);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
#pragma unroll
    for (int j = 0; j < 4; ++j) id[j] = id_next[j];
    have = have_next;
    have_next = have && paged_tile_ids(p, tw, lane, id_next);  // two tiles ahead
    d.tma_hist = (d.tma_hist << 1) | (contig ? 1u : 0u);
    ++d.issued;
    d.n_last = n;
  }
  cp_async_wait_all();  // none of this warp's copies may land after the CTA exits
  return d;
}

// Warp 6 with a paged cache: at the CTA's start, pulls the page-table entries of
// all its pieces into L2 (one prefetch per 128-byte line, addresses inside each
// piece's range of the table), so that the producer's and the softmax warps'
// page-id loads, issued a tile or two ahead, do not wait on DRAM.
__device__ void prefetch_page_ids(const Stage1Params& p, PieceCursor cur, int lane) {
  Piece pc;
  while (cur.next(pc)) {
    const int32_t i0 = pc.kv_row - pc.k0, i1 = i0 + pc.nrows - 1;
    const int32_t e0 = pc.pbase + (p.page_shift >= 0 ? i0 >> p.page_shift : i0 / p.page_size);
    const int32_t e1 = pc.pbase + (p.page_shift >= 0 ? i1 >> p.page_shift : i1 / p.page_size);
    for (int32_t e = (e0 & ~31) + 32 * lane; e <= e1; e += 32 * 32) prefetch_l2(p.page_indices + (e < e0 ? e0 : e));
  }
}

// When the CTA stopped early (a bounded wait ran out) the consumer may not
// have waited for every tile: the producer's last TMA tiles (one per stage,
// the older ones were released through kv_empty) land before the CTA exits.
// Called after all roles have returned.
__device__ void drain_paged(const Cx& cx, const PagedDrain& d) {
  for (uint32_t k = 0; k < 3 && k < d.issued; ++k) {
    if ((d.tma_hist >> k) & 1u) {
      const uint32_t nn = d.n_last - k;
      mbar_wait_drain_tc(cx.bar(L::kKvFull + nn % kStages), (nn / kStages) & 1u);
    }
  }
}

// ---------------------------------------------------------------------------
// Warp 1 (one thread): QK(n) into S[n % 2], then PV(n-1) into O[piece % 2].
struct PendingPV {
  uint32_t n, k;
  bool first, last, valid;
};

__device__ bool issue_pv(const Cx& cx, const PendingPV& t) {
  constexpr uint32_t id_pv = umma_idesc(128, 32, 0, 0, true, true);
  if (!cx.wait(L::kPFull, t.n & 1u)) return false;
  if (t.first && t.k >= 2 && !cx.wait(L::kOEmpty + (t.k & 1u), ((t.k >> 1) - 1) & 1u)) return false;
  tc_fence_after();
  const uint32_t stage = cx.s + L::kOffKv + (t.n % kStages) * kStageBytes;
  const uint32_t pbuf = cx.s + L::kOffP;
  const uint32_t obuf = cx.tmem + kTmemO + (t.k & 1u) * 128;
#pragma unroll
  for (int mb = 0; mb < 4; ++mb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      umma_e4m3(obuf + 32 * mb, pv_desc_a(stage, mb, ks), pv_desc_b(pbuf, ks), id_pv, (ks > 0 || !t.first) ? 1u : 0u);
    }
  // one commit frees the stage and, for the softmax warps, the P buffer
  umma_commit(cx.bar(L::kKvEmpty + (t.n % kStages)));
  if (t.last) umma_commit(cx.bar(L::kOFull + (t.k & 1u)));
  return true;
}

template <bool kPaged>
__device__ void mma_issuer(const Cx& cx, PieceCursor cur) {
  constexpr uint32_t id_qk = umma_idesc(128, 32, 0, 0, false, false);
  Piece pc;
  uint32_t n = 0, k = 0;
  PendingPV pend{0, 0, false, false, false};
  bool ok = true;
  while (ok && cur.next(pc)) {
    if (!cx.wait(L::kQFull, k & 1u)) break;
    const uint32_t qbuf = cx.s + L::kOffQ;
    for (int r0 = 0; r0 < pc.nrows; r0 += kTileRows) {
      const uint32_t s = n & 1u, st = n % kStages;
      if (!cx.wait(L::kKvFull + st, (n / kStages) & 1u) || !cx.wait(L::kRopeFull, n & 1u)) {
        ok = false;
        break;
      }
      // paged: rows gathered by cp.async were written through the generic proxy
      if constexpr (kPaged) fence_async_smem();
      if (n >= 2 && !cx.wait(L::kSEmpty + s, ((n >> 1) - 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t stage = cx.s + L::kOffKv + st * kStageBytes;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {  // the 512 V dims, from the stage
        umma_e4m3(cx.tmem + kTmemS + 32 * s, qk_desc_a(stage, ks), qk_desc_b(qbuf, ks), id_qk, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {  // the 64 rope dims, from the rope slot (no swizzle)
        umma_e4m3(cx.tmem + kTmemS + 32 * s, rope_desc_a(cx.s + L::kOffRope, ks), qk_desc_b(qbuf, 16 + ks), id_qk, 1u);
      }
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

// Paged cache: the page id of this thread's row of the next tile (its load is
// consumed one tile later), and the rope bytes of a row from its page id.
__device__ __forceinline__ PagedRow next_rope_id(const Stage1Params& p, TileWalker& rw, int row) {
  TileRef t;
  return (rw.next(t) && row < t.nvalid) ? page_of(p, t.pbase, t.row - t.k0 + row) : page_of_none();
}

__device__ __forceinline__ void load_rope_paged(const Stage1Params& p, PagedRow id, uint4 (&r)[4]) {
  const int32_t g = phys_row(p, id);
  if (g >= 0) {
    const uint4* src =
        reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.kv) + static_cast<int64_t>(g) * kDqk + 512);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __ldg(src + i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Writes one row's rope bytes into the slot and hands the slot to the MMA warp.
__device__ __forceinline__ void store_rope(const Cx& cx, const SoftmaxCtx& sx, const uint4 (&r)[4]) {
  put_rope_row(cx.g + L::kOffRope, sx.row, r);
  fence_async_smem();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kRopeFull));
}

// Warps 6-7: the Q operand (B of Q.K^T, the layout fill_q writes) of every
// piece after the first, prepared while the piece before it streams, so that
// at a piece boundary the tensor pipe waits only for the copy into the Q
// buffer. Thread t (0..63) takes head t / 4, dims 144 (t % 4) .. +143; the
// codes and the score scale are those fill_q computes (the same per-token
// amax, here over two warps). The scale of piece k goes to ring slot k % 4,
// tagged k + 1, for the softmax warps. The ring cannot be overwritten early:
// piece k + 4's operand waits for the last Q.K^T of piece k + 3, which needs
// a score buffer that the softmax warps freed after they started piece k.
__device__ __forceinline__ bool qprep_all(bool v) {  // both q-prep warps agree
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 64, p;\n selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(v)), "r"(kBarQprep)
               : "memory");
  return r != 0u;
}

template <int QF>
__device__ void qprep_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
  Piece pc;
  if (!cur.next(pc)) return;  // piece 0 is set up by the softmax warps
  const int t = 32 * (warp - 6) + lane;  // 0..63
  const int h = t >> 2, d0 = 144 * (t & 3);
  const float kvsc = __ldg(static_cast<const float*>(p.kv_scale));
  uint8_t* qb = cx.g + L::kOffQ;
  auto qaddr = [&](int row, int d) -> uint32_t* {
    const int unit = (d & 127) >> 4;
    return reinterpret_cast<uint32_t*>(qb + (d >> 7) * kQChunkBytes + (row >> 3) * 1024 + (row & 7) * 128 +
                                       ((unit ^ (row & 7)) << 4) + (d & 15));
  };
  volatile float* ring_c = reinterpret_cast<volatile float*>(cx.g + L::kOffCRing);
  volatile uint32_t* ring_tag = reinterpret_cast<volatile uint32_t*>(cx.g + L::kOffCRing + 16);
  uint32_t* am = reinterpret_cast<uint32_t*>(cx.g + L::kOffQpAmax);
  if (QF == kQBf16Quant && p.wait_late) griddep_wait();  // the scale comes from this call's amax kernel
  for (uint32_t k = 1; cur.next(pc); ++k) {
    uint32_t hi[36], lo[36];
    float c;
    if (QF == kQFp8) {
      const uint8_t* src = static_cast<const uint8_t*>(p.q) + (static_cast<int64_t>(pc.token) * kHeads + h) * kDqk + d0;
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
        hi[4 * i] = v.x; hi[4 * i + 1] = v.y; hi[4 * i + 2] = v.z; hi[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 36; ++i) lo[i] = 0u;
      c = p.sm_scale * kLog2e * kvsc * __ldg(p.q_scale);
    } else {
      const uint16_t* src =
          static_cast<const uint16_t*>(p.q) + (static_cast<int64_t>(pc.token) * kHeads + h) * kDqk + d0;
      uint32_t w[72];
#pragma unroll
      for (int i = 0; i < 18; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
      if (QF == kQBf16Quant) {
        const float qs = *static_cast<const volatile float*>(p.q_scale);
        const float inv = 1.0f / qs;  // correctly rounded, once
#pragma unroll
        for (int i = 0; i < 36; ++i) {  // dims d0 + 4i .. +3
          const float a = quotient_rn(bf16_bits_to_f32(w[2 * i] & 0xFFFFu), qs, inv);
          const float b = quotient_rn(bf16_bits_to_f32(w[2 * i] >> 16), qs, inv);
          const float e = quotient_rn(bf16_bits_to_f32(w[2 * i + 1] & 0xFFFFu), qs, inv);
          const float f = quotient_rn(bf16_bits_to_f32(w[2 * i + 1] >> 16), qs, inv);
          hi[i] = f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(e, f) << 16);
          lo[i] = 0u;
        }
        c = p.sm_scale * kLog2e * kvsc * qs;
      } else {
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 72; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
        mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) am[warp - 6] = mx;
        named_bar_sync(kBarQprep, 64);
        mx = max(am[0], am[1]);
        named_bar_sync(kBarQprep, 64);  // both have read am before the next piece writes it
        const int e = static_cast<int>((mx >> 7) & 0xFF);  // biased exponent of max |q|
        int shift = (mx == 0) ? 0 : 134 - e;               // max |q| 2^shift in [128, 256)
        shift = max(-126, min(126, shift));
        const float up = __uint_as_float(static_cast<uint32_t>(shift + 127) << 23);
        const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
#pragma unroll
        for (int g = 0; g < 36; ++g) {  // dims d0 + 4g .. +3
          const float x0 = bf16_bits_to_f32(w[2 * g] & 0xFFFFu) * up, x1 = bf16_bits_to_f32(w[2 * g] >> 16) * up;
          const float x2 = bf16_bits_to_f32(w[2 * g + 1] & 0xFFFFu) * up,
                      x3 = bf16_bits_to_f32(w[2 * g + 1] >> 16) * up;
          const uint32_t h01 = f32x2_to_e4m3x2(x0, x1), h23 = f32x2_to_e4m3x2(x2, x3);
          const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
          const uint32_t l01 = f32x2_to_e4m3x2(kLoScale * (x0 - d01.x), kLoScale * (x1 - d01.y));
          const uint32_t l23 = f32x2_to_e4m3x2(kLoScale * (x2 - d23.x), kLoScale * (x3 - d23.y));
          hi[g] = h01 | (h23 << 16);
          lo[g] = l01 | (l23 << 16);
        }
        c = p.sm_scale * kLog2e * kvsc * down;
      }
    }
    // the previous piece's last Q.K^T has read the Q buffer
    if (!qprep_all(cx.wait(L::kQEmpty, (k - 1) & 1u))) return;
#pragma unroll
    for (int g = 0; g < 36; ++g) {
      *qaddr(h, d0 + 4 * g) = hi[g];
      *qaddr(16 + h, d0 + 4 * g) = lo[g];
    }
    if (t == 0) {
      ring_c[k & 3u] = c;
      __threadfence_block();
      ring_tag[k & 3u] = k + 1u;
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(cx.bar(L::kQFull), 2);
  }
}

// The score scale of piece k >= 1 from the q-prep ring (bounded wait); a
// negative value on abort.
__device__ __forceinline__ float ring_scale(const Cx& cx, uint32_t k) {
  const volatile float* ring_c = reinterpret_cast<const volatile float*>(cx.g + L::kOffCRing);
  const volatile uint32_t* ring_tag = reinterpret_cast<const volatile uint32_t*>(cx.g + L::kOffCRing + 16);
  if (ring_tag[k & 3u] != k + 1u) {
    const long long t0 = clock64();
    while (ring_tag[k & 3u] != k + 1u) {
      if (*cx.abort_word) return -1.f;
      if (clock64() - t0 > kWaitLimitCycles) {
        *cx.abort_word = 1u;
        atomicOr(cx.flags, kFlagTimeout);
        return -1.f;
      }
    }
  }
  __threadfence_block();
  return ring_c[k & 3u];
}

// The epilogue of a piece, deferred (contiguous cache): its O buffer is
// written out one 128-dim block at a time in the idle time of the next
// piece's tiles (each softmax pass ends waiting for the next scores), so the
// tensor core does not stop at piece boundaries while the softmax warps store
// a whole partial. The paged kernel stores a piece's output at its end (its
// loop has no registers to spare, and the larger code slowed it down).
struct PendingOut {
  Piece pc;
  uint32_t k;      // the piece's index (its O buffer k % 2, factors k % 2)
  int blocks;      // 128-dim blocks still to store (0: none pending)
};

// Stores one block of the pending piece; after the last one, frees its O
// buffer and publishes and counts a split partial. Returns false on abort.
__device__ __forceinline__ bool pending_block(const Stage1Params& p, const Cx& cx, SoftmaxCtx& sx, PendingOut& po) {
  const int mb = 4 - po.blocks;
  if (mb == 0) {
    if (!cx.wait(L::kOFull + (po.k & 1u), (po.k >> 1) & 1u)) return false;
    tc_fence_after();
  }
  const float4* fb = reinterpret_cast<const float4*>(cx.g + L::kOffFac + (po.k & 1u) * 64);
  float f[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = fb[q];
    f[4 * q] = v.x; f[4 * q + 1] = v.y; f[4 * q + 2] = v.z; f[4 * q + 3] = v.w;
  }
  store_o_block(p, po.pc, cx.tmem + sx.lane_base + kTmemO + (po.k & 1u) * 128, sx.row, f, mb);
  if (--po.blocks > 0) return true;
  tc_fence_before();
  __syncwarp();
  if (sx.lane == 0) mbar_arrive(cx.bar(L::kOEmpty + (po.k & 1u)));
  return po.pc.direct || finish_partial(p, cx, sx, po.pc);
}

template <int QF, bool kPaged>
__device__ void softmax_role(const Stage1Params& p, const Cx& cx, PieceCursor cur, int warp, int lane) {
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
  // rope of tiles 0 and 1 into registers, the first Q operand, tile 0 into the
  // slot, tile 2 loads (a paged cache: through the rows' page ids)
  TileWalker rw;
  uint4 rb0[4], rb1[4];  // rope of the even / odd tile in flight
  PagedRow rid = page_of_none();  // paged: the page id of this row of the tile after the next rope load
  rw.init(cur);
  if constexpr (!kPaged) {
    load_rope(p, rw, sx.row, rb0);
    load_rope(p, rw, sx.row, rb1);
  } else {
    rid = next_rope_id(p, rw, sx.row);
    load_rope_paged(p, rid, rb0);
    rid = next_rope_id(p, rw, sx.row);
    load_rope_paged(p, rid, rb1);
  }
  // the first Q operand while those rope rows are in flight
  float c = setup_q<L, QF>(p, cx, sx, pc.token, 0, kvsc);
  if (c < 0.f) return;
  if (lane == 0) mbar_arrive(cx.bar(L::kQ0));
  store_rope(cx, sx, rb0);
  if constexpr (!kPaged) {
    load_rope(p, rw, sx.row, rb0);
  } else {
    rid = next_rope_id(p, rw, sx.row);
    load_rope_paged(p, rid, rb0);
    rid = next_rope_id(p, rw, sx.row);
  }
  uint32_t n = 0, k = 0;
  PendingOut po;
  po.blocks = 0;
  int tiles_left = 0;  // tiles of the CTA after the current one (for the rope slot)
  {
    PieceCursor cnt = cur;
    Piece t;
    while (cnt.next(t)) tiles_left += (t.nrows + kTileRows - 1) / kTileRows;
    tiles_left -= 1;
  }
  while (have) {
    const bool have_next = ahead.next(nxt);
    if (k > 0) {
      c = ring_scale(cx, k);
      if (c < 0.f) return;
    }
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
      // Q.K^T(n) is done: the rope slot takes tile n+1, its registers tile n+3
      if (tiles_left > 0) {
        if constexpr (kPaged) {  // the page id was loaded one tile earlier
          if (n & 1u) {
            store_rope(cx, sx, rb0);
            load_rope_paged(p, rid, rb0);
          } else {
            store_rope(cx, sx, rb1);
            load_rope_paged(p, rid, rb1);
          }
          rid = next_rope_id(p, rw, sx.row);
        } else {
          if (n & 1u) {
            store_rope(cx, sx, rb0);
            load_rope(p, rw, sx.row, rb0);
          } else {
            store_rope(cx, sx, rb1);
            load_rope(p, rw, sx.row, rb1);
          }
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
      const bool valid = sx.row < nr && (r0 > 0 || sx.row >= pc.lead);
      float x[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float v = (__uint_as_float(sr[h]) + __uint_as_float(sr[16 + h]) * (1.0f / kLoScale)) * c;
        x[h] = valid ? v : -INFINITY;
      }
      float* rm = red_max + (n & 1u) * 64;
      {
        float wm[16];
        warp_max16(x, wm);
        store16(rm + sx.wi * 16, wm, lane);
      }
      if (!group_sync(cx, sx)) return;
      bool grew = false;
      float alpha[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float tm = fmaxf(fmaxf(rm[h], rm[16 + h]), fmaxf(rm[32 + h], rm[48 + h]));
        const bool up = tm > m[h] + kMaxSlack;
        alpha[h] = up ? fast_exp2(m[h] - tm) : 1.0f;
        grew |= up;
        m[h] = up ? tm : m[h];
      }
      const bool rescale = grew && r0 > 0;
      float pv[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        pv[h] = fast_exp2(x[h] - m[h]);
        l[h] = l[h] * alpha[h] + pv[h];
        pv[h] *= kPScale;
      }
      // single P buffer: P.V(n-1) must be done (the commit that releases its stage)
      if (n >= 1 && !cx.wait(L::kKvEmpty + (n - 1) % kStages, ((n - 1) / kStages) & 1u)) return;
      put_p_row(cx.g + L::kOffP, sx.row, pv);
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
        rescale_o(cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128, alpha);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kPFull));
      ++n;
      // a block of the previous piece's output while the next scores are computed
      // (contiguous cache; the paged loop has no registers to spare for it)
      if constexpr (!kPaged) {
        if (po.blocks > 0 && !pending_block(p, cx, sx, po)) return;
      }
    }

    // (the next piece's Q operand comes from warps 6-7, qprep_role)
    if constexpr (kPaged) {
      // l over the 128 rows, per head; the output at once
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
      store_o(p, pc, cx.tmem + sx.lane_base + kTmemO + (k & 1u) * 128, sx.row, f);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(L::kOEmpty + (k & 1u)));
      if (!pc.direct && !finish_partial(p, cx, sx, pc)) return;
    } else {
      while (po.blocks > 0)  // the previous piece's output, if this piece was too short to take it all
        if (!pending_block(p, cx, sx, po)) return;
      // l over the 128 rows, per head; the output factors go to the factor
      // buffer of this piece (the last reader of that buffer, two pieces back,
      // is done: its blocks were stored above)
      const float wl = warp_reduce16<false>(l, lane);
      if ((lane & 1) == 0) red_l[sx.wi * 16 + (lane >> 1)] = wl;
      if (!group_sync(cx, sx)) return;
      {
        float f[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float L = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
          f[h] = kvsc / (kPScale * L);
          if (!pc.direct && sx.row == h) p.part_lse[pc.slot * kHeads + h] = m[h] + fast_log2(L);
        }
        if (sx.wi == 0) store16(reinterpret_cast<float*>(cx.g + L::kOffFac) + (k & 1u) * 16, f, lane);
      }
      // every warp sees the factors before any stores a block
      if (!group_sync(cx, sx)) return;
      po.pc = pc;
      po.k = k;
      po.blocks = 4;
      if (!have_next)  // the CTA's last piece: nothing left to overlap with
        while (po.blocks > 0)
          if (!pending_block(p, cx, sx, po)) return;
    }
    pc = nxt;
    have = have_next;
    ++k;
  }
}

template <bool kPaged>
using KvMaps = std::conditional_t<kPaged, PagedMaps, CUtensorMap>;

template <int QF, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1) stage1_tc_kernel(const Stage1Params p,
                                                                const __grid_constant__ KvMaps<kPaged> kvmap) {
  extern __shared__ uint8_t smem_raw[];
  Cx cx;
  PieceCursor cur;
  if (!cta_begin(p, cx, smem_raw, 1, cur)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // tiles start at multiples of 8 rows of their segment, so that with a paged
  // cache the 8-row groups line up with pages of 8k rows; the contiguous cache
  // uses the same tiles, so both forms give identical results
  cur.align8 = 1;
  if constexpr (kPaged) cur.pip = p.page_indptr;
  PagedDrain drain{0u, 0u, 0u};
  if (warp == 0) {
    if constexpr (kPaged)
      drain = producer_paged(p, cx, &kvmap, cur, lane);
    else
      producer(cx, &kvmap, cur, lane);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<kPaged>(cx, cur);
    __syncwarp();
  } else if (warp < 6) {
    softmax_role<QF, kPaged>(p, cx, cur, warp, lane);
  } else {
    if constexpr (kPaged) {
      if (warp == 6) prefetch_page_ids(p, cur, lane);
    }
    qprep_role<QF>(p, cx, cur, warp, lane);
  }
  if constexpr (kPaged) {
    __syncthreads();
    if (*cx.abort_word) drain_paged(cx, drain);
  }
  cta_end(p, cx, 1);
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

cudaError_t make_u8_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t pitch,
                        uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// box_rows = 128 (a whole tile) for a contiguous cache; 8, 16, .., 128 for the
// pool of a paged one.
cudaError_t make_kv_map(CUtensorMap* map, const void* kv, int64_t total_kv, uint32_t box_rows) {
  return make_u8_map(map, kv, kDqk, total_kv, kDqk, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The launch: a programmatic dependent of the kernel before it in the stream
// (with in-call q quantisation that kernel is the amax: the CTAs stream KV
// first and wait before reading the scale).
template <int QF, bool kPaged>
static cudaError_t launch_after(const Stage1Params& p, cudaStream_t stream, const KvMaps<kPaged>& maps) {
  return launch_dependent(stage1_tc_kernel<QF, kPaged>, p.num_splits, kThreads, L::kAlloc, stream, p, maps);
}

template <int QF, bool kPaged>
static cudaError_t launch_q(const Stage1Params& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(stage1_tc_kernel<QF, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if constexpr (kPaged) {
    // the 16 maps of a pool are encoded once per (device, pool) and reused
    thread_local int cached_dev = -1;
    thread_local const void* cached_kv = nullptr;
    thread_local int64_t cached_rows = -1;
    thread_local PagedMaps maps;
    const int64_t rows = static_cast<int64_t>(p.num_pages) * p.page_size;
    if (cached_dev != dev || cached_kv != p.kv || cached_rows != rows) {
      cached_dev = -1;
      for (uint32_t h = 0; h < 16; ++h) {
        e = make_kv_map(&maps.box[h], p.kv, rows, 8 * (h + 1));
        if (e != cudaSuccess) return e;
      }
      cached_dev = dev;
      cached_kv = p.kv;
      cached_rows = rows;
    }
    return launch_after<QF, kPaged>(p, stream, maps);
  } else {
    CUtensorMap map;
    e = make_kv_map(&map, p.kv, p.total_kv, kTileRows);
    if (e != cudaSuccess) return e;
    return launch_after<QF, kPaged>(p, stream, map);
  }
}

}  // namespace tc

cudaError_t launch_stage1_tc_fp8(int q_fmt, const Stage1Params& p, cudaStream_t stream) {
  if (p.paged) {
    if (q_fmt == kQBf16Quant) return tc::launch_q<kQBf16Quant, true>(p, stream);
    return q_fmt == kQBf16 ? tc::launch_q<kQBf16, true>(p, stream) : tc::launch_q<kQFp8, true>(p, stream);
  }
  if (q_fmt == kQBf16Quant) return tc::launch_q<kQBf16Quant, false>(p, stream);
  return q_fmt == kQBf16 ? tc::launch_q<kQBf16, false>(p, stream) : tc::launch_q<kQFp8, false>(p, stream);
}

}  // namespace mla
