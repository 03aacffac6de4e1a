// Even partition of all query-token x KV-row work over the stage-1 CTAs.
//
// The query tokens of a segment are taken in groups of G (G = 1, or 2 when a
// kernel shares one pass over the KV rows between two tokens; a segment's
// last group may be smaller). Each group of segment b owns a run of "virtual
// rows", one per KV row of its segment: group-major, segment order. The total
// is
//   T = sum_b ceil(q_len_b / G) * kv_len_b.
// CTA c of P processes virtual rows [c*T/P, (c+1)*T/P). A run of one group
// inside one CTA is a "piece"; the partial result of its token t goes to
// workspace slot G c + t. Slots are unique: along the virtual-row axis a new
// piece either moves to the next CTA (G c grows by G, at least the group's
// token count) or to the next group (t grows by the previous group's token
// count), so the slot ranges of successive pieces never overlap; there are
// G P + total_q slots. A group whose run lies inside a single CTA is written
// directly.
//
// Both kernels recompute T and locate their position with one block-wide scan
// over the indptr arrays; the scan also validates them (monotone, first entry
// 0, last entry = total) so no later access can leave the buffers.
#pragma once

#include <cstdint>

#include "mla_device.cuh"

namespace mla {

__device__ __forceinline__ int64_t part_start(int64_t c, int64_t total, int64_t parts) {
  return (c * total) / parts;
}

// The CTA whose range contains virtual row x (0 <= x < total).
__device__ __forceinline__ int64_t part_of_row(int64_t x, int64_t total, int64_t parts) {
  return ((x + 1) * parts - 1) / total;
}

struct SegLocate {
  int64_t total;     // T
  int32_t seg;       // located segment, -1 if none
  int64_t seg_vs;    // virtual start of that segment
  int32_t ok;        // indptrs passed the checks
};

template <int kThreads>
__device__ __forceinline__ int64_t block_exclusive_scan_i64(int64_t v, int64_t* sh /*[kThreads/32 + 1]*/,
                                                            int64_t& total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int64_t s = sh[w];
      sh[w] = run;
      run += s;
    }
    sh[kWarps] = run;
  }
  __syncthreads();
  total = sh[kWarps];
  const int64_t excl = sh[warp] + inc - v;
  __syncthreads();
  return excl;
}

// mode 1: locate the segment containing virtual row target(T) (target < T).
// mode 2: locate the segment containing query token `token`.
// All kThreads threads of the block must call this.
// Virtual rows of a segment with q query tokens and kv KV rows, tokens in groups of g.
__device__ __forceinline__ int64_t seg_vrows(int32_t q, int32_t kv, int32_t g) {
  return static_cast<int64_t>((q + g - 1) / g) * static_cast<int64_t>(kv);
}

template <int kThreads, int kMode, class Target>
__device__ SegLocate block_locate(const int32_t* __restrict__ qo, const int32_t* __restrict__ kvp, int batch,
                                  int total_q, int total_kv, int group, Target target, int token, int64_t* sh) {
  const int tid = threadIdx.x;
  const int per = (batch + kThreads - 1) / kThreads;
  const int lo = min(tid * per, batch), hi = min(lo + per, batch);
  int64_t local = 0;
  int valid = 1;
  for (int b = lo; b < hi; ++b) {
    const int32_t q0 = __ldg(qo + b), q1 = __ldg(qo + b + 1);
    const int32_t k0 = __ldg(kvp + b), k1 = __ldg(kvp + b + 1);
    valid &= (q1 >= q0) & (k1 >= k0);
    local += seg_vrows(q1 - q0, k1 - k0, group);
  }
  if (tid == 0) {
    valid &= (__ldg(qo) == 0) & (__ldg(kvp) == 0) & (__ldg(qo + batch) == total_q) &
             (__ldg(kvp + batch) == total_kv);
  }
  valid = __syncthreads_and(valid);
  int64_t total = 0;
  const int64_t excl = block_exclusive_scan_i64<kThreads>(valid ? local : 0, sh, total);
  int64_t* res = sh + kThreads / 32 + 1;  // res[0] = seg, res[1] = seg_vs
  if (tid == 0) res[0] = -1;
  __syncthreads();
  SegLocate out;
  out.ok = valid;
  out.total = total;
  if (valid) {
    if (kMode == 1) {
      const int64_t x = target(total);
      if (lo < hi && x >= excl && x < excl + local) {
        int64_t vs = excl;
        for (int b = lo; b < hi; ++b) {
          const int64_t v = seg_vrows(__ldg(qo + b + 1) - __ldg(qo + b), __ldg(kvp + b + 1) - __ldg(kvp + b), group);
          if (x < vs + v) {
            res[0] = b;
            res[1] = vs;
            break;
          }
          vs += v;
        }
      }
    } else {
      if (lo < hi && token >= __ldg(qo + lo) && token < __ldg(qo + hi)) {
        int64_t vs = excl;
        for (int b = lo; b < hi; ++b) {
          const int32_t q0 = __ldg(qo + b), q1 = __ldg(qo + b + 1);
          if (token >= q0 && token < q1) {
            res[0] = b;
            res[1] = vs;
            break;
          }
          vs += seg_vrows(q1 - q0, __ldg(kvp + b + 1) - __ldg(kvp + b), group);
        }
      }
    }
  }
  __syncthreads();
  out.seg = static_cast<int32_t>(res[0]);
  out.seg_vs = res[1];
  __syncthreads();
  return out;
}

// Walks the pieces of one CTA's range in order. Every thread of the CTA runs
// an identical cursor, so all roles see the same sequence of pieces.
struct Piece {
  int32_t token;      // first query token of the group
  int32_t ntok;       // tokens in the group (1..G)
  int32_t kv_row;     // first absolute KV row of the piece
  int32_t nrows;      // rows in the piece (>= 1)
  int32_t direct;     // the piece is the group's whole run: write the output
  int64_t slot;       // partial slot of the first token (G c + token; token i: + i) when not direct
  int64_t tok_vs;     // virtual start of the group's whole run
  int32_t kvlen;      // its length (the segment's KV rows)
  int32_t seg;        // segment index
  int32_t k0;         // first KV row of the segment
  int32_t lead;       // rows before the piece that its first tile also covers (see align8)
  int32_t pbase;      // paged KV: the segment's first page-table entry (0 otherwise)
};

struct PieceCursor {
  const int32_t* qo;
  const int32_t* kvp;
  int32_t batch;
  int64_t x, end;     // next virtual row, end of this CTA's range
  int32_t seg;        // current segment
  int64_t seg_vs;     // its virtual start
  int64_t cta;
  // nonzero: a piece's rows are taken from the multiple of 8 (counted from the
  // segment's first row) at or before its start; the extra `lead` rows belong
  // to the same segment and are masked by the consumer
  int32_t align8;
  // paged KV: page_indptr, read with the segment's other offsets (else null)
  const int32_t* pip;
  // tokens per group (values below 1 count as 1)
  int32_t group;

  __device__ __forceinline__ bool next(Piece& pc) {
    const int32_t G = group > 1 ? group : 1;
    while (x < end && seg < batch) {
      const int32_t q0 = __ldg(qo + seg), q1 = __ldg(qo + seg + 1);
      const int32_t k0 = __ldg(kvp + seg), k1 = __ldg(kvp + seg + 1);
      const int64_t kvlen = k1 - k0;
      const int64_t vlen = seg_vrows(q1 - q0, k1 - k0, G);
      if (x >= seg_vs + vlen) {  // past this segment (or it is empty)
        seg_vs += vlen;
        ++seg;
        continue;
      }
      const int64_t ti = (x - seg_vs) / kvlen;
      const int64_t tok_vs = seg_vs + ti * kvlen;
      const int64_t row_in = x - tok_vs;
      const int64_t stop = min(end, tok_vs + kvlen);
      const int32_t lead = align8 ? static_cast<int32_t>(row_in & 7) : 0;
      pc.token = static_cast<int32_t>(q0 + G * ti);
      pc.ntok = min(G, q1 - pc.token);
      pc.kv_row = static_cast<int32_t>(k0 + row_in) - lead;
      pc.nrows = static_cast<int32_t>(stop - x) + lead;
      pc.lead = lead;
      pc.direct = (row_in == 0 && stop == tok_vs + kvlen) ? 1 : 0;
      pc.slot = G * cta + pc.token;
      pc.tok_vs = tok_vs;
      pc.kvlen = static_cast<int32_t>(kvlen);
      pc.seg = seg;
      pc.k0 = k0;
      pc.pbase = pip ? __ldg(pip + seg) : 0;
      x = stop;
      return true;
    }
    return false;
  }
};

}  // namespace mla
