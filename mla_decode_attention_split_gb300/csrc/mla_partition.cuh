// Even partition of all query-token x KV-row work over the stage-1 CTAs.
//
// Each query token t of segment b owns a run of "virtual rows", one per KV row
// of its segment: token-major, segment order. The total is
//   T = sum_b q_len_b * kv_len_b.
// CTA c of P processes virtual rows [c*T/P, (c+1)*T/P). A run of one token
// inside one CTA is a "piece"; its partial result goes to workspace slot
// c + t (unique, since along the virtual-row axis each new piece increments c,
// t or both). A token whose run lies inside a single CTA is written directly.
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
template <int kThreads, int kMode, class Target>
__device__ SegLocate block_locate(const int32_t* __restrict__ qo, const int32_t* __restrict__ kvp, int batch,
                                  int total_q, int total_kv, Target target, int token, int64_t* sh) {
  const int tid = threadIdx.x;
  const int per = (batch + kThreads - 1) / kThreads;
  const int lo = min(tid * per, batch), hi = min(lo + per, batch);
  int64_t local = 0;
  int valid = 1;
  for (int b = lo; b < hi; ++b) {
    const int32_t q0 = __ldg(qo + b), q1 = __ldg(qo + b + 1);
    const int32_t k0 = __ldg(kvp + b), k1 = __ldg(kvp + b + 1);
    valid &= (q1 >= q0) & (k1 >= k0);
    local += static_cast<int64_t>(q1 - q0) * static_cast<int64_t>(k1 - k0);
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
          const int64_t v = static_cast<int64_t>(__ldg(qo + b + 1) - __ldg(qo + b)) *
                            static_cast<int64_t>(__ldg(kvp + b + 1) - __ldg(kvp + b));
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
          vs += static_cast<int64_t>(q1 - q0) * static_cast<int64_t>(__ldg(kvp + b + 1) - __ldg(kvp + b));
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
  int32_t token;      // query token index
  int32_t kv_row;     // first absolute KV row of the piece
  int32_t nrows;      // rows in the piece (>= 1)
  int32_t direct;     // the piece is the token's whole run: write the output
  int64_t slot;       // partial slot (c + token) when not direct
  int64_t tok_vs;     // virtual start of the token's whole run
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

  __device__ __forceinline__ bool next(Piece& pc) {
    while (x < end && seg < batch) {
      const int32_t q0 = __ldg(qo + seg), q1 = __ldg(qo + seg + 1);
      const int32_t k0 = __ldg(kvp + seg), k1 = __ldg(kvp + seg + 1);
      const int64_t kvlen = k1 - k0;
      const int64_t vlen = static_cast<int64_t>(q1 - q0) * kvlen;
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
      pc.token = static_cast<int32_t>(q0 + ti);
      pc.kv_row = static_cast<int32_t>(k0 + row_in) - lead;
      pc.nrows = static_cast<int32_t>(stop - x) + lead;
      pc.lead = lead;
      pc.direct = (row_in == 0 && stop == tok_vs + kvlen) ? 1 : 0;
      pc.slot = cta + pc.token;
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
