// C-ABI entry points of the MLA decode library (declared in mla_decode.h):
// argument checks, the split planner, workspace carving and kernel launches.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "mla_decode.h"
#include "mla_internal.h"

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

int sm_count_of_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int32_t kMaxSplits = 4096;

// Split planner: a cost model of the slowest CTA, in units of one 128-row
// tile of streaming. A "piece" is one token's run of rows inside one CTA.
//  * Every piece a CTA holds costs kPieceCost more (query setup, epilogue,
//    partial write and count), and a piece that does not start on an 8-row
//    boundary of its segment may take one more tile.
//  * The CTA that merges a token reads one partial per split of it
//    (kMergeCost each).
//  * P a multiple of the token count gives every CTA one piece of one
//    segment; P a divisor of it gives every CTA whole segments. Otherwise the
//    worst CTA straddles a boundary and holds one piece more.
// Segments are taken as equally long (the planner sees only the totals).
// Constants from decode timings on the fp8 tensor-core kernel over split
// counts: one piece costs about 4 tiles, one merged partial a quarter tile.
// With query tokens in groups of g sharing each pass, a unit of work is a
// group, and its merge reads g partials per split.
constexpr double kPieceCost = 4.0, kMergeCost = 0.25;

double split_cost(int64_t p, int64_t nseg, int64_t lv, int64_t g) {
  if (p % nseg == 0) {  // k CTAs per segment, one piece each
    const int64_t k = p / nseg;
    const int64_t rows = (lv + k - 1) / k;
    const int64_t lead = (lv % k == 0 && (lv / k) % 8 == 0) ? 0 : 7;
    return kPieceCost + static_cast<double>((rows + lead + 127) / 128) + (k > 1 ? kMergeCost * k * g : 0.0);
  }
  if (nseg % p == 0) {  // whole segments per CTA, no merges
    const int64_t j = nseg / p;
    return static_cast<double>(j) * (kPieceCost + static_cast<double>((lv + 127) / 128));
  }
  const double r = static_cast<double>(nseg) * static_cast<double>(lv) / static_cast<double>(p);
  const double lvd = static_cast<double>(lv);
  const double pieces = std::min(static_cast<double>(nseg), std::ceil(r / lvd) + 1.0);
  const double tiles = std::ceil(r / 128.0) + pieces;
  const double k = r < lvd ? std::ceil(lvd / r) + 1.0 : 2.0;
  return kPieceCost * pieces + tiles + kMergeCost * k * g;
}

int32_t plan_splits(int64_t total_q, int64_t batch, int64_t total_kv, int sm_count, int64_t group = 1) {
  if (sm_count <= 0) sm_count = 1;
  if (total_q <= 0 || batch <= 0 || total_kv <= 0) return 1;
  // one unit of work per group of query tokens: its segment's rows (average length)
  const int64_t g = group > 1 ? group : 1;
  const int64_t nseg = (total_q + g - 1) / g;
  const int64_t lv = std::max<int64_t>(1, total_kv / batch);
  const int64_t maxp = std::min<int64_t>(sm_count, nseg * lv);  // at least one row per CTA
  int64_t best = 1;
  double best_cost = split_cost(1, nseg, lv, g);
  for (int64_t p = 2; p <= maxp; ++p) {
    const double c = split_cost(p, nseg, lv, g);
    if (c <= best_cost + 1e-9) {  // ties go to more CTAs
      best = p;
      best_cost = std::min(best_cost, c);
    }
  }
  return static_cast<int32_t>(best);
}

size_t kv_bytes(mla_dtype_t dt, int64_t total_kv) {
  switch (dt) {
    case MLA_DTYPE_BF16: return static_cast<size_t>(total_kv) * MLA_D_QK * 2;
    case MLA_DTYPE_FP8_E4M3: return static_cast<size_t>(total_kv) * MLA_D_QK;
    case MLA_DTYPE_MXFP4: return static_cast<size_t>(total_kv) * (MLA_D_QK / 2);
  }
  return 0;
}

}  // namespace

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: unsupported dtype combination";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA runtime error";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded device wait expired";
    case MLA_ERR_DEVICE_CHECK: return "MLA_ERR_DEVICE_CHECK: indptr arrays failed the device checks";
    case MLA_ERR_TOO_LARGE:
      return "MLA_ERR_TOO_LARGE: the call needs more scratch than the library's fixed device array holds";
  }
  return "unknown mla_status_t";
}

mla_status_t mla_plan(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype, int32_t sm_count,
                      int32_t* num_splits) {
  (void)kv_dtype;
  if (!num_splits || batch < 0 || total_q < 0 || total_kv < 0) return MLA_ERR_INVALID_ARG;
  if (sm_count <= 0) sm_count = sm_count_of_current_device();
  *num_splits = plan_splits(total_q, batch, total_kv, sm_count);
  return MLA_OK;
}

mla_status_t mla_decode_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                                       int32_t num_splits, size_t* bytes) {
  if (!bytes || batch < 0 || total_q < 0 || total_kv < 0 || num_splits < 0 || num_splits > kMaxSplits)
    return MLA_ERR_INVALID_ARG;
  if (num_splits == 0) {
    const mla_status_t st = mla_plan(batch, total_q, total_kv, kv_dtype, 0, &num_splits);
    if (st != MLA_OK) return st;
  }
  *bytes = mla::workspace_bytes_for(num_splits, total_q);
  return MLA_OK;
}

}  // extern "C"

namespace {

// Shared by mla_decode and mla_decode_paged. With a page table (pg != NULL)
// kv_indptr is ignored: the logical row offsets are built on the device into
// the workspace, after the part mla_decode_workspace_size covers.
mla_status_t decode_impl(const void* q, const void* kv, const void* kv_scale, const int32_t* qo_indptr,
                         const int32_t* kv_indptr, void* out, mla_dtype_t kv_dtype, const mla_decode_opts* opts,
                         const mla_paged_kv* pg, void* stream) {
  if (!opts) return MLA_ERR_INVALID_ARG;
  const int32_t batch = opts->batch, total_q = opts->total_q, total_kv = opts->total_kv;
  if (batch < 1 || total_q < 0 || total_kv < 0) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_DTYPE_BF16 && kv_dtype != MLA_DTYPE_FP8_E4M3 && kv_dtype != MLA_DTYPE_MXFP4)
    return MLA_ERR_INVALID_ARG;
  if (opts->q_dtype != MLA_DTYPE_BF16 && opts->q_dtype != MLA_DTYPE_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (!qo_indptr || (!pg && !kv_indptr)) return MLA_ERR_INVALID_ARG;
  if (pg) {
    if (pg->page_size < 1 || pg->num_pages < 0 || !pg->page_indptr || !pg->page_indices ||
        (pg->page_size > 1 && !pg->last_page_len) || (total_kv > 0 && pg->num_pages < 1) ||
        static_cast<int64_t>(pg->num_pages) * pg->page_size > INT32_MAX)
      return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_DTYPE_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
  }
  if (total_q > 0 && (!q || !out || !aligned16(q) || !aligned16(out))) return MLA_ERR_INVALID_ARG;
  if (total_kv > 0 && (!kv || !aligned16(kv))) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_DTYPE_BF16 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_DTYPE_MXFP4 && !aligned16(kv_scale)) return MLA_ERR_INVALID_ARG;
  if (opts->q_dtype == MLA_DTYPE_FP8_E4M3 && !opts->q_scale) return MLA_ERR_INVALID_ARG;
  if (opts->quantize_q && opts->q_dtype != MLA_DTYPE_BF16) return MLA_ERR_UNSUPPORTED;
  // query tokens per KV pass: 1, 2 (fp8 or bf16 KV) or 4 (fp8 KV with fp8 q)
  const int32_t G = opts->token_group <= 1 ? 1 : opts->token_group;
  if (opts->token_group < 0 || (G != 1 && G != 2 && G != 4)) return MLA_ERR_INVALID_ARG;
  if (G > 1 && (kv_dtype == MLA_DTYPE_MXFP4 || pg)) return MLA_ERR_UNSUPPORTED;
  const int q_fmt = opts->quantize_q ? static_cast<int>(mla::kQBf16Quant) : static_cast<int>(opts->q_dtype);
  if (G == 4 && (kv_dtype != MLA_DTYPE_FP8_E4M3 || q_fmt == mla::kQBf16)) return MLA_ERR_UNSUPPORTED;
  if (!mla::stage1_supported(kv_dtype, q_fmt)) return MLA_ERR_UNSUPPORTED;
  int32_t splits = opts->num_splits;
  if (splits < 0 || splits > kMaxSplits) return MLA_ERR_INVALID_ARG;
  if (splits == 0) splits = plan_splits(total_q, batch, total_kv, sm_count_of_current_device(), G);
  // G tokens per group: G num_splits + total_q partial slots
  const size_t base = mla::workspace_bytes_for(G * static_cast<int64_t>(splits), total_q);
  const size_t need = base + (pg ? mla::paged_extra_bytes(batch) : 0);
  if (!opts->workspace || opts->workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(opts->workspace) & 255u) != 0)
    return MLA_ERR_WORKSPACE;
  if (total_q == 0) return MLA_OK;

  mla::Stage1Params p;
  p.q = q;
  p.kv = kv;
  p.kv_scale = kv_scale;
  p.q_scale = opts->quantize_q ? reinterpret_cast<const float*>(static_cast<uint32_t*>(opts->workspace) + mla::kHdrQScale)
                               : opts->q_scale;
  p.qo_indptr = qo_indptr;
  p.kv_indptr = pg ? reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(opts->workspace) + base) : kv_indptr;
  p.paged = pg ? 1 : 0;
  p.page_indptr = pg ? pg->page_indptr : nullptr;
  p.page_indices = pg ? pg->page_indices : nullptr;
  p.page_size = pg ? pg->page_size : 0;
  p.wait_late = (!pg && opts->quantize_q) ? 1 : 0;
  p.group = G;
  // the cooperative merge pays when a group's merge is spread over two or more CTAs on average; it needs
  // every CTA resident at once (one CTA per SM)
  const int64_t groups = (static_cast<int64_t>(total_q) + G - 1) / G;
  p.coop_merge = (splits <= sm_count_of_current_device() && 2 * groups <= splits) ? 1 : 0;
  p.page_shift = -1;
  for (int32_t sh = 0; sh < 31 && pg; ++sh)
    if ((int32_t{1} << sh) == pg->page_size) p.page_shift = sh;
  p.num_pages = pg ? pg->num_pages : 0;
  p.batch = batch;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.num_splits = splits;
  p.sm_scale = opts->sm_scale > 0.f ? opts->sm_scale : static_cast<float>(1.0 / std::sqrt(576.0));
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(opts->workspace);
  p.dev_flags = reinterpret_cast<uint32_t*>(ws);
  const int64_t slots = G * static_cast<int64_t>(splits) + total_q;
  p.tok_cnt = reinterpret_cast<uint32_t*>(ws + mla::kHeaderBytes);
  p.part_o = reinterpret_cast<float*>(ws + mla::kHeaderBytes + mla::counter_bytes(total_q));
  p.part_lse = p.part_o + slots * mla::kHeads * mla::kDv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    return !opts->profile_events[i] ||
           cudaEventRecord(static_cast<cudaEvent_t>(opts->profile_events[i]), st) == cudaSuccess;
  };
  if (!mark(0)) return MLA_ERR_CUDA;
  // one launch: stage 1 also merges split tokens and zeroes tokens of empty
  // segments; with no KV rows at all every output row is zero
  if (total_kv > 0) {
    if (pg && mla::launch_paged_prepare(pg->page_indptr, pg->last_page_len, batch, pg->page_size,
                                        const_cast<int32_t*>(p.kv_indptr), p.dev_flags, st) != cudaSuccess)
      return MLA_ERR_CUDA;
    if (opts->quantize_q &&
        mla::launch_q_scale(q, static_cast<int64_t>(total_q) * mla::kHeads * mla::kDqk, p.dev_flags, st) != cudaSuccess)
      return MLA_ERR_CUDA;
    // fp8 KV groups have their own kernels; the bf16 kernel takes p.group itself
    const bool fp8 = kv_dtype == MLA_DTYPE_FP8_E4M3;
    const bool q8 = q_fmt != mla::kQBf16;
    const cudaError_t le = (G == 4)                 ? mla::launch_stage1_quad(q_fmt, p, st)
                           : (G == 2 && fp8 && q8) ? mla::launch_stage1_duo(q_fmt, p, st)
                           : (G == 2 && fp8)       ? mla::launch_stage1_pair(p, st)
                                                   : mla::launch_stage1(kv_dtype, q_fmt, p, st);
    if (le != cudaSuccess) return MLA_ERR_CUDA;
  } else if (cudaMemsetAsync(out, 0, static_cast<size_t>(total_q) * mla::kHeads * mla::kDv * 2, st) != cudaSuccess) {
    return MLA_ERR_CUDA;
  }
  if (!mark(1)) return MLA_ERR_CUDA;
  if (!mark(2)) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode(const void* q, const void* kv, const void* kv_scale, const int32_t* qo_indptr,
                        const int32_t* kv_indptr, void* out, mla_dtype_t kv_dtype, const mla_decode_opts* opts,
                        void* stream) {
  return decode_impl(q, kv, kv_scale, qo_indptr, kv_indptr, out, kv_dtype, opts, nullptr, stream);
}

mla_status_t mla_decode_group_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                                             int32_t num_splits, int32_t token_group, size_t* bytes) {
  if (!bytes || batch < 0 || total_q < 0 || total_kv < 0 || num_splits < 0 || num_splits > kMaxSplits ||
      token_group < 0 || (token_group > 2 && token_group != 4))
    return MLA_ERR_INVALID_ARG;
  const int64_t g = token_group > 1 ? token_group : 1;
  if (num_splits == 0) num_splits = plan_splits(total_q, batch, total_kv, sm_count_of_current_device(), g);
  *bytes = mla::workspace_bytes_for(g * num_splits, total_q);
  return MLA_OK;
}

mla_status_t mla_decode_pairs_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                                             int32_t num_splits, size_t* bytes) {
  return mla_decode_group_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, 2, bytes);
}

mla_status_t mla_decode_paged_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                                             int32_t num_splits, size_t* bytes) {
  const mla_status_t st = mla_decode_workspace_size(batch, total_q, total_kv, kv_dtype, num_splits, bytes);
  if (st == MLA_OK) *bytes += mla::paged_extra_bytes(batch);
  return st;
}

mla_status_t mla_decode_paged(const void* q, const void* kv_pages, const void* kv_scale, const int32_t* qo_indptr,
                              const mla_paged_kv* paged, void* out, mla_dtype_t kv_dtype,
                              const mla_decode_opts* opts, void* stream) {
  if (!paged) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv_pages, kv_scale, qo_indptr, nullptr, out, kv_dtype, opts, paged, stream);
}

mla_status_t mla_decode_from_host(const void* h_q, const void* h_kv, const void* h_kv_scale, const float* h_q_scale,
                                  const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, void* h_out,
                                  mla_dtype_t kv_dtype, const mla_decode_opts* opts, const mla_device_buffers* dev,
                                  void* stream) {
  if (!opts || !dev || !h_qo_indptr || !h_kv_indptr) return MLA_ERR_INVALID_ARG;
  const int64_t batch = opts->batch, total_q = opts->total_q, total_kv = opts->total_kv;
  if (batch < 1 || total_q < 0 || total_kv < 0) return MLA_ERR_INVALID_ARG;
  if ((total_q > 0 && (!h_q || !h_out || !dev->q || !dev->out)) || (total_kv > 0 && (!h_kv || !dev->kv)) ||
      !dev->qo_indptr || !dev->kv_indptr)
    return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t qbytes = static_cast<size_t>(total_q) * MLA_NUM_HEADS * MLA_D_QK *
                        (opts->q_dtype == MLA_DTYPE_BF16 ? 2 : 1);
  auto h2d = [&](void* d, const void* h, size_t n) {
    return n == 0 || cudaMemcpyAsync(d, h, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  bool ok = h2d(dev->q, h_q, qbytes) && h2d(dev->kv, h_kv, kv_bytes(kv_dtype, total_kv)) &&
            h2d(dev->qo_indptr, h_qo_indptr, sizeof(int32_t) * (batch + 1)) &&
            h2d(dev->kv_indptr, h_kv_indptr, sizeof(int32_t) * (batch + 1));
  if (ok && kv_dtype == MLA_DTYPE_FP8_E4M3) {
    if (!h_kv_scale || !dev->kv_scale) return MLA_ERR_INVALID_ARG;
    ok = h2d(dev->kv_scale, h_kv_scale, sizeof(float));
  } else if (ok && kv_dtype == MLA_DTYPE_MXFP4) {
    if ((!h_kv_scale || !dev->kv_scale) && total_kv > 0) return MLA_ERR_INVALID_ARG;
    ok = h2d(dev->kv_scale, h_kv_scale, static_cast<size_t>(total_kv) * (MLA_D_QK / MLA_MX_BLOCK));
  }
  if (ok && opts->q_dtype == MLA_DTYPE_FP8_E4M3) {
    if (!h_q_scale || !dev->q_scale) return MLA_ERR_INVALID_ARG;
    ok = h2d(dev->q_scale, h_q_scale, sizeof(float));
  }
  if (!ok) return MLA_ERR_CUDA;
  mla_decode_opts o = *opts;
  o.q_scale = dev->q_scale;
  const mla_status_t s = mla_decode(dev->q, dev->kv, dev->kv_scale, dev->qo_indptr, dev->kv_indptr, dev->out,
                                    kv_dtype, &o, stream);
  if (s != MLA_OK) return s;
  const size_t obytes = static_cast<size_t>(total_q) * MLA_NUM_HEADS * MLA_D_V * 2;
  if (obytes && cudaMemcpyAsync(h_out, dev->out, obytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_dequant_rows(const void* kv, const void* kv_scale, mla_dtype_t kv_dtype, int32_t total_kv,
                              int32_t row0, int32_t nrows, float* d_out, void* stream) {
  if (!kv || !d_out || !aligned16(kv) || total_kv < 0 || row0 < 0 || nrows < 0 ||
      static_cast<int64_t>(row0) + nrows > total_kv)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_DTYPE_MXFP4 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_DTYPE_BF16 && kv_dtype != MLA_DTYPE_FP8_E4M3 && kv_dtype != MLA_DTYPE_MXFP4)
    return MLA_ERR_INVALID_ARG;
  if (mla::launch_dequant(kv, kv_scale, kv_dtype, total_kv, row0, nrows, d_out, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_get_device_error(const void* workspace, void* stream, uint32_t* flags) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  uint32_t f = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&f, workspace, sizeof(f), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (flags) *flags = f;
  if (f & MLA_DEVFLAG_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (f & (MLA_DEVFLAG_BAD_INDPTR | MLA_DEVFLAG_BAD_PAGE)) return MLA_ERR_DEVICE_CHECK;
  return MLA_OK;
}

mla_status_t mla_reset_device_error(void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // header word 1: how many token counters the last call used (they may be
  // left part-counted when a call stopped on an error)
  uint32_t words[2] = {0u, 0u};
  if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  const size_t n = mla::kHeaderBytes + mla::counter_bytes(words[1]);
  if (cudaMemsetAsync(workspace, 0, n, st) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_validate_inputs(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                                 int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype, const void* kv_scale,
                                 void* stream, int64_t* bad_index) {
  if (bad_index) *bad_index = -1;
  if (!qo_indptr || !kv_indptr || batch < 1 || total_q < 0 || total_kv < 0) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_DTYPE_BF16 && kv_dtype != MLA_DTYPE_FP8_E4M3 && kv_dtype != MLA_DTYPE_MXFP4)
    return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n = static_cast<size_t>(batch) + 1;
  std::vector<int32_t> qo(n), kvp(n);
  if (cudaMemcpyAsync(qo.data(), qo_indptr, n * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(kvp.data(), kv_indptr, n * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MLA_ERR_CUDA;
  // the first offending entry of qo_indptr, then of kv_indptr (index batch + 1 + i)
  auto first_bad = [&](const std::vector<int32_t>& a, int32_t total) -> int64_t {
    if (a[0] != 0) return 0;
    for (size_t i = 1; i < n; ++i)
      if (a[i] < a[i - 1]) return static_cast<int64_t>(i);
    if (a[n - 1] != total) return static_cast<int64_t>(n - 1);
    return -1;
  };
  int64_t bad = first_bad(qo, total_q);
  if (bad < 0) {
    bad = first_bad(kvp, total_kv);
    if (bad >= 0) bad += static_cast<int64_t>(n);
  }
  if (bad >= 0) {
    if (bad_index) *bad_index = bad;
    return MLA_ERR_DEVICE_CHECK;
  }
  if (kv_dtype == MLA_DTYPE_MXFP4 && total_kv > 0) {
    // e8m0 0xFF is NaN: the decode's output for such a row is unspecified
    if (!kv_scale) return MLA_ERR_INVALID_ARG;
    const size_t nb = static_cast<size_t>(total_kv) * (MLA_D_QK / MLA_MX_BLOCK);
    constexpr size_t kChunk = size_t{1} << 20;
    std::vector<uint8_t> buf(std::min(nb, kChunk));
    for (size_t off = 0; off < nb; off += kChunk) {
      const size_t len = std::min(kChunk, nb - off);
      if (cudaMemcpyAsync(buf.data(), static_cast<const uint8_t*>(kv_scale) + off, len, cudaMemcpyDeviceToHost,
                          st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        return MLA_ERR_CUDA;
      for (size_t i = 0; i < len; ++i)
        if (buf[i] == 0xFFu) {
          if (bad_index) *bad_index = static_cast<int64_t>(2 * n + off + i);
          return MLA_ERR_DEVICE_CHECK;
        }
    }
  }
  return MLA_OK;
}

mla_status_t mla_event_elapsed_ms(void* ev_start, void* ev_end, float* ms) {
  if (!ev_start || !ev_end || !ms) return MLA_ERR_INVALID_ARG;
  if (cudaEventSynchronize(static_cast<cudaEvent_t>(ev_end)) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaEventElapsedTime(ms, static_cast<cudaEvent_t>(ev_start), static_cast<cudaEvent_t>(ev_end)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The allocation-free variant: the workspace is this fixed device array.
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

// Device address of g_static_workspace on each device, looked up on the first
// call made with that device current (the host-side symbol is not an address).
void* g_static_ws_ptr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" mla_status_t mla_decode_static_workspace(const void* q, const void* kv, const void* kv_scale,
                                                    const int32_t* qo_indptr, const int32_t* kv_indptr, void* out,
                                                    mla_dtype_t kv_dtype, const mla_decode_opts* opts, void* stream) {
  if (!opts) return MLA_ERR_INVALID_ARG;
  if (opts->batch < 1 || opts->total_q < 0 || opts->total_kv < 0 || opts->num_splits < 0 ||
      opts->num_splits > kMaxSplits)
    return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  if (!g_static_ws_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return MLA_ERR_CUDA;
    g_static_ws_ptr[dev] = ptr;
  }
  if (opts->token_group < 0 || (opts->token_group > 2 && opts->token_group != 4)) return MLA_ERR_INVALID_ARG;
  mla_decode_opts o = *opts;
  if (o.num_splits == 0)
    o.num_splits = plan_splits(o.total_q, o.batch, o.total_kv, sm_count_of_current_device(),
                               o.token_group > 1 ? o.token_group : 1);
  const int64_t slot_splits = (o.token_group > 1 ? o.token_group : 1) * static_cast<int64_t>(o.num_splits);
  if (mla::workspace_bytes_for(slot_splits, o.total_q) > MLA_STATIC_WORKSPACE_BYTES) return MLA_ERR_TOO_LARGE;
  // the error flags and the token counters are the scratch that must start at zero
  if (cudaMemsetAsync(g_static_ws_ptr[dev], 0, mla::kHeaderBytes + mla::counter_bytes(o.total_q),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  o.workspace = g_static_ws_ptr[dev];
  o.workspace_bytes = MLA_STATIC_WORKSPACE_BYTES;
  return mla_decode(q, kv, kv_scale, qo_indptr, kv_indptr, out, kv_dtype, &o, stream);
}

extern "C" mla_status_t mla_static_workspace_device_error(void* stream, uint32_t* flags) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  if (flags) *flags = 0;
  // no call on this device yet: nothing can have set a flag
  if (!g_static_ws_ptr[dev]) return MLA_OK;
  return mla_get_device_error(g_static_ws_ptr[dev], stream, flags);
}
