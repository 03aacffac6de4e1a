// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

namespace mla {

constexpr int kHeads = 16;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kMxBlock = 32;

// Workspace layout: [header 256 B: word 0 = error flags, word 1 = token count
// of the last call that used the counters][token counters: total_q u32, padded
// to 256 B][part_o: slots x 16 x 512 f32][part_lse: slots x 16 f32], slots =
// num_splits + total_q. The counters are zero between calls.
constexpr size_t kHeaderBytes = 256;
inline size_t counter_bytes(int64_t total_q) { return static_cast<size_t>((total_q * 4 + 255) / 256) * 256; }

struct Stage1Params {
  const void* q;
  const void* kv;
  const void* kv_scale;
  const float* q_scale;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  int32_t batch;
  int32_t total_q;
  int32_t total_kv;
  int32_t num_splits;
  float sm_scale;
  void* out;          // bf16 [total_q][16][512]
  float* part_o;      // [slots][16][512]
  float* part_lse;    // [slots][16] (log2 domain)
  uint32_t* dev_flags;
  uint32_t* tok_cnt;  // [total_q] partials finished per token
  // paged KV: kv is [num_pages][page_size][576]; kv_indptr then holds the
  // logical row offsets built from the page table (mla_paged.cu)
  const int32_t* page_indptr;   // [batch+1] page-table entries of each segment
  const int32_t* page_indices;  // page ids
  int32_t page_size;
  int32_t page_shift;  // log2(page_size) when it is a power of two, else -1
  int32_t num_pages;
  int32_t paged;
  int32_t group;      // query tokens per group sharing a pass over the KV rows (1, 2 or 4)
  int32_t wait_late;  // the kernel just before is this call's q amax: wait for it only before reading the scale
  // nonzero when every CTA of the launch is resident at once (num_splits <= SM count, one CTA per SM):
  // the CTAs that hold pieces of a split token then share its merge at their end (merge_coop)
  int32_t coop_merge;
};

// KV formats / query formats as template tags (values match mla_dtype_t).
enum KvFormat : int { kKvBf16 = 0, kKvFp8 = 1, kKvMxfp4 = 2 };
enum QFormat : int { kQBf16 = 0, kQFp8 = 1, kQBf16Quant = 2 /* bf16 q quantised to e4m3 in setup */ };

// Header words of the workspace.
enum HeaderWord : int { kHdrFlags = 0, kHdrCounters = 1, kHdrQAmax = 2, kHdrQScale = 3, kHdrQBlocks = 4 };

cudaError_t launch_stage1(int kv_fmt, int q_fmt, const Stage1Params& p, cudaStream_t stream);
// fp8 KV on the tcgen05 tensor cores (mla_stage1_tc.cu)
cudaError_t launch_stage1_tc_fp8(int q_fmt, const Stage1Params& p, cudaStream_t stream);
// bf16 KV on the tcgen05 tensor cores (mla_stage1_bf.cu)
cudaError_t launch_stage1_tc_bf16(int q_fmt, const Stage1Params& p, cudaStream_t stream);
// mxfp4 KV on the tcgen05 tensor cores (mla_stage1_mx.cu)
cudaError_t launch_stage1_tc_mxfp4(int q_fmt, const Stage1Params& p, cudaStream_t stream);
cudaError_t launch_dequant(const void* kv, const void* kv_scale, int kv_fmt, int32_t total_kv, int32_t row0,
                           int32_t nrows, float* out, cudaStream_t stream);
bool stage1_supported(int kv_fmt, int q_fmt);
// fp8 KV and bf16 q, query tokens of a segment in pairs sharing each KV tile (p.group = 2;
// mla_stage1_pair.cu)
cudaError_t launch_stage1_pair(const Stage1Params& p, cudaStream_t stream);
// fp8 KV and fp8 q, query tokens of a segment in groups of four sharing each KV tile (p.group = 4;
// mla_stage1_quad.cu)
cudaError_t launch_stage1_quad(int q_fmt, const Stage1Params& p, cudaStream_t stream);
// fp8 KV and fp8 q, token pairs with the two tokens' softmax in two warp groups (p.group = 2;
// mla_stage1_duo.cu)
cudaError_t launch_stage1_duo(int q_fmt, const Stage1Params& p, cudaStream_t stream);
// amax of bf16 q over n elements -> header word kHdrQScale = max(amax, 1e-12) / 448 (mla_qquant.cu)
cudaError_t launch_q_scale(const void* q, int64_t n, uint32_t* header, cudaStream_t stream);
// paged KV: logical row offsets [batch+1] from the page table (mla_paged.cu)
cudaError_t launch_paged_prepare(const int32_t* page_indptr, const int32_t* last_page_len, int32_t batch,
                                 int32_t page_size, int32_t* kv_indptr_out, uint32_t* flags, cudaStream_t stream);
// bytes after the decode workspace for the logical row offsets of a paged call
inline size_t paged_extra_bytes(int64_t batch) { return static_cast<size_t>(((batch + 1) * 4 + 255) / 256) * 256; }


// Launches a stage-1 kernel as a programmatic dependent of the kernel before it
// in the stream (programmatic stream serialization): its CTAs may be placed
// while that kernel ends; each waits (griddepcontrol.wait) before it touches
// global memory that the kernel before may write.
template <class... KArgs, class... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), int grid, int block, int smem, cudaStream_t stream,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline size_t workspace_bytes_for(int64_t num_splits, int64_t total_q) {
  const int64_t slots = num_splits + total_q;
  return kHeaderBytes + counter_bytes(total_q) + static_cast<size_t>(slots) * kHeads * kDv * sizeof(float) +
         static_cast<size_t>(slots) * kHeads * sizeof(float);
}

}  // namespace mla
