/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * The operation is DeepSeek-R1 forward_absorb Multi-head Latent Attention
 * decode as stated on kernelbot-amd-mixed-mla-675627 ("MLA decode kernel --
 * submission template", the module docstring: config block, KV buffer format,
 * input tuple and output; the naive reference `custom_kernel_bf16` gives the
 * arithmetic):
 *
 *   for each batch entry b, query token t in [qo_indptr[b], qo_indptr[b+1]),
 *   head h in [0,16):
 *     s_j      = sm_scale * <q[t,h,0:576], K_j>,   K_j = dequant(kv[j, 0:576])
 *     out[t,h] = sum_j softmax_j(s) * V_j,          V_j = K_j[0:512]
 *   for j in [kv_indptr[b], kv_indptr[b+1]).
 *
 * All query tokens of a segment attend to all of its KV rows (no causal
 * mask); a segment with no KV rows yields zeros. The computation is split-K
 * flash decoding: the KV rows of all segments are partitioned evenly over
 * `num_splits` CTAs (stage 1: fused QK^T + online softmax + PV with fp8/mxfp4
 * dequantisation in the operand path), and per-split partial outputs are merged
 * with LSE weights (the pages' stage 2), as in kernelbot-amd-mixed-mla-753817
 * (module docstring, `mla_flash_decode_stage1`, `mla_flash_decode_stage2`).
 * The merge runs inside the same launch: the CTA that finishes a token's last
 * partial merges it, so one decode call is one kernel launch (two with
 * in-call q quantisation or a page table: a small kernel runs first).
 *
 * Conventions for every entry point:
 *   - Pointers named d_* or documented "device" are CUDA device pointers that
 *     the caller owns; the library never frees or retains them. Host pointers
 *     are documented as such.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Calls that launch work are asynchronous: MLA_OK means "enqueued". A launch
 *     failure returns MLA_ERR_CUDA. No call synchronises unless documented.
 *   - The library allocates no device memory per call. It keeps only a cached
 *     per-device SM count, the kernels' shared-memory attributes and (per host
 *     thread) the tensor maps of the last paged pool.
 *   - Decode kernels are launched as programmatic dependents of the kernel
 *     before them in `stream` (programmatic stream serialization): their CTAs
 *     may be placed while that kernel ends, and they wait for it to complete
 *     before reading or writing global memory. Stream order is kept as for a
 *     normal launch. A kernel the caller launches after a decode call with the
 *     same attribute must itself wait (griddepcontrol.wait /
 *     cudaGridDependencySynchronize) before it reads `out`.
 *   - Calls make no allocation or synchronisation inside, so they can be
 *     captured into a CUDA graph.
 *   - No C++ exception crosses this interface.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 16   /* query heads (after tensor-parallel split)         */
#define MLA_D_QK 576       /* kv_lora_rank 512 + qk_rope_head_dim 64            */
#define MLA_D_V 512        /* v_head_dim = kv_lora_rank                         */
#define MLA_MX_BLOCK 32    /* elements per e8m0 scale in the mxfp4 KV cache     */

/* Storage formats. kernelbot-amd-mixed-mla-675627, input tuple: kv_data holds
 * "bf16", "fp8" (per-tensor scale) and "mxfp4" (fp4x2 + fp8_e8m0 scale).      */
typedef enum {
  MLA_DTYPE_BF16 = 0,     /* bfloat16                                           */
  MLA_DTYPE_FP8_E4M3 = 1, /* OCP e4m3fn codes, value = code * per-tensor scale  */
  MLA_DTYPE_MXFP4 = 2     /* OCP MX: e2m1 nibbles (element 2i low, 2i+1 high),
                             one e8m0 scale 2^(e-127) per 32 elements           */
} mla_dtype_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer      */
  MLA_ERR_UNSUPPORTED = 2,  /* a dtype combination the library does not have  */
  MLA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required     */
  MLA_ERR_CUDA = 4,         /* a CUDA runtime call failed                     */
  MLA_ERR_TIMEOUT = 5,      /* device flag: a bounded wait in a kernel expired */
  MLA_ERR_DEVICE_CHECK = 6, /* device flag: indptr arrays failed the kernels'
                               bounds/monotonicity checks; work was skipped   */
  MLA_ERR_TOO_LARGE = 7     /* the call needs more scratch than the library's
                               fixed device array holds (see
                               mla_decode_static_workspace)                   */
} mla_status_t;

/* Device error flags, as returned by mla_get_device_error().                  */
#define MLA_DEVFLAG_TIMEOUT 0x1u  /* a bounded wait (~1 s) ran out. Besides a fault of
                                     the library, this can happen when a call that
                                     splits query tokens over two or more CTAs each
                                     (its CTAs then share the merges at their end and
                                     wait for one another) cannot place all of its
                                     CTAs on the GPU within that time, e.g. next to a
                                     long persistent kernel on another stream */
#define MLA_DEVFLAG_BAD_INDPTR 0x2u
#define MLA_DEVFLAG_BAD_PAGE 0x4u  /* mla_decode_paged: a page id >= num_pages */

typedef struct {
  int32_t batch;          /* number of segments = len(qo_indptr) - 1, >= 1         */
  int32_t total_q;        /* rows of q and out (= qo_indptr[batch]), >= 0          */
  int32_t total_kv;       /* rows of the KV cache (= kv_indptr[batch]), >= 0       */
  float sm_scale;         /* softmax scale; <= 0 selects 1/sqrt(576)               */
  mla_dtype_t q_dtype;    /* MLA_DTYPE_BF16, or MLA_DTYPE_FP8_E4M3 (a8w8)          */
  const float* q_scale;   /* device, one float: q = code * q_scale; NULL unless
                             q_dtype == MLA_DTYPE_FP8_E4M3                         */
  int32_t num_splits;     /* KV partitions (stage-1 CTAs); 0 = use mla_plan()      */
  void* workspace;        /* device scratch of mla_decode_workspace_size() bytes,
                             256-byte aligned, owned by the caller                 */
  size_t workspace_bytes;
  void* profile_events[3]; /* optional cudaEvent_t handles (NULL = none), recorded
                              on `stream` before and after the decode launch
                              (events 1 and 2 are recorded back to back: the
                              merge runs inside the launch)                      */
  int32_t quantize_q;     /* nonzero: quantise bf16 q to e4m3 inside the call and
                             run the a8w8 path, as the pages do before calling
                             their a8w8 kernel (kernelbot-amd-mixed-mla-753817,
                             `_quantize_fp8`): one per-tensor scale
                             s = max(amax|q|, 1e-12) / 448 and codes
                             RNE(q / s) saturated to +-448, all in fp32. Needs
                             q_dtype == MLA_DTYPE_BF16 and an fp8 KV cache
                             (else MLA_ERR_UNSUPPORTED); adds one small launch
                             (the amax). The scale is kept in the workspace
                             header.                                            */
  int32_t token_group;    /* query tokens of a segment that share one pass over
                             its KV rows (multi-token decode, q_len > 1; the
                             grouping of kernelbot-amd-mixed-mla-586148
                             `_flash_splitk`, whose Q block spans the q_len x
                             16 rows of a segment): 0 or 1 = one token per
                             pass; 2 = pairs (fp8 or bf16 KV; mxfp4:
                             MLA_ERR_UNSUPPORTED); 4 = groups of four (fp8 KV
                             with fp8 q or quantize_q; otherwise
                             MLA_ERR_UNSUPPORTED). The last group of a segment
                             holds the remaining tokens. Other values:
                             MLA_ERR_INVALID_ARG. Not with a page table. The
                             workspace must be sized by
                             mla_decode_group_workspace_size(). With pairs each
                             token's arithmetic is unchanged (with
                             num_splits = 1 the output equals that of the call
                             without grouping bit for bit); groups of four add
                             a weight's e4m3 remainder into the same
                             accumulator as its leading part (same tolerance,
                             different rounding).                            */
} mla_decode_opts;

/* Split planner (the pages choose the split count from batch size and KV
 * length: kernelbot-amd-mixed-mla-586148 "Adaptive split-K", -753817
 * `_choose_kv_splits`, -739756 `_get_config`). Here the KV rows of all
 * segments are divided evenly over the CTAs, so the planner picks only how
 * many partitions P <= sm_count to use (one CTA per SM). It minimises a cost
 * model of the slowest CTA: the tiles it streams, a fixed cost per token run
 * it holds (so P a multiple or a divisor of the token count, where no CTA
 * straddles a segment boundary, is preferred), and the merge of the splits
 * of a token. Segment lengths are taken as equal (total_kv / batch). Host
 * only; no device access. sm_count <= 0 queries the current device.
 * Writes the partition count to *num_splits. Errors: MLA_ERR_INVALID_ARG for
 * negative sizes or a NULL output.                                           */
mla_status_t mla_plan(int32_t batch, int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                      int32_t sm_count, int32_t* num_splits);

/* Bytes of device workspace that mla_decode() needs for these sizes and this
 * partition count (0 = what mla_plan() would choose on the current device).
 * The workspace holds a 256-byte header (the device error flags), one 32-bit
 * counter per query token (padded to 256 bytes) and the per-split partial
 * outputs: (num_splits + total_q) slots of 16x512 fp32 plus 16 fp32 LSE
 * values. It must be zero-filled before its first use; every call leaves the
 * counters at zero again, and mla_reset_device_error() restores them after an
 * error. Host only.                                                          */
mla_status_t mla_decode_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv,
                                       mla_dtype_t kv_dtype, int32_t num_splits, size_t* bytes);

/* The decode.
 *   q         device, [total_q][16][576] bf16, or e4m3 codes when
 *             opts->q_dtype == MLA_DTYPE_FP8_E4M3; 16-byte aligned
 *   kv        device, [total_kv][576] bf16 / e4m3 codes, or [total_kv][288]
 *             fp4x2 bytes for mxfp4; 16-byte aligned
 *   kv_scale  device: NULL (bf16), one float (fp8), or [total_kv][18] e8m0
 *             bytes (mxfp4; 16-byte aligned). mxfp4 rows are used as e2m1
 *             values rebased to the row's largest block scale R: every block
 *             whose scale is within 28 of R is used exactly; blocks further
 *             below count as zero (their elements are under 2^-28 of the
 *             row's largest block); a NaN scale code (0xFF) gives unspecified
 *             output values.
 *   qo_indptr, kv_indptr  device int32 [batch+1]: monotone, [0] = 0,
 *             qo_indptr[batch] = total_q, kv_indptr[batch] = total_kv. The
 *             kernels check this and, on a violation, skip the work and set
 *             MLA_DEVFLAG_BAD_INDPTR (no out-of-bounds access).
 *   out       device, [total_q][16][512] bf16 (round to nearest even)
 * Errors: MLA_ERR_INVALID_ARG (NULL/misaligned pointers, bad sizes),
 * MLA_ERR_UNSUPPORTED (dtype combination), MLA_ERR_WORKSPACE (too small),
 * MLA_ERR_CUDA (launch failed). Asynchronous on `stream`.                     */
mla_status_t mla_decode(const void* q, const void* kv, const void* kv_scale,
                        const int32_t* qo_indptr, const int32_t* kv_indptr, void* out,
                        mla_dtype_t kv_dtype, const mla_decode_opts* opts, void* stream);

/* Bytes of device workspace for a call with opts->token_group = G > 1: as
 * mla_decode_workspace_size(), with G * num_splits + total_q partial slots
 * (a piece of a group writes one partial per token). token_group 0 or 1 gives
 * the size of mla_decode_workspace_size(). Host only. Errors as
 * mla_decode_workspace_size(); MLA_ERR_INVALID_ARG for a token_group other
 * than 0, 1, 2 or 4.                                                         */
mla_status_t mla_decode_group_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv,
                                             mla_dtype_t kv_dtype, int32_t num_splits, int32_t token_group,
                                             size_t* bytes);

/* mla_decode_group_workspace_size() with token_group = 2.                    */
mla_status_t mla_decode_pairs_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv,
                                             mla_dtype_t kv_dtype, int32_t num_splits, size_t* bytes);

/* Paged KV cache: the page-table form of kernelbot-amd-mixed-mla-753817, which
 * hands `kv_indices`, `kv_last_page_len` and `page_size` (1 there) to the
 * vendor a8w8 decode. Segment b owns page-table entries
 * [page_indptr[b], page_indptr[b+1]); its KV row i is row i % page_size of
 * page page_indices[page_indptr[b] + i / page_size]. A segment with n_b > 0
 * pages has (n_b - 1) * page_size + last_page_len[b] rows; with
 * page_size == 1 it has n_b rows and last_page_len is not read (the pages pass
 * the segment lengths there, which only that reading accepts). All arrays are
 * device int32 and caller-owned.                                              */
typedef struct {
  const int32_t* page_indptr;   /* [batch+1], monotone, page_indptr[0] = 0       */
  const int32_t* page_indices;  /* [page_indptr[batch]] page ids in [0, num_pages) */
  const int32_t* last_page_len; /* [batch], each in [1, page_size]; may be NULL
                                   when page_size == 1                           */
  int32_t page_size;            /* KV rows per page, >= 1                        */
  int32_t num_pages;            /* pages in the pool kv_pages points to;
                                   num_pages * page_size < 2^31                  */
} mla_paged_kv;

/* Workspace bytes for mla_decode_paged(): mla_decode_workspace_size() plus
 * room for the logical row offsets of the segments (batch+1 int32, padded to
 * 256 bytes). total_kv is the logical row count (the sum of the segment
 * lengths). Host only. Errors as mla_decode_workspace_size().                 */
mla_status_t mla_decode_paged_workspace_size(int32_t batch, int32_t total_q, int32_t total_kv,
                                             mla_dtype_t kv_dtype, int32_t num_splits, size_t* bytes);

/* The decode over a paged KV cache (fp8 e4m3 only; other KV dtypes return
 * MLA_ERR_UNSUPPORTED). Arguments as mla_decode(), except:
 *   kv_pages  device, [num_pages][page_size][576] e4m3 codes, 16-byte aligned
 *   paged     the page table (above), host struct of device pointers
 *   opts->total_kv  the logical KV row count, sum of the segment lengths
 * One extra small launch builds the logical row offsets from the page table
 * into the workspace. If page_indptr is not monotone from 0, a last-page
 * length is outside [1, page_size], or the lengths do not sum to
 * opts->total_kv, no KV row is read and MLA_DEVFLAG_BAD_INDPTR is set. A page
 * id outside [0, num_pages) sets MLA_DEVFLAG_BAD_PAGE; that row is not read
 * and the output of its token is unspecified. Results are bitwise those of
 * mla_decode() on the same rows laid out contiguously with the same
 * num_splits. Errors as mla_decode(). Asynchronous on `stream`.              */
mla_status_t mla_decode_paged(const void* q, const void* kv_pages, const void* kv_scale,
                              const int32_t* qo_indptr, const mla_paged_kv* paged, void* out,
                              mla_dtype_t kv_dtype, const mla_decode_opts* opts, void* stream);

/* Device buffers (caller-owned) that mla_decode_from_host() stages into.      */
typedef struct {
  void* q;             /* bytes of q                                        */
  void* kv;            /* bytes of the KV cache                             */
  void* kv_scale;      /* fp8: 4 bytes; mxfp4: total_kv*18 bytes; else NULL  */
  float* q_scale;      /* 4 bytes when q is fp8, else NULL                  */
  int32_t* qo_indptr;  /* batch+1 ints                                      */
  int32_t* kv_indptr;  /* batch+1 ints                                      */
  void* out;           /* total_q*16*512 bf16                               */
} mla_device_buffers;

/* The same decode from HOST buffers: enqueues one cudaMemcpyAsync per input
 * (host -> the caller's device buffers), mla_decode(), and the copy of the
 * output back to h_out. Host buffers should be pinned for the copies to be
 * asynchronous. The call returns once everything is enqueued; synchronise
 * `stream` before reading h_out. h_q_scale is a host float (fp8 q) or NULL;
 * opts->q_scale is ignored (dev->q_scale is used).                            */
mla_status_t mla_decode_from_host(const void* h_q, const void* h_kv, const void* h_kv_scale,
                                  const float* h_q_scale, const int32_t* h_qo_indptr,
                                  const int32_t* h_kv_indptr, void* h_out, mla_dtype_t kv_dtype,
                                  const mla_decode_opts* opts, const mla_device_buffers* dev,
                                  void* stream);

/* Dequantisation through the decode kernels' own operand path: KV rows
 * [row0, row0+nrows) are loaded and converted exactly as stage 1 does and
 * written as fp32 to d_out [nrows][576] (device, 4-byte aligned).
 *  - bf16, fp8: the rows are pushed through the same tensor-core instruction
 *    against an identity operand; kv_scale is not read (fp8: value = code,
 *    the per-tensor scale is the caller's).
 *  - mxfp4: kv_scale = the e8m0 block scales [total_kv][18] (required). The
 *    rows go through stage 1's conversion to rebased e5m2 operand bytes and
 *    the row exponent R; value = byte * 2^(R - 140). Blocks more than 28
 *    binades below the row's largest block are 0, as in the decode; a NaN
 *    scale (0xFF) is outside the domain.
 * The result equals the format's definition bit for bit wherever that value
 * is representable in fp32 (and, for mxfp4, the block is not flushed).
 * Asynchronous. Errors: MLA_ERR_INVALID_ARG.                                  */
mla_status_t mla_dequant_rows(const void* kv, const void* kv_scale, mla_dtype_t kv_dtype,
                              int32_t total_kv, int32_t row0, int32_t nrows, float* d_out,
                              void* stream);

/* Host-side input check, for callers that do not trust their indptr arrays
 * (the pages' interface trusts them: kernelbot-amd-mixed-mla-675627, module
 * docstring, where qo_indptr and kv_indptr are built by the harness). Copies
 * qo_indptr and kv_indptr (device, int32 [batch+1]) to the host and checks
 * what mla_decode() assumes: [0] = 0, monotone non-decreasing,
 * qo_indptr[batch] = total_q and kv_indptr[batch] = total_kv. For an mxfp4
 * cache it also scans kv_scale (device, [total_kv][18] e8m0) for the NaN
 * code 0xFF. Synchronises `stream`; allocates host memory only.
 * Returns MLA_OK, or MLA_ERR_DEVICE_CHECK with *bad_index (may be NULL) set to
 * the first offending element: i for qo_indptr[i], batch + 1 + i for
 * kv_indptr[i], 2 (batch + 1) + j for byte j of kv_scale. MLA_ERR_INVALID_ARG
 * for NULL arrays or negative sizes, MLA_ERR_CUDA if a copy fails.          */
mla_status_t mla_validate_inputs(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                                 int32_t total_q, int32_t total_kv, mla_dtype_t kv_dtype,
                                 const void* kv_scale, void* stream, int64_t* bad_index);

/* Reads the device error flags that kernels set in `workspace` (OR of
 * MLA_DEVFLAG_*). Synchronises `stream`. Returns MLA_OK, MLA_ERR_TIMEOUT or
 * MLA_ERR_DEVICE_CHECK (timeout wins); *flags may be NULL.                    */
mla_status_t mla_get_device_error(const void* workspace, void* stream, uint32_t* flags);

/* Clears the device error flags (flags are sticky until cleared) and the token
 * counters that a call stopped by an error may have left non-zero.
 * Synchronises `stream` (it reads how many counters the last call used).      */
mla_status_t mla_reset_device_error(void* workspace, void* stream);

/* Milliseconds between two CUDA events (cudaEvent_t passed as void*) that
 * have completed, e.g. the profile_events of mla_decode_opts. Synchronises
 * on ev_end. Errors: MLA_ERR_INVALID_ARG (NULL), MLA_ERR_CUDA.                */
mla_status_t mla_event_elapsed_ms(void* ev_start, void* ev_end, float* ms);

/* The decode for callers that cannot allocate device memory. Not part of the
 * method on the pages (they have no counterpart): it exists for callers that
 * must not call cudaMalloc at decode time -- code that runs while a CUDA
 * stream is being captured into a graph, or engines that reserve all device
 * memory up front and forbid allocations afterwards -- and so cannot provide
 * the workspace that mla_decode() needs.
 *
 * Same arguments and results as mla_decode(); opts->workspace and
 * opts->workspace_bytes are ignored. The scratch (device error flags and
 * per-split partials) is a fixed MLA_STATIC_WORKSPACE_BYTES array inside the
 * library, reserved on every GPU that loads the library until the process
 * exits. This call allocates nothing: no cudaMalloc/cudaFree and no
 * allocating library routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture.
 *   - Calls whose scratch need (mla_decode_workspace_size()) exceeds
 *     MLA_STATIC_WORKSPACE_BYTES return MLA_ERR_TOO_LARGE and launch nothing.
 *   - Every call shares the one array and clears its error flags at the start;
 *     two calls that overlap on the GPU (different streams, no ordering) race
 *     on it and produce undefined results. Calls on one stream are ordered.
 *   - Argument errors are returned as for mla_decode(); the device error
 *     flags (bounded-wait timeouts, indptr checks) are read with
 *     mla_static_workspace_device_error().                                   */
#define MLA_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)
mla_status_t mla_decode_static_workspace(const void* q, const void* kv, const void* kv_scale,
                                         const int32_t* qo_indptr, const int32_t* kv_indptr,
                                         void* out, mla_dtype_t kv_dtype,
                                         const mla_decode_opts* opts, void* stream);

/* The device error flags of mla_decode_static_workspace() on the current
 * device (the flags live in the library's fixed array, which the caller cannot
 * address): MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_CHECK as
 * mla_get_device_error(), and the OR of MLA_DEVFLAG_* in *flags (may be NULL).
 * Flags are those of the last call on this device (each call clears them when
 * it starts). Synchronises `stream`; allocates nothing.                      */
mla_status_t mla_static_workspace_device_error(void* stream, uint32_t* flags);

/* Static description of a status code.                                        */
const char* mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
