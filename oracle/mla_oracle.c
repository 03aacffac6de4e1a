/*
 * TEST INFRASTRUCTURE ONLY -- the oracle for MLA decode attention.
 *
 * A plain, slow, single-threaded fp64 CPU implementation of what the GPU path
 * computes. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may call it; the product path never does. It shares no code with the CUDA
 * library (no headers, helpers or tables).
 *
 * What it computes (kernelbot-amd-mixed-mla-675627, "MLA decode kernel --
 * submission template": the module docstring's problem statement and the naive
 * bf16 reference `custom_kernel_bf16`):
 *
 *   For each batch entry b, each query token t in [qo_indptr[b], qo_indptr[b+1])
 *   and each head h:
 *     Q      = dequant(q[t, h, 0:D])                         (D = 576)
 *     K_j    = dequant(kv[j, 0:D]),  V_j = K_j[0:DV]          (DV = 512)
 *              for j in [kv_indptr[b], kv_indptr[b+1])
 *     s_j    = sm_scale * sum_d Q_d K_{j,d}                  (sm_scale = 1/sqrt(576))
 *     out    = sum_j exp(s_j - M) V_j / sum_j exp(s_j - M),  M = max_j s_j
 *     lse    = M + log(sum_j exp(s_j - M))                    (natural log)
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *   - every query token of a segment attends to all of that segment's KV rows
 *     (no causal mask), as the naive reference does for q_len > 1;
 *   - a segment with no KV rows gives out = 0 and lse = -inf;
 *   - fp8 is OCP e4m3fn (bias 7, no infinities, S.1111.111 is NaN), dequantised
 *     as code * per-tensor scale;
 *   - mxfp4 is OCP MX: fp4x2 bytes hold element 2i in the low nibble and 2i+1
 *     in the high nibble; e2m1 has bias 1; one e8m0 scale (2^(e-127), 0xFF =
 *     NaN) per 32 consecutive elements of a row, stored [rows][D/32] bytes.
 *
 * Parity pins live in tests/test_oracle_*.py: format decoders against the
 * torch CPU float8 dtypes, attention against brute force in 50-digit
 * arithmetic, a torch float64 cross-check of the naive reference formula, and
 * invariants (single row, identical keys, permutation, split + LSE merge).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_MXFP4 = 2 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_NOMEM = 2 };

/* ---- number formats -------------------------------------------------------
 * A minifloat with `ebits` exponent bits, `mbits` mantissa bits and exponent
 * bias `bias`, sign in the bit above the exponent. Exponent field 0 encodes
 * subnormals (m / 2^mbits) * 2^(1 - bias). No infinity/NaN handling here: the
 * callers below add each format's special codes.                              */
double orc_decode_minifloat(uint32_t bits, int ebits, int mbits, int bias) {
  uint32_t mant = bits & ((1u << mbits) - 1u);
  uint32_t expo = (bits >> mbits) & ((1u << ebits) - 1u);
  uint32_t sign = (bits >> (mbits + ebits)) & 1u;
  double frac = (double)mant / (double)(1u << mbits);
  double mag;
  if (expo == 0)
    mag = ldexp(frac, 1 - bias);
  else
    mag = ldexp(1.0 + frac, (int)expo - bias);
  return sign ? -mag : mag;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
double orc_decode_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn"): 4 exponent bits, 3 mantissa bits, bias 7, the two
 * codes with all exponent and mantissa bits set are NaN, no infinities. */
double orc_decode_e4m3fn(uint8_t code) {
  if ((code & 0x7F) == 0x7F) return NAN;
  return orc_decode_minifloat(code, 4, 3, 7);
}

/* OCP FP4 E2M1: 2 exponent bits, 1 mantissa bit, bias 1, no special codes. */
double orc_decode_e2m1(uint8_t nibble) { return orc_decode_minifloat(nibble & 0xF, 2, 1, 1); }

/* OCP E8M0 scale: 2^(e - 127); 0xFF is NaN. */
double orc_decode_e8m0(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* Vectorised decode for tests: kind 0 = bf16 (uint16 input), 1 = e4m3fn,
 * 2 = e2m1 (one nibble per input byte), 3 = e8m0, 4 = generic minifloat with
 * (ebits, mbits, bias) taken from `params`. */
int orc_decode_array(int kind, int64_t n, const void* src, double* dst, const int32_t* params) {
  if (n < 0 || (n > 0 && (!src || !dst))) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) {
    switch (kind) {
      case 0: dst[i] = orc_decode_bf16(((const uint16_t*)src)[i]); break;
      case 1: dst[i] = orc_decode_e4m3fn(((const uint8_t*)src)[i]); break;
      case 2: dst[i] = orc_decode_e2m1(((const uint8_t*)src)[i]); break;
      case 3: dst[i] = orc_decode_e8m0(((const uint8_t*)src)[i]); break;
      case 4:
        if (!params) return ORC_ERR_ARG;
        dst[i] = orc_decode_minifloat(((const uint32_t*)src)[i], params[0], params[1], params[2]);
        break;
      default: return ORC_ERR_ARG;
    }
  }
  return ORC_OK;
}

/* ---- dequantisation of one row ------------------------------------------ */

/* Row j of the KV cache, all D elements, as doubles.
 *   bf16 : kv is uint16[total_kv][D]
 *   fp8  : kv is uint8[total_kv][D], kv_scale -> one float (per tensor)
 *   mxfp4: kv is uint8[total_kv][D/2] (element 2i low nibble, 2i+1 high),
 *          kv_scale is uint8[total_kv][D/32] e8m0 codes                        */
static void decode_kv_row(const void* kv, const void* kv_scale, int kv_dtype, int64_t j, int D,
                          double* dst) {
  if (kv_dtype == ORC_BF16) {
    const uint16_t* row = (const uint16_t*)kv + j * (int64_t)D;
    for (int d = 0; d < D; ++d) dst[d] = orc_decode_bf16(row[d]);
  } else if (kv_dtype == ORC_FP8_E4M3) {
    const uint8_t* row = (const uint8_t*)kv + j * (int64_t)D;
    double scale = (double)(*(const float*)kv_scale);
    for (int d = 0; d < D; ++d) dst[d] = orc_decode_e4m3fn(row[d]) * scale;
  } else {
    const uint8_t* row = (const uint8_t*)kv + j * (int64_t)(D / 2);
    const uint8_t* srow = (const uint8_t*)kv_scale + j * (int64_t)(D / 32);
    for (int d = 0; d < D; ++d) {
      uint8_t byte = row[d / 2];
      uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      dst[d] = orc_decode_e2m1(nib) * orc_decode_e8m0(srow[d / 32]);
    }
  }
}

/* Query row (token t, head h): bf16 as is, or fp8 e4m3fn code * q_scale. */
static void decode_q_row(const void* q, int q_dtype, const float* q_scale, int64_t t, int h, int H,
                         int D, double* dst) {
  int64_t base = (t * H + h) * (int64_t)D;
  if (q_dtype == ORC_BF16) {
    for (int d = 0; d < D; ++d) dst[d] = orc_decode_bf16(((const uint16_t*)q)[base + d]);
  } else {
    double s = (double)(*q_scale);
    for (int d = 0; d < D; ++d) dst[d] = orc_decode_e4m3fn(((const uint8_t*)q)[base + d]) * s;
  }
}

/* ---- attention for one query row ----------------------------------------
 * Q[D] against the n decoded rows K[n][D] (V = first DV columns of each row).
 * scores[] is caller scratch of length n. Writes out[DV] and *lse.            */
static void attend_one(const double* Q, const double* K, int64_t n, int D, int DV, double sm_scale,
                       double* scores, double* out, double* lse) {
  for (int d = 0; d < DV; ++d) out[d] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double M = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    const double* k = K + j * (int64_t)D;
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += Q[d] * k[d];
    s *= sm_scale;
    scores[j] = s;
    if (s > M) M = s;
  }
  double denom = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double w = exp(scores[j] - M);
    const double* v = K + j * (int64_t)D;
    for (int d = 0; d < DV; ++d) out[d] += w * v[d];
    denom += w;
  }
  for (int d = 0; d < DV; ++d) out[d] /= denom;
  *lse = M + log(denom);
}

static int check_indptr(const int32_t* qo, const int32_t* kvp, int batch, int64_t total_q,
                        int64_t total_kv) {
  if (batch < 0 || !qo || !kvp) return 0;
  if (qo[0] != 0 || kvp[0] != 0) return 0;
  for (int b = 0; b < batch; ++b) {
    if (qo[b + 1] < qo[b] || kvp[b + 1] < kvp[b]) return 0;
  }
  if (qo[batch] != total_q || kvp[batch] != total_kv) return 0;
  return 1;
}

/* Segmented attention over already-decoded fp64 arrays.
 *   q   [total_q][H][D], kv [total_kv][D] (V = kv[:, :DV])
 *   out [total_q][H][DV], lse [total_q][H] (may be NULL)                      */
int orc_attention_f64(const double* q, const double* kv, const int32_t* qo_indptr,
                      const int32_t* kv_indptr, int batch, int64_t total_q, int64_t total_kv, int H,
                      int D, int DV, double sm_scale, double* out, double* lse) {
  if (H <= 0 || D <= 0 || DV <= 0 || DV > D || !out) return ORC_ERR_ARG;
  if (!check_indptr(qo_indptr, kv_indptr, batch, total_q, total_kv)) return ORC_ERR_ARG;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t len = kv_indptr[b + 1] - kv_indptr[b];
    if (len > max_len) max_len = len;
  }
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  if (!scores) return ORC_ERR_NOMEM;
  for (int b = 0; b < batch; ++b) {
    const double* K = kv + (int64_t)kv_indptr[b] * D;
    int64_t n = kv_indptr[b + 1] - kv_indptr[b];
    for (int64_t t = qo_indptr[b]; t < qo_indptr[b + 1]; ++t) {
      for (int h = 0; h < H; ++h) {
        double l;
        attend_one(q + (t * H + h) * (int64_t)D, K, n, D, DV, sm_scale, scores,
                   out + (t * H + h) * (int64_t)DV, &l);
        if (lse) lse[t * H + h] = l;
      }
    }
  }
  free(scores);
  return ORC_OK;
}

/* The full path from raw encodings, for the (token, head) pairs listed in
 * rows_t/rows_h (n_rows of them); out is [n_rows][DV], lse [n_rows] or NULL.
 * Pass n_rows = -1 to compute every (token, head) in order, with out laid out
 * [total_q][H][DV]. Each segment's KV rows are decoded once into scratch.     */
int orc_mla_decode(const void* q, int q_dtype, const float* q_scale, const void* kv, int kv_dtype,
                   const void* kv_scale, const int32_t* qo_indptr, const int32_t* kv_indptr,
                   int batch, int64_t total_q, int64_t total_kv, int H, int D, int DV,
                   double sm_scale, int64_t n_rows, const int32_t* rows_t, const int32_t* rows_h,
                   double* out, double* lse) {
  if (!q || !kv || !out || H <= 0 || D <= 0 || DV <= 0 || DV > D) return ORC_ERR_ARG;
  if (q_dtype != ORC_BF16 && q_dtype != ORC_FP8_E4M3) return ORC_ERR_ARG;
  if (q_dtype == ORC_FP8_E4M3 && !q_scale) return ORC_ERR_ARG;
  if (kv_dtype != ORC_BF16 && kv_dtype != ORC_FP8_E4M3 && kv_dtype != ORC_MXFP4) return ORC_ERR_ARG;
  if (kv_dtype != ORC_BF16 && !kv_scale) return ORC_ERR_ARG;
  if (kv_dtype == ORC_MXFP4 && (D % 32) != 0) return ORC_ERR_ARG;
  if (!check_indptr(qo_indptr, kv_indptr, batch, total_q, total_kv)) return ORC_ERR_ARG;
  if (n_rows >= 0 && n_rows > 0 && (!rows_t || !rows_h)) return ORC_ERR_ARG;

  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t len = kv_indptr[b + 1] - kv_indptr[b];
    if (len > max_len) max_len = len;
  }
  size_t kbytes = sizeof(double) * (size_t)(max_len > 0 ? max_len : 1) * (size_t)D;
  double* K = (double*)malloc(kbytes);
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  double* Q = (double*)malloc(sizeof(double) * (size_t)D);
  if (!K || !scores || !Q) {
    free(K); free(scores); free(Q);
    return ORC_ERR_NOMEM;
  }
  int rc = ORC_OK;
  for (int b = 0; b < batch; ++b) {
    int64_t t0 = qo_indptr[b], t1 = qo_indptr[b + 1];
    if (t1 == t0) continue;
    /* Is any requested row in this segment? */
    int wanted = (n_rows < 0);
    for (int64_t r = 0; !wanted && r < n_rows; ++r)
      if (rows_t[r] >= t0 && rows_t[r] < t1) wanted = 1;
    if (!wanted) continue;
    int64_t n = kv_indptr[b + 1] - kv_indptr[b];
    for (int64_t j = 0; j < n; ++j)
      decode_kv_row(kv, kv_scale, kv_dtype, kv_indptr[b] + j, D, K + j * (int64_t)D);
    if (n_rows < 0) {
      for (int64_t t = t0; t < t1; ++t)
        for (int h = 0; h < H; ++h) {
          double l;
          decode_q_row(q, q_dtype, q_scale, t, h, H, D, Q);
          attend_one(Q, K, n, D, DV, sm_scale, scores, out + (t * H + h) * (int64_t)DV, &l);
          if (lse) lse[t * H + h] = l;
        }
    } else {
      for (int64_t r = 0; r < n_rows; ++r) {
        if (rows_t[r] < t0 || rows_t[r] >= t1) continue;
        if (rows_h[r] < 0 || rows_h[r] >= H) { rc = ORC_ERR_ARG; continue; }
        double l;
        decode_q_row(q, q_dtype, q_scale, rows_t[r], rows_h[r], H, D, Q);
        attend_one(Q, K, n, D, DV, sm_scale, scores, out + r * (int64_t)DV, &l);
        if (lse) lse[r] = l;
      }
    }
  }
  free(K); free(scores); free(Q);
  return rc;
}

/* Merge of per-split results of one query row (split-K flash decoding, the
 * stage-2 reductions of kernelbot-amd-mixed-mla-586148 `_reduce_splitk` and
 * kernelbot-amd-mixed-mla-753817 `mla_flash_decode_stage2`):
 *   o[s][DV] is split s's normalised output, lse[s] its natural-log LSE.
 *   out = sum_s exp(lse_s - L) o_s / sum_s exp(lse_s - L), L = max_s lse_s.
 * Splits with lse = -inf carry weight 0; if every split is empty, out = 0.    */
void orc_lse_combine(int nsplit, int DV, const double* o, const double* lse, double* out,
                     double* lse_out) {
  double L = -INFINITY;
  for (int s = 0; s < nsplit; ++s)
    if (lse[s] > L) L = lse[s];
  for (int d = 0; d < DV; ++d) out[d] = 0.0;
  if (L == -INFINITY) {
    if (lse_out) *lse_out = -INFINITY;
    return;
  }
  double wsum = 0.0;
  for (int s = 0; s < nsplit; ++s) {
    double w = exp(lse[s] - L);
    for (int d = 0; d < DV; ++d) out[d] += w * o[(int64_t)s * DV + d];
    wsum += w;
  }
  for (int d = 0; d < DV; ++d) out[d] /= wsum;
  if (lse_out) *lse_out = L + log(wsum);
}
