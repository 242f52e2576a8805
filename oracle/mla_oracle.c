/*
 * CPU oracle for MLA paged decode in absorbed form.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load or call this file; the CUDA library never does, and the two share no
 * code, headers or constants.
 *
 * What it computes (PaddleNLP issue #10157, "Multi-head Latent Attention (MLA)
 * 算子 / 总体概述": one MLA step is Data Load -> QK GEMM -> Softmax Update ->
 * PV GEMM, with num_token > 1 supported in the decoder; page 2 of the same
 * material, section 2.4.3, runs it with --mla_use_matrix_absorption 1, i.e. on
 * the compressed latent).  The pages name the steps but do not write the math;
 * the plain reading used here is, for every request b, new token i < s_q and
 * head h:
 *
 *   n      = seqlen[b] - s_q + i + 1          visible keys, causal within the
 *                                             s_q new tokens (the verify step
 *                                             of "MTP 高效推理", same page)
 *   k_t    = KV[block_table[b][t/64]][t%64]   576 channels (512 latent + 64 RoPE)
 *   s_t    = scale * sum_c q[b,i,h,c] k_t[c]  fp64
 *   m      = max_t s_t,  Z = sum_t exp(s_t - m)
 *   lse    = m + ln Z                         natural log, scale included
 *   out[c] = sum_t exp(s_t - m) / Z * k_t[c]  c < 512 (V is the latent part)
 *
 * n <= 0 gives out = 0 and lse = -inf.  For the fp8 cache, k_t[c] is the e4m3
 * value times the fp32 scale of its token and channel group (groups of 128
 * channels, the last one 64 wide).  For fp8 variant B each token is one
 * 656-byte record: latent channel c < 512 is its e4m3 code times the record's
 * fp32 scale c/128, and the RoPE channels are bf16 values stored in the record.
 *
 * Every value is computed in double from the exact input values, as plain
 * loops, parallel over query rows with OpenMP.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_PAGE 64
#define ORC_DQK 576
#define ORC_DV 512
#define ORC_NGROUP 5

enum { ORC_KV_BF16 = 0, ORC_KV_FP8 = 1, ORC_KV_F64 = 2, ORC_KV_FP8B = 3 };
/* fp8 variant B token record: e4m3 latent [0,512), 4 fp32 scales [512,528), RoPE bf16 [528,656) */
enum { ORC_FP8B_RECORD = 656 };
enum { ORC_OK = 0, ORC_BAD_ARG = -1, ORC_BAD_PAGE = -2, ORC_NOMEM = -3 };

/* bf16 -> double: a bf16 is the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* e4m3 (OCP FP8 E4M3FN) -> double, from the format definition: 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
 * (value = mantissa/8 * 2^-6); no infinities; S.1111.111 is NaN. */
double oracle_e4m3_to_f64(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Channel group of the fp8 scale for channel c: [0,128) [128,256) [256,384)
 * [384,512) [512,576). */
static int fp8_group(int c) { return c < 512 ? c / 128 : 4; }

typedef struct {
  const void* q;          /* bf16 [B, s_q, H, 576] or f64 when kv_dtype == F64 */
  const void* kv;         /* [P, 64, 576] bf16 / e4m3 / f64 */
  const float* scales;    /* [P, 64, 5] for fp8 */
  int kv_dtype;
  const int32_t* block_table;
  const int32_t* seqlens;
  int B, s_q, H, num_pages, max_pages;
  double scale;
} orc_args;

static double q_at(const orc_args* a, int64_t row, int c) {
  if (a->kv_dtype == ORC_KV_F64) return ((const double*)a->q)[row * ORC_DQK + c];
  return oracle_bf16_to_f64(((const uint16_t*)a->q)[row * ORC_DQK + c]);
}

/* Data Load step: fetch key/value row t of request b through the block table
 * into k[576] as doubles.  Returns 0, or ORC_BAD_PAGE for an id outside the pool. */
static int fetch_key(const orc_args* a, int b, int t, double* k) {
  int page = a->block_table[(int64_t)b * a->max_pages + t / ORC_PAGE];
  int slot = t % ORC_PAGE;
  if (page < 0 || page >= a->num_pages) return ORC_BAD_PAGE;
  int64_t base = ((int64_t)page * ORC_PAGE + slot) * ORC_DQK;
  if (a->kv_dtype == ORC_KV_BF16) {
    const uint16_t* kv = (const uint16_t*)a->kv;
    for (int c = 0; c < ORC_DQK; ++c) k[c] = oracle_bf16_to_f64(kv[base + c]);
  } else if (a->kv_dtype == ORC_KV_FP8) {
    const uint8_t* kv = (const uint8_t*)a->kv;
    const float* sc = a->scales + ((int64_t)page * ORC_PAGE + slot) * ORC_NGROUP;
    for (int c = 0; c < ORC_DQK; ++c) k[c] = oracle_e4m3_to_f64(kv[base + c]) * (double)sc[fp8_group(c)];
  } else if (a->kv_dtype == ORC_KV_FP8B) {
    const uint8_t* rec = (const uint8_t*)a->kv + ((int64_t)page * ORC_PAGE + slot) * ORC_FP8B_RECORD;
    float sc[4];
    memcpy(sc, rec + 512, sizeof(sc));
    for (int c = 0; c < 512; ++c) k[c] = oracle_e4m3_to_f64(rec[c]) * (double)sc[c / 128];
    for (int c = 512; c < ORC_DQK; ++c) {
      uint16_t v;
      memcpy(&v, rec + 528 + 2 * (c - 512), sizeof(v));
      k[c] = oracle_bf16_to_f64(v);
    }
  } else {
    const double* kv = (const double*)a->kv;
    for (int c = 0; c < ORC_DQK; ++c) k[c] = kv[base + c];
  }
  return ORC_OK;
}

/* One query row (flat id = b*s_q*H + i*H + h): QK scores, softmax, PV.
 * p_out (optional, length >= n) receives the softmax weights. */
static int one_row(const orc_args* a, int64_t row, double* out, double* lse, double* p_out, double* s_buf,
                   double* k) {
  const int64_t R = (int64_t)a->s_q * a->H;
  const int b = (int)(row / R);
  const int i = (int)((row % R) / a->H);
  const int64_t n64 = (int64_t)a->seqlens[b] - a->s_q + i + 1;
  int n = n64 > 0 ? (int)n64 : 0;
  for (int c = 0; c < ORC_DV; ++c) out[c] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return ORC_OK;
  }
  if ((int64_t)(n - 1) / ORC_PAGE >= a->max_pages) return ORC_BAD_ARG;
  double qv[ORC_DQK];
  for (int c = 0; c < ORC_DQK; ++c) qv[c] = q_at(a, row, c);
  /* QK GEMM: s_t = scale * <q, k_t> */
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    int rc = fetch_key(a, b, t, k);
    if (rc) return rc;
    double dot = 0.0;
    for (int c = 0; c < ORC_DQK; ++c) dot += qv[c] * k[c];
    s_buf[t] = a->scale * dot;
    if (s_buf[t] > m) m = s_buf[t];
  }
  /* Softmax: Z = sum exp(s - m), lse = m + ln Z */
  double Z = 0.0;
  for (int t = 0; t < n; ++t) Z += exp(s_buf[t] - m);
  *lse = m + log(Z);
  /* PV GEMM: out = sum_t p_t * v_t over the 512 latent channels */
  for (int t = 0; t < n; ++t) {
    double p = exp(s_buf[t] - m) / Z;
    if (p_out) p_out[t] = p;
    int rc = fetch_key(a, b, t, k);
    if (rc) return rc;
    for (int c = 0; c < ORC_DV; ++c) out[c] += p * k[c];
  }
  return ORC_OK;
}

/*
 * Compute out [n_rows, 512] and lse [n_rows] (doubles) for the listed flat row
 * ids (row_ids == NULL: every row, in order).  p_debug, when non-NULL, is an
 * [n_rows, p_stride] array that receives the softmax weights of each row.
 * Returns 0 or a negative error (bad argument, page id outside the pool).
 */
int oracle_mla_decode(const void* q, const void* kv, const float* kv_scales, int kv_dtype,
                      const int32_t* block_table, const int32_t* seqlens, int B, int s_q, int H,
                      int num_pages, int max_pages, double softmax_scale, const int64_t* row_ids,
                      int64_t n_rows, double* out, double* lse, double* p_debug, int64_t p_stride) {
  if (!q || !kv || !block_table || !seqlens || !out || !lse) return ORC_BAD_ARG;
  if (B < 1 || s_q < 1 || H < 1 || num_pages < 1 || max_pages < 1) return ORC_BAD_ARG;
  if (kv_dtype == ORC_KV_FP8 && !kv_scales) return ORC_BAD_ARG;
  if (kv_dtype < 0 || kv_dtype > 3) return ORC_BAD_ARG;
  orc_args a = {q, kv, kv_scales, kv_dtype, block_table, seqlens, B, s_q, H, num_pages, max_pages,
                softmax_scale};
  const int64_t total = (int64_t)B * s_q * H;
  if (!row_ids) n_rows = total;
  int64_t max_n = 0;
  for (int b = 0; b < B; ++b)
    if (seqlens[b] > max_n) max_n = seqlens[b];
  if (max_n < 1) max_n = 1;
  int status = ORC_OK;
#pragma omp parallel
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)max_n);
    double* k = (double*)malloc(sizeof(double) * ORC_DQK);
    if (!s_buf || !k) {
#pragma omp critical
      status = ORC_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t r = 0; r < n_rows; ++r) {
        int64_t row = row_ids ? row_ids[r] : r;
        int rc;
        if (row < 0 || row >= total)
          rc = ORC_BAD_ARG;
        else
          rc = one_row(&a, row, out + r * ORC_DV, lse + r, p_debug ? p_debug + r * p_stride : NULL, s_buf, k);
        if (rc) {
#pragma omp critical
          status = rc;
        }
      }
    }
    free(s_buf);
    free(k);
  }
  return status;
}

/* Thread count used by the next oracle_mla_decode calls (n >= 1); a timing
 * knob only, the arithmetic is the same for any count. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
