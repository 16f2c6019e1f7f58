/*
 * Paged-KV attention oracle: plain fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library, and it never reads a value
 * the CUDA library produced.
 *
 * What it computes (the plain definition, no tiling, no splitting):
 *
 *   For every sequence row b of a packed (varlen) batch, every new query token
 *   i of that row (0 <= i < q_b, q_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]) and
 *   every query head h, with the KV head kh = h / (Hq / Hkv):
 *
 *     last = L_b - q_b + i         (bottom-right causal alignment: the new
 *                                   tokens are the last q_b keys of the row)
 *     if L_b == 0 or last < 0:  out = 0
 *     key j (0 <= j <= last) lives at page block_table[b][j / P], slot j % P
 *     x_j = s * sum_c q[c] * k_j[c]          (k_j already times k_scale)
 *     m   = max_j x_j,   w_j = exp(x_j - m)
 *     out = (sum_j w_j * v_j) / (sum_j w_j)  (v_j already times v_scale)
 *
 * Sources (vllm-rlt PR #128, "Purpose", prefill bullet list): the packed
 * interface with cu_seqlens_q, one block table per sequence and bottom-right
 * causal alignment; K/V gathered through the block table; GQA.  Same page,
 * "Test Plan" item 3: empty rows give a zero output.  1Cat-vLLM PR #616
 * (original description, "Test Plan"/"Test Result"): fp8_e5m2 KV cache, page
 * sizes that are multiples of 16, a dense exact reference.
 *
 * Number formats are decoded exactly into double from their definitions:
 *   binary16  : 1 sign, 5 exponent bits (bias 15), 10 fraction bits
 *   bfloat16  : the upper half of an IEEE binary32
 *   fp8 E5M2  : 1 sign, 5 exponent bits (bias 15), 2 fraction bits, with
 *               subnormals; exponent 31 encodes inf/NaN
 * All arithmetic is IEEE double; exp() is the C library's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E5M2 = 3 };

typedef struct {
  int32_t num_rows;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t max_pages_per_row;
  int32_t q_dtype;
  int32_t kv_dtype;
  double softmax_scale;
  double k_scale;
  double v_scale;
} oracle_problem;

/* binary16 -> double, from the field layout. */
static double dec_f16(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)f, -24);                 /* 2^-14 * f/2^10 */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(1024.0 + (double)f, e - 25);             /* 2^(e-15)*(1+f/2^10) */
  return s ? -v : v;
}

/* bfloat16 -> double: the 16 bits are the top half of a binary32. */
static double dec_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp8 E5M2 -> double, from the field layout. */
static double dec_e5m2(uint8_t x) {
  int s = (x >> 7) & 1, e = (x >> 2) & 31, f = x & 3;
  double v;
  if (e == 0) v = ldexp((double)f, -16);                  /* 2^-14 * f/4 */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(4.0 + (double)f, e - 17);                /* 2^(e-15)*(1+f/4) */
  return s ? -v : v;
}

static double load_elem(const void* base, int dtype, int64_t idx) {
  switch (dtype) {
    case OR_F32: { float f; memcpy(&f, (const char*)base + 4 * idx, 4); return (double)f; }
    case OR_F16: { uint16_t h; memcpy(&h, (const char*)base + 2 * idx, 2); return dec_f16(h); }
    case OR_BF16: { uint16_t h; memcpy(&h, (const char*)base + 2 * idx, 2); return dec_bf16(h); }
    case OR_E5M2: return dec_e5m2(((const uint8_t*)base)[idx]);
    default: return NAN;
  }
}

/* Exported so the tests can pin the format decoders on their own. */
int oracle_decode(int dtype, const void* src, int64_t n, double* dst) {
  if (dtype < OR_F32 || dtype > OR_E5M2) return -1;
  for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, dtype, i);
  return 0;
}

/* One output vector: query token `t` (global index into the packed q), head h. */
static void attend_one(const oracle_problem* p, int b, int64_t t, int h,
                       const int32_t* cu, const int32_t* lens, const int32_t* bt,
                       const void* q, const void* kc, const void* vc,
                       double* xbuf, double* qv, double* out) {
  const int d = p->head_dim, P = p->page_size;
  const int g = p->num_q_heads / p->num_kv_heads;
  const int kh = h / g;
  const int64_t qb = (int64_t)cu[b + 1] - cu[b];
  const int64_t L = lens[b];
  const int64_t i = t - cu[b];
  const int64_t last = L - qb + i;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (L <= 0 || last < 0) return;

  for (int c = 0; c < d; ++c)
    qv[c] = load_elem(q, p->q_dtype, (t * p->num_q_heads + h) * (int64_t)d + c);

  /* logits */
  double m = -INFINITY;
  for (int64_t j = 0; j <= last; ++j) {
    const int64_t page = bt[(int64_t)b * p->max_pages_per_row + j / P];
    const int64_t base = ((page * P + j % P) * p->num_kv_heads + kh) * (int64_t)d;
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
      acc += qv[c] * (load_elem(kc, p->kv_dtype, base + c) * p->k_scale);
    const double x = p->softmax_scale * acc;
    xbuf[j] = x;
    if (x > m) m = x;
  }
  /* weights and weighted sum of values */
  double den = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    const double w = exp(xbuf[j] - m);
    den += w;
    const int64_t page = bt[(int64_t)b * p->max_pages_per_row + j / P];
    const int64_t base = ((page * P + j % P) * p->num_kv_heads + kh) * (int64_t)d;
    for (int c = 0; c < d; ++c)
      out[c] += w * (load_elem(vc, p->kv_dtype, base + c) * p->v_scale);
  }
  for (int c = 0; c < d; ++c) out[c] /= den;
}

/*
 * Computes out[n, Hq, d] (double) for the query tokens listed in `tokens`
 * (global indices into the packed q), or for every token when tokens == NULL
 * (then n = cu_seqlens_q[num_rows]).  Returns 0, or -1 on a malformed problem.
 */
int oracle_paged_attention(const oracle_problem* p, const int32_t* cu_seqlens_q,
                           const int32_t* seq_lens, const int32_t* block_table,
                           const void* q, const void* k_cache, const void* v_cache,
                           const int64_t* tokens, int64_t n_tokens, double* out,
                           int n_threads) {
  if (!p || p->num_rows < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
      p->num_q_heads % p->num_kv_heads || p->head_dim <= 0 || p->page_size <= 0)
    return -1;
  const int64_t total_q = p->num_rows ? cu_seqlens_q[p->num_rows] : 0;
  if (!tokens) n_tokens = total_q;
  int64_t max_len = 1;
  for (int b = 0; b < p->num_rows; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];

  /* row of each requested token */
  int32_t* row_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_tokens ? n_tokens : 1));
  if (!row_of) return -2;
  for (int64_t n = 0; n < n_tokens; ++n) {
    const int64_t t = tokens ? tokens[n] : n;
    if (t < 0 || t >= total_q) { free(row_of); return -1; }
    int lo = 0, hi = p->num_rows - 1;           /* largest b with cu[b] <= t */
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (cu_seqlens_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    row_of[n] = lo;
  }

  const int64_t work = n_tokens * p->num_q_heads;
  const int d = p->head_dim;
#ifdef _OPENMP
  /* this call's team size only: later calls with n_threads <= 0 use all cores */
  const int team = n_threads > 0 ? n_threads : omp_get_max_threads();
#else
  (void)n_threads;
#endif
  int err = 0;
#pragma omp parallel num_threads(team)
  {
    double* xbuf = (double*)malloc(sizeof(double) * (size_t)max_len);
    double* qv = (double*)malloc(sizeof(double) * (size_t)d);
    if (!xbuf || !qv) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t w = 0; w < work; ++w) {
        const int64_t n = w / p->num_q_heads;
        const int h = (int)(w % p->num_q_heads);
        const int64_t t = tokens ? tokens[n] : n;
        attend_one(p, row_of[n], t, h, cu_seqlens_q, seq_lens, block_table, q, k_cache,
                   v_cache, xbuf, qv, out + w * (int64_t)d);
      }
    }
    free(xbuf);
    free(qv);
  }
  free(row_of);
  return err;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
