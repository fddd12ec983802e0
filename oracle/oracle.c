/*
 * Plain CPU oracle for attention over a paged FP8 E4M3 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the package's smoke check and the benchmark's CPU-baseline leg may build,
 * load or call it; the library itself never does.  It shares no code, header,
 * table or constant with the CUDA sources.
 *
 * What it computes (sources are the pages this project follows):
 *  - E4M3 decode and encode: the FP8 E4M3 format named as the KV-cache and Q
 *    storage type in "[Kernel] Integrate FA4 SM90 FP8 MMA for Gemma-4 full
 *    attention" (vLLM PR 60372, Overview) and vLLM PR 63139 (Overview: "E4M3
 *    Q/K/V").  The bit layout (1 sign, 4 exponent bits with bias 7, 3 mantissa
 *    bits, no infinities, S.1111.111 = NaN, max 448) is the OCP 8-bit
 *    floating-point definition of E4M3; decode is written from that closed form.
 *  - Q quantization: sliding-window layers quantize Q to FP8 (PR 63139,
 *    Overview, "Sliding-window layers (head dim 256) quantize Q to FP8").
 *    Reading used: q8 = round-to-nearest-even, saturating, of the fp32 quotient
 *    q / q_descale.
 *  - Attention: softmax(scale * q.k) v over the keys each query may see, read
 *    through the block table of 64-token pages (PR 60372 review thread,
 *    "page_size == tile_n, which is 64 for d512"; vLLM PR 48666 summary,
 *    flash_attn_varlen_func snippet), with K/V dequantized as code * descale
 *    (PR 48666 summary: K/V descales folded in-kernel).  Query i of a sequence
 *    with Lq queries and Lk keys sits at position p = Lk - Lq + i (bottom-right
 *    alignment of the varlen interface); it sees keys [lo, hi] with
 *    lo = max(0, p - window_left) when window_left >= 0 (else 0) and
 *    hi = p when causal (else Lk - 1), clipped to Lk - 1.  lse = m + ln(l),
 *    natural log; an empty visible set gives o = 0 and lse = -inf.
 *
 *  - KV-cache write: the kernels that reshape newly generated keys and values
 *    and write them into the paged cache, FP8 conversion included ("Why FP8 is
 *    slower than BF16", the KV-cache writes row of the profiling table and the
 *    paragraph after it).  Reading used: token t goes to slot s = slot_mapping[t]
 *    (page s / 64, row s % 64 of the [pages][64][Hkv][D] cache), a negative slot
 *    is a padding token that writes nothing, and each element is quantized like
 *    Q: E4M3_RNE_sat(fl32(x / descale)) with the per-tensor K or V descale.
 *
 *  - Attention sinks: listed as a feature of the d512 kernel ("[Kernel]
 *    Integrate FA4 SM90 FP8 MMA for Gemma-4 full attention", review comment
 *    on the d512 specialization: "including sinks").  Reading used (the page
 *    defines no formula): a per-query-head logit sink_h joins the softmax
 *    denominator and attends to no value, o = sum_j e^{s_j} v_j /
 *    (sum_j e^{s_j} + e^{sink_h}) and lse = ln(sum_j e^{s_j} + e^{sink_h}).
 *  - Combining attention partials by their LSE: the context call of
 *    decode-context parallelism, in which each rank attends over its shard of
 *    the keys and returns its output and LSE ("[Kernel] Integrate FA4 SM90 FP8
 *    MMA for Gemma-4 full attention", review thread on DCP: the non-causal
 *    context call run as local attention with a window covering every key,
 *    and a DCP=2 emulation).  With parts s over disjoint key sets,
 *    L = ln sum_s exp(LSE_s) and O = sum_s exp(LSE_s - L) O_s; parts with
 *    LSE = -inf add nothing, and a row with no part gives O = 0, L = -inf.
 *
 * Everything is fp64 except the places the method fixes fp32 (the quotients
 * q / q_descale and x / k_descale, x / v_descale before rounding to E4M3).  No blocking, fusion or reordering:
 * one query row at a time, keys in increasing order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_PAGE 64

/* ------------------------------------------------------------------ E4M3 */

/* Closed-form value of an E4M3 code.  NaN for S.1111.111 (0x7F, 0xFF). */
double or_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Round a non-negative double holding an exact value to the nearest integer,
 * ties to even. */
static double round_half_even(double n) {
  double f = floor(n);
  double d = n - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Encode an fp32 value as E4M3: round to nearest, ties to the even code,
 * saturating to +-448 (also for +-inf), NaN -> 0x7F with the sign kept,
 * zero and underflow keep the sign (-0 -> 0x80). */
uint8_t or_e4m3_encode(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a;
  int code;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal binade: grid step 2^-9; n = 8 lands exactly on 2^-6 = code 0x08 */
    code = (int)round_half_even(ldexp(a, 9));
  } else {
    int E;
    double f = frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int eb = E - 1;           /* a in [2^eb, 2^(eb+1)), eb in [-6, 8] */
    double n = ldexp(a, 3 - eb); /* in [8, 16): 1.mmm scaled by 8 */
    int r = (int)round_half_even(n);
    (void)f;
    if (r == 16) {
      eb += 1;
      r = 8;
    }
    code = ((eb + 7) << 3) | (r - 8);
  }
  return (uint8_t)(sign | (uint8_t)code);
}

/* or_e4m3_encode over an array. */
void or_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i]);
}

/* The 256 decoded values, filled once from the closed form above. */
static double g_dec[256];
static pthread_once_t g_dec_once = PTHREAD_ONCE_INIT;
static void fill_dec(void) {
  int c;
  for (c = 0; c < 256; ++c) g_dec[c] = or_e4m3_decode((uint8_t)c);
}
static const double* dec_table(void) {
  pthread_once(&g_dec_once, fill_dec);
  return g_dec;
}

static float bf16_bits_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* q8 = E4M3_RNE_sat(fl32(q / q_descale)).  The quotient is formed in double
 * and rounded once to float, which equals the correctly rounded fp32 quotient
 * (double carries more than 2*24+2 bits).  A NaN quotient (NaN input, 0/0,
 * inf/inf) encodes as 0x7F carrying the sign bit of the input q: the sign of
 * a NaN produced by a division is not fixed by IEEE 754, so the input's sign
 * is the one kept. */
void or_quantize_q(const uint16_t* q_bf16, int64_t n, float q_descale, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) {
    float x = bf16_bits_to_float(q_bf16[i]);
    float v = (float)((double)x / (double)q_descale);
    if (isnan(v))
      out[i] = (uint8_t)(0x7F | ((q_bf16[i] >> 8) & 0x80));
    else
      out[i] = or_e4m3_encode(v);
  }
}

/* ------------------------------------------------------------------ KV-cache write */

/* One element: the same rule as or_quantize_q (fp32 quotient, RNE-saturating
 * E4M3, a NaN quotient to 0x7F with the input's sign). */
static uint8_t quant_elem(uint16_t bits, float descale) {
  float x = bf16_bits_to_float(bits);
  float v = (float)((double)x / (double)descale);
  if (isnan(v)) return (uint8_t)(0x7F | ((bits >> 8) & 0x80));
  return or_e4m3_encode(v);
}

/* Writes token t of key/value (bf16 bit patterns, row t at t * token_stride
 * elements, num_heads_kv * head_dim contiguous elements per row) into slot
 * slot_mapping[t] of k_cache / v_cache ([num_pages][64][num_heads_kv][head_dim]
 * bytes).  Negative slots are skipped; slots at or past num_pages * 64 are
 * counted and skipped.  Returns the number of such bad slots. */
int64_t or_kv_cache_write(const uint16_t* key, const uint16_t* value, int64_t key_token_stride,
                          int64_t value_token_stride, const int64_t* slot_mapping, int64_t num_tokens,
                          int num_heads_kv, int head_dim, float k_descale, float v_descale, uint8_t* k_cache,
                          uint8_t* v_cache, int64_t num_pages) {
  int64_t t, bad = 0;
  const int64_t row = (int64_t)num_heads_kv * head_dim;
  for (t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    int64_t page, off, e;
    if (s < 0) continue;
    if (s >= num_pages * OR_PAGE) {
      ++bad;
      continue;
    }
    page = s / OR_PAGE;
    off = s % OR_PAGE;
    for (e = 0; e < row; ++e) {
      const int64_t dst = (page * OR_PAGE + off) * row + e;
      k_cache[dst] = quant_elem(key[t * key_token_stride + e], k_descale);
      v_cache[dst] = quant_elem(value[t * value_token_stride + e], v_descale);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ LSE combine */

/* o_parts: bf16 bit patterns [num_parts][total_q][hq][d]; lse_parts: f32
 * [num_parts][hq][total_q] (natural log).  out: fp64 [total_q][hq][d];
 * lse: fp64 [hq][total_q]. */
void or_lse_combine(const uint16_t* o_parts, const float* lse_parts, int num_parts, int64_t total_q, int hq, int d,
                    double* out, double* lse) {
  int64_t t;
  int h, s, e;
  const int64_t rows = total_q * hq;
  for (t = 0; t < total_q; ++t) {
    for (h = 0; h < hq; ++h) {
      double m = -INFINITY, sum = 0.0, L;
      double* o = out + (t * hq + h) * d;
      for (e = 0; e < d; ++e) o[e] = 0.0;
      for (s = 0; s < num_parts; ++s) {
        const double ls = lse_parts[(int64_t)s * rows + (int64_t)h * total_q + t];
        if (ls > m) m = ls;
      }
      if (m == -INFINITY) {
        lse[(int64_t)h * total_q + t] = -INFINITY;
        continue;
      }
      for (s = 0; s < num_parts; ++s) {
        const double ls = lse_parts[(int64_t)s * rows + (int64_t)h * total_q + t];
        if (ls != -INFINITY) sum += exp(ls - m);
      }
      L = m + log(sum);
      lse[(int64_t)h * total_q + t] = L;
      for (s = 0; s < num_parts; ++s) {
        const double ls = lse_parts[(int64_t)s * rows + (int64_t)h * total_q + t];
        const uint16_t* os = o_parts + ((int64_t)s * rows + t * hq + h) * d;
        double wgt;
        if (ls == -INFINITY) continue;
        wgt = exp(ls - L);
        for (e = 0; e < d; ++e) o[e] += wgt * (double)bf16_bits_to_float(os[e]);
      }
    }
  }
}

/* ------------------------------------------------------------------ attention */

typedef struct {
  int q_is_e4m3;           /* 1: q holds E4M3 codes (dequant: code * q_descale); 0: bf16 bits */
  const void* q;           /* [total_q][Hq][D] */
  const uint8_t* k_cache;  /* [num_pages][64][Hkv][D] E4M3 codes */
  const uint8_t* v_cache;  /* same layout */
  int64_t num_pages;
  const int32_t* block_table; /* [batch][max_pages_per_seq] */
  int max_pages_per_seq;
  const int32_t* cu_seqlens_q; /* [batch + 1] */
  const int32_t* seqused_k;    /* [batch] */
  int batch, total_q, num_heads_q, num_heads_kv, head_dim;
  float q_descale;             /* per tensor */
  const float* k_descale;      /* indexed b * descale_batch_stride + hk * descale_head_stride */
  const float* v_descale;
  int descale_batch_stride, descale_head_stride;
  float softmax_scale;
  int window_left; /* < 0: no window */
  int causal;
  const float* sinks; /* [Hq] sink logits (natural-log units), or NULL */
} or_attn_args;

/* Visible key range [*lo, *hi] of query i in a sequence with Lq queries and
 * Lk keys; returns 0 when the range is empty. */
int or_visible_range(int Lq, int Lk, int i, int window_left, int causal, int* lo, int* hi) {
  long p = (long)Lk - (long)Lq + (long)i;
  long l = 0, h = (long)Lk - 1;
  if (window_left >= 0) l = p - window_left > 0 ? p - window_left : 0;
  if (causal && p < h) h = p;
  *lo = (int)l;
  *hi = (int)h;
  return l <= h && Lk > 0;
}

/* Sequence b with cu_seqlens_q[b] <= t < cu_seqlens_q[b + 1], or -1. */
static int find_seq(const or_attn_args* a, int t) {
  int lo = 0, hi = a->batch - 1, b = -1;
  while (lo <= hi) { /* largest b with cu_seqlens_q[b] <= t */
    int mid = lo + (hi - lo) / 2;
    if (a->cu_seqlens_q[mid] <= t) {
      b = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  if (b < 0 || t >= a->cu_seqlens_q[b + 1]) return -1;
  return b;
}

/* Decoded q row (with q_descale for E4M3 input) into qd[D]. */
static void load_q(const or_attn_args* a, int t, int h, double* qd) {
  const double* dec = dec_table();
  int d, D = a->head_dim;
  size_t base = ((size_t)t * a->num_heads_q + h) * D;
  for (d = 0; d < D; ++d) {
    if (a->q_is_e4m3)
      qd[d] = dec[((const uint8_t*)a->q)[base + d]] * (double)a->q_descale;
    else
      qd[d] = (double)bf16_bits_to_float(((const uint16_t*)a->q)[base + d]);
  }
}

/* Byte offset of key/value row j of sequence b, KV head hk, or -1 on a bad page id. */
static int64_t kv_row_offset(const or_attn_args* a, int b, int j, int hk) {
  int32_t phys = a->block_table[(size_t)b * a->max_pages_per_seq + j / OR_PAGE];
  if (phys < 0 || phys >= a->num_pages) return -1;
  return (((int64_t)phys * OR_PAGE + (j % OR_PAGE)) * a->num_heads_kv + hk) * a->head_dim;
}

/* One query row (token t, head h).  Writes o[D] and *lse.  If probs != NULL
 * it also receives the softmax weight of every key 0..Lk-1 (0 outside J).
 * Returns 0 on success, -1 on a bad page id, -2 on a bad token. */
static int attend_row(const or_attn_args* a, int t, int h, double* o, double* lse, double* probs,
                      double* qd, double* s) {
  const double* dec = dec_table();
  int b = find_seq(a, t);
  int D = a->head_dim, G, hk, Lq, Lk, i, lo, hi, j, d;
  double kd, vd, m, l;
  if (b < 0) return -2;
  G = a->num_heads_q / a->num_heads_kv;
  hk = h / G;
  Lq = a->cu_seqlens_q[b + 1] - a->cu_seqlens_q[b];
  Lk = a->seqused_k[b];
  i = t - a->cu_seqlens_q[b];
  kd = (double)a->k_descale[(size_t)b * a->descale_batch_stride + (size_t)hk * a->descale_head_stride];
  vd = (double)a->v_descale[(size_t)b * a->descale_batch_stride + (size_t)hk * a->descale_head_stride];
  for (d = 0; d < D; ++d) o[d] = 0.0;
  if (probs)
    for (j = 0; j < Lk; ++j) probs[j] = 0.0;
  if (!or_visible_range(Lq, Lk, i, a->window_left, a->causal, &lo, &hi)) {
    /* no key: the sink alone (if any) makes up the denominator, o = 0 */
    *lse = a->sinks ? (double)a->sinks[h] : -INFINITY;
    return 0;
  }
  load_q(a, t, h, qd);
  /* logits over the visible set only */
  m = -INFINITY;
  for (j = lo; j <= hi; ++j) {
    int64_t off = kv_row_offset(a, b, j, hk);
    double acc = 0.0;
    if (off < 0) return -1;
    for (d = 0; d < D; ++d) acc += qd[d] * (dec[a->k_cache[off + d]] * kd);
    s[j - lo] = (double)a->softmax_scale * acc;
    if (s[j - lo] > m) m = s[j - lo];
  }
  /* a sink is one more logit in the denominator that attends to no value */
  if (a->sinks && (double)a->sinks[h] > m) m = (double)a->sinks[h];
  l = 0.0;
  for (j = lo; j <= hi; ++j) l += exp(s[j - lo] - m);
  if (a->sinks) l += exp((double)a->sinks[h] - m);
  for (j = lo; j <= hi; ++j) {
    int64_t off = kv_row_offset(a, b, j, hk);
    double w = exp(s[j - lo] - m) / l;
    if (probs) probs[j] = w;
    for (d = 0; d < D; ++d) o[d] += w * (dec[a->v_cache[off + d]] * vd);
  }
  *lse = m + log(l);
  return 0;
}

typedef struct {
  const or_attn_args* a;
  const int32_t* rows; /* pairs (token, head), or NULL for all rows in (token, head) order */
  int64_t nrows;
  double* out;
  double* lse;
  int64_t next;
  int status;
  pthread_mutex_t mu;
} work_t;

static void* worker(void* arg) {
  work_t* w = (work_t*)arg;
  const or_attn_args* a = w->a;
  int max_lk = a->max_pages_per_seq * OR_PAGE;
  double* qd = (double*)malloc(sizeof(double) * (size_t)a->head_dim);
  double* s = (double*)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
  for (;;) {
    int64_t r, r_end;
    pthread_mutex_lock(&w->mu);
    r = w->next;
    w->next += 16;
    pthread_mutex_unlock(&w->mu);
    if (r >= w->nrows) break;
    r_end = r + 16 < w->nrows ? r + 16 : w->nrows;
    for (; r < r_end; ++r) {
      int t, h, rc;
      if (w->rows) {
        t = w->rows[2 * r];
        h = w->rows[2 * r + 1];
      } else {
        t = (int)(r / a->num_heads_q);
        h = (int)(r % a->num_heads_q);
      }
      rc = attend_row(a, t, h, w->out + r * a->head_dim, w->lse + r, NULL, qd, s);
      if (rc != 0) {
        pthread_mutex_lock(&w->mu);
        w->status = rc;
        pthread_mutex_unlock(&w->mu);
      }
    }
  }
  free(qd);
  free(s);
  return NULL;
}

static int check_args(const or_attn_args* a) {
  int b;
  if (a->num_heads_kv <= 0 || a->num_heads_q % a->num_heads_kv != 0 || a->head_dim <= 0) return -3;
  for (b = 0; b < a->batch; ++b) {
    if (a->seqused_k[b] < 0 || a->seqused_k[b] > a->max_pages_per_seq * OR_PAGE) return -4;
    if (a->cu_seqlens_q[b + 1] < a->cu_seqlens_q[b]) return -4;
  }
  return 0;
}

/* Attention for `nrows` (token, head) pairs (rows == NULL: every pair, in
 * token-major order, out laid out [total_q][Hq][D]).  out[r][D], lse[r].
 * Returns 0, or a negative code (-1 bad page id, -2 bad token, -3 bad heads,
 * -4 bad lengths).  nthreads <= 0 uses every online core. */
int or_paged_attention(const or_attn_args* a, const int32_t* rows, int64_t nrows, double* out, double* lse,
                       int nthreads) {
  work_t w;
  pthread_t* th;
  int i, rc = check_args(a);
  if (rc) return rc;
  if (!rows) nrows = (int64_t)a->total_q * a->num_heads_q;
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  w.a = a;
  w.rows = rows;
  w.nrows = nrows;
  w.out = out;
  w.lse = lse;
  w.next = 0;
  w.status = 0;
  pthread_mutex_init(&w.mu, NULL);
  th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &w);
  for (i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&w.mu);
  return w.status;
}

/* Softmax weights of one query row over keys 0..Lk-1 (0 outside the visible
 * set), plus its output row and lse.  probs must hold Lk doubles. */
int or_attention_probs(const or_attn_args* a, int token, int head, double* probs, double* o, double* lse) {
  int rc = check_args(a);
  int max_lk = a->max_pages_per_seq * OR_PAGE;
  double* qd;
  double* s;
  if (rc) return rc;
  qd = (double*)malloc(sizeof(double) * (size_t)a->head_dim);
  s = (double*)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
  rc = attend_row(a, token, head, o, lse, probs, qd, s);
  free(qd);
  free(s);
  return rc;
}

int or_page_size(void) { return OR_PAGE; }
