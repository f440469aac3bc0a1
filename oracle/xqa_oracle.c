/*
 * Paged-KV decode attention: float64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference legs may load this code.  It shares no
 * code, header, table or helper with the CUDA library; it never includes
 * include/xqa.h.
 *
 * What it computes (FlashInfer "flashinfer.xqa.xqa" API page, parameter list
 * and the shape-inference note; vLLM Kimi-K3 MultiHeadLatentAttention page,
 * __init__ "head_size"/"scale" and _attention's forward_mqa call for the MLA
 * variant): exact softmax attention, in float64, of every query row against
 * the logical token sequence that the page table describes.
 *
 *   for each batch b, query token i < q_seq_len, query head h:
 *     L    = seq_lens[b]                     (includes the q_seq_len new tokens)
 *     p    = L - q_seq_len + i               (the query's own position)
 *     kvh  = h / G, g = h % G, G = Hq / Hkv  (head_group_ratio)
 *     K[t] = k_cache row of token t: page page_table[b][t / page_size],
 *            slot t % page_size, head kvh                (NHD or HND layout)
 *     V[t] = first Dv elements of the v_cache row of token t
 *     visible(t) = t < L
 *                  and (W == 0 or t > p - W)                  sliding window
 *                  and (t < L - q_seq_len or mask bit (i, t - (L - q_seq_len)))
 *     s_t  = softmax_scale * q_scale * kv_scale * sum_d q[b,i,h,d] K[t,d]
 *     M    = max(max_t s_t, sigma),  sigma = sinks[kvh][g] or -inf
 *     Z    = sum_t exp(s_t - M) + exp(sigma - M)
 *     out  = rcp_out_scale * kv_scale * sum_t exp(s_t - M) V[t] / Z
 *   (out = 0 when nothing is visible and there is no sink.)
 *
 * Element decodes follow the formats' bit definitions: bfloat16 is the high
 * half of an IEEE binary32; binary16 is 1-5-10 with bias 15; float8 e4m3fn is
 * 1-4-3 with bias 7, subnormals, no infinities and S.1111.111 = NaN.
 *
 * Mask words: the mask row of (b, i) holds ((q_seq_len + 31) / 32) * 2 uint16
 * values; consecutive pairs form little-endian 32-bit words, and bit (j % 32)
 * of word (j / 32) set means query token i may attend to speculative key j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes used by this oracle's own Python wrapper */
#define ORC_F16 0
#define ORC_BF16 1
#define ORC_E4M3 2

static double orc_decode_bf16(uint16_t bits) {
  uint32_t wide = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &wide, sizeof f);
  return (double)f;
}

static double orc_decode_f16(uint16_t bits) {
  int sign = bits >> 15;
  int expo = (bits >> 10) & 0x1f;
  int mant = bits & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24); /* subnormal: mant/1024 * 2^-14 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + mant), expo - 25); /* (1 + mant/1024) 2^(e-15) */
  }
  return sign ? -v : v;
}

static double orc_decode_e4m3(uint8_t bits) {
  int sign = bits >> 7;
  int expo = (bits >> 3) & 0xf;
  int mant = bits & 0x7;
  double v;
  if (expo == 15 && mant == 7) return NAN;
  if (expo == 0) {
    v = ldexp((double)mant, -9); /* subnormal: mant/8 * 2^-6 */
  } else {
    v = ldexp((double)(8 + mant), expo - 10); /* (1 + mant/8) 2^(e-7) */
  }
  return sign ? -v : v;
}

static double orc_load(const void* base, int dtype, int64_t idx) {
  if (dtype == ORC_E4M3) return orc_decode_e4m3(((const uint8_t*)base)[idx]);
  if (dtype == ORC_BF16) return orc_decode_bf16(((const uint16_t*)base)[idx]);
  return orc_decode_f16(((const uint16_t*)base)[idx]);
}

/* Exported so that tests can compare every code against a library decode. */
double oracle_decode(int dtype, uint32_t bits) {
  if (dtype == ORC_E4M3) return orc_decode_e4m3((uint8_t)bits);
  if (dtype == ORC_BF16) return orc_decode_bf16((uint16_t)bits);
  return orc_decode_f16((uint16_t)bits);
}

typedef struct {
  const void* q;
  int q_dtype;
  const void* k_cache;
  const void* v_cache;
  int kv_dtype;
  int layout_hnd; /* 0: [pages, page_size, Hkv, D]; 1: [pages, Hkv, page_size, D] */
  int64_t num_pages;
  const int32_t* page_table; /* [B, pages_per_seq] */
  int pages_per_seq;
  const uint32_t* seq_lens; /* [B] */
  int batch, num_q_heads, num_kv_heads, head_dim, v_head_dim, page_size, q_seq_len;
  const float* sinks; /* [Hkv, G] or NULL */
  double q_scale, kv_scale, softmax_scale;
  int sliding_win_size;
  double rcp_out_scale;
  const uint16_t* mask; /* [B, q_seq_len, ((q_seq_len + 31) / 32) * 2] or NULL */
} orc_problem;

/* Offset of element d of token t's row for kv head kvh, or -1 if the page
 * table entry points outside the pool. */
static int64_t orc_row_offset(const orc_problem* P, int b, int64_t t, int kvh) {
  int64_t page = P->page_table[(int64_t)b * P->pages_per_seq + t / P->page_size];
  int64_t slot = t % P->page_size;
  if (page < 0 || page >= P->num_pages) return -1;
  if (P->layout_hnd)
    return ((page * P->num_kv_heads + kvh) * P->page_size + slot) * P->head_dim;
  return ((page * P->page_size + slot) * P->num_kv_heads + kvh) * P->head_dim;
}

static int orc_mask_bit(const orc_problem* P, int b, int i, int64_t j) {
  int64_t words_u16 = ((P->q_seq_len + 31) / 32) * 2;
  const uint16_t* row = P->mask + ((int64_t)b * P->q_seq_len + i) * words_u16;
  uint32_t word = (uint32_t)row[2 * (j / 32)] | ((uint32_t)row[2 * (j / 32) + 1] << 16);
  return (word >> (j % 32)) & 1u;
}

/* One output row: unit = (b * q_seq_len + i) * Hq + h.  Returns 0, or -1 for
 * an out-of-range page, or -2 for a sequence longer than the page table. */
static int orc_one_row(const orc_problem* P, int64_t unit, double* out_row, double* logits,
                       double* lse) {
  int Hq = P->num_q_heads, G = P->num_q_heads / P->num_kv_heads;
  int h = (int)(unit % Hq);
  int i = (int)((unit / Hq) % P->q_seq_len);
  int b = (int)(unit / ((int64_t)Hq * P->q_seq_len));
  int kvh = h / G, g = h % G;
  int64_t L = P->seq_lens[b];
  if (L > (int64_t)P->pages_per_seq * P->page_size) return -2;
  int64_t spec0 = L - P->q_seq_len; /* first speculative (new) token */
  int64_t pos = spec0 + i;
  const int64_t q_off = (((int64_t)b * P->q_seq_len + i) * Hq + h) * P->head_dim;
  const double logit_scale = P->softmax_scale * P->q_scale * P->kv_scale;

  /* step 1: logits of the visible keys (-inf marks an invisible key) */
  double m = -INFINITY;
  for (int64_t t = 0; t < L; ++t) {
    int visible = 1;
    if (P->sliding_win_size > 0 && !(t > pos - P->sliding_win_size)) visible = 0;
    if (visible && P->mask && t >= spec0 && !orc_mask_bit(P, b, i, t - spec0)) visible = 0;
    if (!visible) {
      logits[t] = -INFINITY;
      continue;
    }
    int64_t off = orc_row_offset(P, b, t, kvh);
    if (off < 0) return -1;
    double dot = 0.0;
    for (int d = 0; d < P->head_dim; ++d)
      dot += orc_load(P->q, P->q_dtype, q_off + d) * orc_load(P->k_cache, P->kv_dtype, off + d);
    logits[t] = logit_scale * dot;
    if (logits[t] > m) m = logits[t];
  }
  double sigma = P->sinks ? (double)P->sinks[kvh * G + g] : -INFINITY;
  if (sigma > m) m = sigma;

  /* step 2: normaliser and weighted sum of values */
  for (int d = 0; d < P->v_head_dim; ++d) out_row[d] = 0.0;
  *lse = -INFINITY;
  if (m == -INFINITY) return 0; /* nothing visible and no sink */
  double z = exp(sigma - m);
  for (int64_t t = 0; t < L; ++t) {
    if (logits[t] == -INFINITY) continue;
    double w = exp(logits[t] - m);
    z += w;
    int64_t off = orc_row_offset(P, b, t, kvh);
    for (int d = 0; d < P->v_head_dim; ++d) out_row[d] += w * orc_load(P->v_cache, P->kv_dtype, off + d);
  }
  for (int d = 0; d < P->v_head_dim; ++d) out_row[d] = P->rcp_out_scale * P->kv_scale * out_row[d] / z;
  /* log-sum-exp of the row's logits (natural log), the sink included: the
   * normaliser that the output was divided by, as merge_attn_states takes it */
  *lse = m + log(z);
  return 0;
}

/*
 * Computes the rows listed in `units` (unit = (b * q_seq_len + i) * Hq + h)
 * into out[n_units][v_head_dim], or every row into out[B][q_seq_len][Hq][Dv]
 * when units is NULL.  Returns 0 on success, a negative code on bad input.
 */
int oracle_xqa_attention(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                         int kv_dtype, int layout_hnd, int64_t num_pages, const int32_t* page_table,
                         int pages_per_seq, const uint32_t* seq_lens, int batch, int num_q_heads,
                         int num_kv_heads, int head_dim, int v_head_dim, int page_size,
                         int q_seq_len, const float* sinks, double q_scale, double kv_scale,
                         double softmax_scale, int sliding_win_size, double rcp_out_scale,
                         const uint16_t* mask, const int64_t* units, int64_t n_units, double* out,
                         double* lse, int n_threads) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -3;
  if (head_dim <= 0 || v_head_dim <= 0 || v_head_dim > head_dim || page_size <= 0) return -3;
  if (q_seq_len <= 0 || pages_per_seq <= 0 || sliding_win_size < 0) return -3;
  orc_problem P = {q, q_dtype, k_cache, v_cache, kv_dtype, layout_hnd, num_pages, page_table,
                   pages_per_seq, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                   v_head_dim, page_size, q_seq_len, sinks, q_scale, kv_scale, softmax_scale,
                   sliding_win_size, rcp_out_scale, mask};
  int64_t total = (int64_t)batch * q_seq_len * num_q_heads;
  int64_t n = units ? n_units : total;
  int64_t max_len = (int64_t)pages_per_seq * page_size;
  int status = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double* logits = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t k = 0; k < n; ++k) {
      int64_t unit = units ? units[k] : k;
      double row_lse = -INFINITY;
      int rc = (unit < 0 || unit >= total) ? -3
                                           : orc_one_row(&P, unit, out + k * v_head_dim, logits, &row_lse);
      if (lse) lse[k] = row_lse;
      if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
        status = rc;
      }
    }
    free(logits);
  }
  return status;
}

/*
 * merge_attn_states (vLLM Kimi-K3 MultiHeadLatentAttention page, the prefill
 * path with chunked context): two attention results over disjoint key sets,
 * each normalised by its own sum, with their log-sum-exps, combine into the
 * result over the union:
 *   M = max(lse_p, lse_s),  w_p = exp(lse_p - M),  w_s = exp(lse_s - M),
 *   out = (w_p * out_p + w_s * out_s) / (w_p + w_s),  lse = M + log(w_p + w_s).
 * Rows t >= n_with_prefix have no prefix: they take the suffix unchanged.  A
 * side whose lse is -inf (no visible key) gets weight 0; both -inf gives 0.
 * Layout: out_*[T][H][D], lse_*[T][H]; all float64.
 */
void oracle_merge_attn_states(const double* out_p, const double* lse_p, const double* out_s,
                              const double* lse_s, int64_t T, int64_t H, int64_t D,
                              int64_t n_with_prefix, double* out, double* lse) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t r = t * H + h;
      double wp = 0.0, ws = 1.0, M = lse_s[r];
      if (t < n_with_prefix) {
        M = lse_p[r] > lse_s[r] ? lse_p[r] : lse_s[r];
        wp = M == -INFINITY ? 0.0 : exp(lse_p[r] - M);
        ws = M == -INFINITY ? 0.0 : exp(lse_s[r] - M);
      }
      const double z = wp + ws;
      for (int64_t d = 0; d < D; ++d)
        out[r * D + d] = z == 0.0 ? 0.0 : (wp * out_p[r * D + d] + ws * out_s[r * D + d]) / z;
      lse[r] = z == 0.0 ? -INFINITY : M + log(z);
    }
}

/*
 * OCP FP8 E4M3FN encoding of x (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities, S.1111.111 is NaN): round to nearest, ties to even, and
 * saturate finite values beyond the largest magnitude 448 to +-448.  NaN maps
 * to 0x7f.
 */
uint32_t oracle_encode_e4m3(double x) {
  if (isnan(x)) return 0x7fu;
  uint32_t sign = signbit(x) ? 0x80u : 0u;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7eu;
  /* the representable magnitudes are k * 2^(e-3) for normals (e >= -6, k in
   * 8..15) and k * 2^-9 for subnormals (k in 0..7): scale to the spacing and
   * round the integer k, ties to even */
  int ex = 0;
  if (a > 0.0) frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
  int e = a > 0.0 ? ex - 1 : -7;
  if (e < -6) e = -6;
  double q = ldexp(a, 3 - e); /* position in units of the spacing at exponent e */
  double k = floor(q);
  double rem = q - k;
  if (rem > 0.5 || (rem == 0.5 && fmod(k, 2.0) != 0.0)) k += 1.0;
  if (k >= 16.0) { k = 8.0; e += 1; } /* carried into the next binade */
  if (e > 8 || (e == 8 && k > 14.0)) return sign | 0x7eu;
  uint32_t code;
  if (k < 8.0) code = (uint32_t)k; /* subnormal (only possible at e = -6) */
  else code = ((uint32_t)(e + 7) << 3) | ((uint32_t)k - 8u);
  return sign | code;
}
