/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged attention over a
 * block-table-addressed KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where the method is stated:
 *  - KV lives in fixed-size physical blocks (16 tokens) that a per-sequence
 *    block table maps logical positions to ("03 - Engines Papers", section 2
 *    "Efficient Memory Management ... PagedAttention (vLLM)", Key trick;
 *    "The LLM inference engine playbook", Theme 3).
 *  - The attention kernel must gather K/V from those non-contiguous blocks
 *    ("03 - Engines Papers", section 2, What to extract).  The oracle does the
 *    gather explicitly into a contiguous fp64 buffer and then evaluates the
 *    plain definition softmax(scale * q K^T) V with an exact two-pass max.
 *    That is the value the online-softmax recurrence (Milakov & Gimelshein,
 *    "References" page) reaches up to rounding order.
 *  - Partial attentions over disjoint key ranges combine by their
 *    log-sum-exp ("03 - Engines Papers", section 12 Cascade Inference; the
 *    split-K reduction of "The LLM inference engine playbook", Theme 4).
 *  - A prefill chunk attends causally over its own paged KV: a query at
 *    absolute position p sees keys 0..p, later chunks' K/V being absent
 *    ("03 - Engines Papers", section 3 Sarathi / Sarathi-Serve).
 *  - GQA: query head h reads kv head h / (Hq / Hkv) ("References" page, GQA).
 *
 * Conventions: bf16 values arrive as raw uint16 bit patterns and are widened
 * exactly to fp64.  Outputs are fp64.  lse is in natural-log units of the
 * scaled scores; an empty key range gives out = 0 and lse = -inf.
 * Every function returns 0 on success and -1 on invalid metadata (an index
 * outside the pool or a length outside the table); it never aborts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_bits_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------------- */
/* Slot scatter: k_cache[slot / bs][slot % bs][h][:] = key[t][h][:].       */
/* A negative slot is padding and is skipped.                              */
/* ---------------------------------------------------------------------- */
int oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                             int64_t key_token_stride, int64_t value_token_stride,
                             uint16_t *k_cache, uint16_t *v_cache,
                             const int64_t *slot_mapping, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks) {
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) return -1;
    int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int c = 0; c < head_dim; ++c) {
        int64_t dst = ((blk * block_size + off) * num_kv_heads + h) * (int64_t)head_dim + c;
        k_cache[dst] = key[(int64_t)t * key_token_stride + (int64_t)h * head_dim + c];
        v_cache[dst] = value[(int64_t)t * value_token_stride + (int64_t)h * head_dim + c];
      }
    }
  }
  return 0;
}

/* Copy-on-write support: whole physical block src -> dst, K and V. */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int64_t *pairs,
                       int num_pairs, int num_kv_heads, int head_dim, int block_size,
                       int64_t num_blocks) {
  int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;
  for (int i = 0; i < num_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -1;
    for (int64_t e = 0; e < block_elems; ++e) {
      k_cache[dst * block_elems + e] = k_cache[src * block_elems + e];
      v_cache[dst * block_elems + e] = v_cache[src * block_elems + e];
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Gather of one sequence's keys/values for one kv head, positions [a, b), */
/* through its block table, into contiguous fp64 rows.                     */
/* ---------------------------------------------------------------------- */
static int gather_rows(const uint16_t *cache, const int32_t *table_row, int kvh,
                       int64_t a, int64_t b, int num_kv_heads, int head_dim,
                       int block_size, int64_t num_blocks, double *rows) {
  for (int64_t j = a; j < b; ++j) {
    int64_t blk = table_row[j / block_size];
    int64_t off = j % block_size;
    if (blk < 0 || blk >= num_blocks) return -1;
    const uint16_t *src = cache + ((blk * block_size + off) * num_kv_heads + kvh) * (int64_t)head_dim;
    for (int c = 0; c < head_dim; ++c) rows[(j - a) * head_dim + c] = bf16_bits_to_f64(src[c]);
  }
  return 0;
}

/* Plain attention of one query over n contiguous rows:
 *   x_j = scale * <q, K_j>,  m = max_j x_j,  w_j = exp(x_j - m),
 *   out = sum_j w_j V_j / sum_j w_j,  lse = m + ln(sum_j w_j).            */
static void attend(const double *q, const double *K, const double *V, int64_t n,
                   int head_dim, double scale, double *x, double *out, double *lse) {
  for (int c = 0; c < head_dim; ++c) out[c] = 0.0;
  if (n <= 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int c = 0; c < head_dim; ++c) dot += q[c] * K[j * head_dim + c];
    x[j] = scale * dot;
    if (x[j] > m) m = x[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double w = exp(x[j] - m);
    sum += w;
    for (int c = 0; c < head_dim; ++c) out[c] += w * V[j * head_dim + c];
  }
  for (int c = 0; c < head_dim; ++c) out[c] /= sum;
  *lse = m + log(sum);
}

/* ---------------------------------------------------------------------- */
/* Decode: one query per sequence, attending over positions [0, seq_len).  */
/* q [S, Hq, D] bf16, out [S, Hq, D] fp64, lse [S, Hq] fp64 (nullable).    */
/* ---------------------------------------------------------------------- */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *seq_lens, int num_seqs, int num_q_heads,
                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                  double scale, double *out, double *lse) {
  int group = num_q_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t pair = 0; pair < (int64_t)num_seqs * num_kv_heads; ++pair) {
    int s = (int)(pair / num_kv_heads), kvh = (int)(pair % num_kv_heads);
    int64_t n = seq_lens[s];
    if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size) {
      bad = 1;
      continue;
    }
    double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *qv = (double *)malloc(sizeof(double) * head_dim);
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    if (gather_rows(k_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, K) ||
        gather_rows(v_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, V)) {
      bad = 1;
    } else {
      for (int g = 0; g < group; ++g) {
        int h = kvh * group + g;
        const uint16_t *qsrc = q + ((int64_t)s * num_q_heads + h) * head_dim;
        for (int c = 0; c < head_dim; ++c) qv[c] = bf16_bits_to_f64(qsrc[c]);
        double l;
        attend(qv, K, V, n, head_dim, scale, x, out + ((int64_t)s * num_q_heads + h) * head_dim, &l);
        if (lse) lse[(int64_t)s * num_q_heads + h] = l;
      }
    }
    free(K);
    free(V);
    free(x);
    free(qv);
  }
  return bad ? -1 : 0;
}

/* Decode restricted to listed (sequence, q head) pairs; used to check
 * sampled outputs of very large batches and to time a bounded sample.
 * pairs [n_pairs, 2]; out [n_pairs, D]; lse [n_pairs] (nullable).        */
int oracle_decode_pairs(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, double scale,
                        const int32_t *pairs, int n_pairs, double *out, double *lse) {
  int group = num_q_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_pairs; ++i) {
    int s = pairs[2 * i], h = pairs[2 * i + 1];
    int kvh = h / group;
    int64_t n = seq_lens[s];
    if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size) {
      bad = 1;
      continue;
    }
    double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *qv = (double *)malloc(sizeof(double) * head_dim);
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    if (gather_rows(k_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, K) ||
        gather_rows(v_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, V)) {
      bad = 1;
    } else {
      const uint16_t *qsrc = q + ((int64_t)s * num_q_heads + h) * head_dim;
      for (int c = 0; c < head_dim; ++c) qv[c] = bf16_bits_to_f64(qsrc[c]);
      double l;
      attend(qv, K, V, n, head_dim, scale, x, out + (int64_t)i * head_dim, &l);
      if (lse) lse[i] = l;
    }
    free(K);
    free(V);
    free(x);
    free(qv);
  }
  return bad ? -1 : 0;
}

/* Attention of sequence s's query for q head h over the key range [a, b)
 * only: the partial result of one split of the keys.  out [D], lse [1].   */
int oracle_attend_range(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq, int s, int h,
                        int64_t a, int64_t b, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, double scale,
                        double *out, double *lse) {
  int group = num_q_heads / num_kv_heads;
  int kvh = h / group;
  if (a < 0 || b < a || b > (int64_t)max_blocks_per_seq * block_size) return -1;
  int64_t n = b - a;
  double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
  double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
  double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double *qv = (double *)malloc(sizeof(double) * head_dim);
  const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
  int rc = 0;
  if (gather_rows(k_cache, row, kvh, a, b, num_kv_heads, head_dim, block_size, num_blocks, K) ||
      gather_rows(v_cache, row, kvh, a, b, num_kv_heads, head_dim, block_size, num_blocks, V)) {
    rc = -1;
  } else {
    const uint16_t *qsrc = q + ((int64_t)s * num_q_heads + h) * head_dim;
    for (int c = 0; c < head_dim; ++c) qv[c] = bf16_bits_to_f64(qsrc[c]);
    attend(qv, K, V, n, head_dim, scale, x, out, lse);
  }
  free(K);
  free(V);
  free(x);
  free(qv);
  return rc;
}

/* ---------------------------------------------------------------------- */
/* Log-sum-exp merge of partial attentions.                                */
/* part_o [S, Hq, P_max, D], part_lse [S, Hq, P_max], num_parts [S]:       */
/*   L = max_p lse_p, w_p = exp(lse_p - L),                                */
/*   out = sum_p w_p o_p / sum_p w_p,  lse = L + ln(sum_p w_p).            */
/* A part with lse = -inf carries no keys and has weight 0.                */
/* ---------------------------------------------------------------------- */
int oracle_merge(const double *part_o, const double *part_lse, const int32_t *num_parts,
                 int num_seqs, int num_q_heads, int head_dim, int max_parts, double *out,
                 double *lse) {
  for (int s = 0; s < num_seqs; ++s) {
    int np = num_parts[s];
    if (np < 0 || np > max_parts) return -1;
    for (int h = 0; h < num_q_heads; ++h) {
      const double *lp = part_lse + ((int64_t)s * num_q_heads + h) * max_parts;
      const double *op = part_o + ((int64_t)s * num_q_heads + h) * max_parts * head_dim;
      double *o = out + ((int64_t)s * num_q_heads + h) * head_dim;
      double L = -INFINITY;
      for (int p = 0; p < np; ++p)
        if (lp[p] > L) L = lp[p];
      for (int c = 0; c < head_dim; ++c) o[c] = 0.0;
      if (L == -INFINITY) {
        if (lse) lse[(int64_t)s * num_q_heads + h] = -INFINITY;
        continue;
      }
      double wsum = 0.0;
      for (int p = 0; p < np; ++p) {
        double w = exp(lp[p] - L);
        wsum += w;
        for (int c = 0; c < head_dim; ++c) o[c] += w * op[(int64_t)p * head_dim + c];
      }
      for (int c = 0; c < head_dim; ++c) o[c] /= wsum;
      if (lse) lse[(int64_t)s * num_q_heads + h] = L + log(wsum);
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Causal prefill chunks.  Chunk c owns query rows [cu_q_lens[c],          */
/* cu_q_lens[c+1]) of q [Tq, Hq, D]; row i of the chunk sits at absolute   */
/* position p = q_start_pos[c] + i and attends over keys 0..p of the       */
/* chunk's sequence (block table row c), which holds seq_lens[c] tokens.   */
/* out [Tq, Hq, D] fp64, lse [Tq, Hq] fp64 (nullable).                     */
/* ---------------------------------------------------------------------- */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *cu_q_lens, const int32_t *q_start_pos,
                   const int32_t *seq_lens, int num_chunks, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                   double scale, double *out, double *lse) {
  int group = num_q_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t pair = 0; pair < (int64_t)num_chunks * num_kv_heads; ++pair) {
    int c = (int)(pair / num_kv_heads), kvh = (int)(pair % num_kv_heads);
    int64_t n = seq_lens[c];
    int64_t q0 = cu_q_lens[c], q1 = cu_q_lens[c + 1];
    int64_t p0 = q_start_pos[c];
    if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size || q1 < q0 || p0 < 0 ||
        p0 + (q1 - q0) > n) {
      bad = 1;
      continue;
    }
    double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *qv = (double *)malloc(sizeof(double) * head_dim);
    const int32_t *row = block_tables + (int64_t)c * max_blocks_per_seq;
    if (gather_rows(k_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, K) ||
        gather_rows(v_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks, V)) {
      bad = 1;
    } else {
      for (int64_t t = q0; t < q1; ++t) {
        int64_t p = p0 + (t - q0); /* keys 0..p are visible */
        for (int g = 0; g < group; ++g) {
          int h = kvh * group + g;
          const uint16_t *qsrc = q + (t * num_q_heads + h) * head_dim;
          for (int cc = 0; cc < head_dim; ++cc) qv[cc] = bf16_bits_to_f64(qsrc[cc]);
          double l;
          attend(qv, K, V, p + 1, head_dim, scale, x, out + (t * num_q_heads + h) * head_dim, &l);
          if (lse) lse[t * num_q_heads + h] = l;
        }
      }
    }
    free(K);
    free(V);
    free(x);
    free(qv);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------- */
/* FP8 (E4M3) KV cache: both engines ship FP8 KV caches with per-tensor or  */
/* per-head scales ("The LLM inference engine playbook", Theme 3, shrinking */
/* the cache).  E4M3 as the format defines it: a sign bit, 4 exponent bits  */
/* (bias 7) and 3 mantissa bits; exponent field 0 holds subnormals m*2^-9;  */
/* no infinity; 0x7F and 0xFF are NaN; the largest finite magnitude is      */
/* (1 + 6/8) * 2^8 = 448.                                                   */
/* ---------------------------------------------------------------------- */
double oracle_e4m3_value(uint8_t code) {
  int e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e - 7) */
  return (code & 0x80) ? -v : v;
}

/* The E4M3 code nearest to v, ties to the even code (even mantissa);
 * magnitudes of 448 and above (infinity included) give +-448; NaN gives 0x7F.
 * Below 2^-6 the grid has step 2^-9 (codes 0..8 are code * 2^-9); in
 * [2^k, 2^(k+1)) it has step 2^(k-3), and a rounding up to 2^(k+1) carries
 * into the exponent field. */
int oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  int sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int code;
  if (a < ldexp(1.0, -6)) {
    code = (int)nearbyint(a * 512.0); /* exact scaling; round half to even */
  } else {
    int k;
    frexp(a, &k);
    k -= 1; /* a in [2^k, 2^(k+1)) */
    double q = nearbyint(ldexp(a, 3 - k)); /* in [8, 16] */
    code = ((k + 7) << 3) + (int)q - 8;
  }
  if (code > 0x7E) code = 0x7E;
  return sign | code;
}

/* Quantizing scatter: code = E4M3(x / scale[h]), the division in IEEE fp32. */
int oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value,
                                 int64_t key_token_stride, int64_t value_token_stride,
                                 uint8_t *k_cache, uint8_t *v_cache, const int64_t *slot_mapping,
                                 const float *k_scales, const float *v_scales, int num_tokens,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int64_t num_blocks) {
  int bad = 0;
  /* tokens in parallel: valid slots are distinct, so no two write one byte */
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) {
      bad = 1;
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int c = 0; c < head_dim; ++c) {
        int64_t dst = (slot * num_kv_heads + h) * (int64_t)head_dim + c;
        float xk = (float)bf16_bits_to_f64(key[(int64_t)t * key_token_stride + (int64_t)h * head_dim + c]);
        float xv = (float)bf16_bits_to_f64(value[(int64_t)t * value_token_stride + (int64_t)h * head_dim + c]);
        float rk = xk / k_scales[h];
        float rv = xv / v_scales[h];
        k_cache[dst] = (uint8_t)oracle_e4m3_encode(rk);
        v_cache[dst] = (uint8_t)oracle_e4m3_encode(rv);
      }
    }
  }
  return bad ? -1 : 0;
}

/* Gather with dequantization: rows of value(code) * scale, in fp64 (exact). */
static int gather_rows_e4m3(const uint8_t *cache, const int32_t *table_row, int kvh, int64_t a,
                            int64_t b, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, double scale, double *rows) {
  for (int64_t j = a; j < b; ++j) {
    int64_t blk = table_row[j / block_size];
    int64_t off = j % block_size;
    if (blk < 0 || blk >= num_blocks) return -1;
    const uint8_t *src = cache + ((blk * block_size + off) * num_kv_heads + kvh) * (int64_t)head_dim;
    for (int c = 0; c < head_dim; ++c) rows[(j - a) * head_dim + c] = oracle_e4m3_value(src[c]) * scale;
  }
  return 0;
}

/* Decode over E4M3 pools: the decode definition on the dequantized cache. */
int oracle_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                      const float *k_scales, const float *v_scales,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, double scale,
                      double *out, double *lse) {
  int group = num_q_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t pair = 0; pair < (int64_t)num_seqs * num_kv_heads; ++pair) {
    int s = (int)(pair / num_kv_heads), kvh = (int)(pair % num_kv_heads);
    int64_t n = seq_lens[s];
    if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size) {
      bad = 1;
      continue;
    }
    double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * head_dim);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *qv = (double *)malloc(sizeof(double) * head_dim);
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    if (gather_rows_e4m3(k_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks,
                         (double)k_scales[kvh], K) ||
        gather_rows_e4m3(v_cache, row, kvh, 0, n, num_kv_heads, head_dim, block_size, num_blocks,
                         (double)v_scales[kvh], V)) {
      bad = 1;
    } else {
      for (int g = 0; g < group; ++g) {
        int h = kvh * group + g;
        const uint16_t *qsrc = q + ((int64_t)s * num_q_heads + h) * head_dim;
        for (int c = 0; c < head_dim; ++c) qv[c] = bf16_bits_to_f64(qsrc[c]);
        double l;
        attend(qv, K, V, n, head_dim, scale, x, out + ((int64_t)s * num_q_heads + h) * head_dim, &l);
        if (lse) lse[(int64_t)s * num_q_heads + h] = l;
      }
    }
    free(K);
    free(V);
    free(x);
    free(qv);
  }
  return bad ? -1 : 0;
}

/* Threads the OpenMP runtime will use (reported beside CPU timings). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) { omp_set_num_threads(n); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
