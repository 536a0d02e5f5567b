/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library; it reads the same documented memory layout and nothing else.
 *
 * What it computes is the plain definition of attention over a block-paged
 * KV cache:
 *   - "Block-Paged KV Cache (FP8/FP16)" -- figure "vllm.cpp ARCHITECTURE
 *     OVERVIEW" of "Building and Deploying vllm.cpp ..." (the sigmablogger
 *     build/deploy walkthrough); block size 16 from its "Step 4: Serving Qwen"
 *     launch commands (--block-size 16).
 *   - "paged attention (block-paged KV cache)" and "chunked prefill" -- section
 *     "What's implemented (CPU, behaviorally tested)" of the "vllm.cpp"
 *     repository listing (Engine core and Model forward bullets).
 *   - fp8 pages of one byte per element, E4M3 or E5M2 -- table in "2. CLI
 *     Configuration Parameters" (--kv-cache-dtype) and the table in "Step 6:
 *     Status of TurboQuant Support" of the walkthrough (its vllm.cpp row names
 *     E4M3/E5M2 block-paged KV allocation).
 *   - a prefix-cache hit binds a new sequence's block table to existing
 *     physical pages -- "1. Technical Mechanics of the Radix Cache" (Zero-Copy
 *     Cache Hits) of the walkthrough.
 * The pages give no formula; the oracle is softmax(scale * q K^T) V with an
 * explicit gather through the block table, written out in fp64.
 *
 * Layout (the reading this build takes where the pages are silent):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *                      bf16 or fp16 bit patterns (uint16), or E4M3 / E5M2
 *                      bytes (uint8)
 *   q, new k / v rows: [tokens][heads][head_dim] bf16 bit patterns; fp16 bit
 *                      patterns with an fp16 cache (the cache of an fp16
 *                      model, whose activations are fp16 too)
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]
 *   context_lens     : int32 [num_seqs], KV tokens including this step's
 *   slot_mapping     : int64 [tokens], slot = block * block_size + offset, <0 skip
 *   query head h reads kv head h / (num_q_heads / num_kv_heads)
 *
 * Parity pins: every function here is pinned by tests that do not reuse its
 * code (brute-force dense attention through torch's CPU SDPA, closed forms,
 * invariants, torch's float8_e4m3fn and float8_e5m2 codecs); see
 * tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KV_BF16 0
#define KV_FP8_E4M3 1
#define KV_FP8_E5M2 2
#define KV_F16 3

/* scales apply to the 8-bit formats only */
static int kv_is_8bit(int kv_dtype) { return kv_dtype == KV_FP8_E4M3 || kv_dtype == KV_FP8_E5M2; }

/* ---------------------------------------------------------------- bf16 */

/* bf16 is the upper 16 bits of an IEEE binary32: widening is exact. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------------- fp16 */

/*
 * IEEE 754 binary16: 1 sign bit, 5 exponent bits with bias 15, 10 mantissa
 * bits.  Exponent field 0 encodes subnormals m/1024 * 2^-14; exponent 31
 * encodes infinity (m = 0) and NaN (m != 0); otherwise (1 + m/1024) *
 * 2^(e - 15).  Every value is exact in double.
 */
double pa_oracle_f16_decode(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 10) & 31;
  int m = b & 1023;
  double v;
  if (e == 31)
    v = m ? NAN : INFINITY;
  else if (e == 0)
    v = ldexp((double)m, -24);
  else
    v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* The value of every fp16 code, filled once from pa_oracle_f16_decode. */
static double f16_value[65536];
static int f16_value_ready;

static void f16_table_init(void) {
  if (f16_value_ready) return;
  for (int c = 0; c < 65536; ++c) f16_value[c] = pa_oracle_f16_decode((uint16_t)c);
  f16_value_ready = 1;
}

/* A query or new-row element: fp16 bits with an fp16 cache, bf16 bits otherwise. */
static double act_to_double(int kv_dtype, uint16_t b) {
  if (kv_dtype == KV_F16) {
    f16_table_init();
    return f16_value[b];
  }
  return bf16_bits_to_double(b);
}

/* ---------------------------------------------------------------- E4M3 */

/*
 * OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  No infinities; exponent 1111 with mantissa 111 is
 * NaN (bytes 0x7F and 0xFF); every other pattern is finite.  Exponent field 0
 * encodes subnormals m/8 * 2^(1-7).
 */
double pa_oracle_e4m3_decode(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* All 256 codes decoded once (the same definition, cached for speed). */
static double e4m3_value[256];
static int e4m3_value_ready = 0;

static void e4m3_table_init(void) {
  if (e4m3_value_ready) return;
  for (int c = 0; c < 256; ++c) e4m3_value[c] = pa_oracle_e4m3_decode((uint8_t)c);
  e4m3_value_ready = 1;
}

/*
 * Round-to-nearest-even with saturation to the largest finite magnitude
 * (448), NaN -> 0x7F.  Chosen the plainest way: search all 127 non-negative
 * finite codes for the nearest value; on a tie take the code whose mantissa
 * is even (codes are monotone in value, so that is the even code).
 */
uint8_t pa_oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  e4m3_table_init();
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  /* saturation: everything at or beyond the largest finite value, +-inf
     included, maps to +-448 (a distance search cannot decide this once
     |x| dwarfs 448 in fp64) */
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double v = e4m3_value[c];
    double err = fabs(a - v);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------- E5M2 */

/*
 * OCP 8-bit floating point, E5M2 variant: 1 sign bit, 5 exponent bits with
 * bias 15, 2 mantissa bits, IEEE-style specials: exponent 11111 is +-inf
 * (mantissa 0) or NaN (mantissa != 0).  Exponent field 0 encodes subnormals
 * m/4 * 2^(1-15).  Largest finite magnitude 1.75 * 2^15 = 57344.
 */
double pa_oracle_e5m2_decode(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 2) & 0x1F;
  int m = byte & 0x3;
  double v;
  if (e == 0x1F) {
    if (m != 0) return NAN;
    v = INFINITY;
  } else if (e == 0) {
    v = ldexp((double)m / 4.0, 1 - 15);
  } else {
    v = ldexp(1.0 + (double)m / 4.0, e - 15);
  }
  return sign ? -v : v;
}

static double e5m2_value[256];
static int e5m2_value_ready = 0;

static void e5m2_table_init(void) {
  if (e5m2_value_ready) return;
  for (int c = 0; c < 256; ++c) e5m2_value[c] = pa_oracle_e5m2_decode((uint8_t)c);
  e5m2_value_ready = 1;
}

/*
 * Round-to-nearest-even onto the finite E5M2 values with saturation to the
 * largest finite magnitude (57344; +-inf saturates too), NaN -> 0x7F: the same
 * plain nearest-code search as for E4M3, over the 124 non-negative finite
 * codes 0x00 .. 0x7B.
 */
uint8_t pa_oracle_e5m2_encode(double x) {
  if (isnan(x)) return 0x7F;
  e5m2_table_init();
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 57344.0) return (uint8_t)(sign | 0x7B);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7B; ++c) {
    double v = e5m2_value[c];
    double err = fabs(a - v);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* Element (t, d) of one kv head, decoded to a real number (scale applied). */
static double kv_elem(int kv_dtype, const void *cache, int64_t row_index, int head_dim, int d,
                      double scale) {
  if (kv_dtype == KV_BF16) {
    const uint16_t *c = (const uint16_t *)cache;
    return bf16_bits_to_double(c[row_index * head_dim + d]);
  }
  if (kv_dtype == KV_F16) {
    const uint16_t *c = (const uint16_t *)cache;
    f16_table_init();
    return f16_value[c[row_index * head_dim + d]];
  }
  const uint8_t *c = (const uint8_t *)cache;
  if (kv_dtype == KV_FP8_E5M2) {
    e5m2_table_init();
    return e5m2_value[c[row_index * head_dim + d]] * scale;
  }
  e4m3_table_init();
  return e4m3_value[c[row_index * head_dim + d]] * scale;
}

/* Row index of logical token t of kv head kh for a sequence's block table. */
static int64_t cache_row(const int32_t *table_row, int block_size, int num_kv_heads, int kh, int t) {
  int64_t blk = table_row[t / block_size];
  int off = t % block_size;
  return (blk * num_kv_heads + kh) * block_size + off;
}

/* ---------------------------------------------------------- cache write */

/*
 * The 8-bit code of one bf16 input x under one scale: e4m3 / e5m2 of
 * fl32(fl32(x) / scale).
 */
static uint8_t encode_bf16(int kv_dtype, uint16_t x, float scale) {
  float q = bf16_bits_to_float(x) / scale;
  return kv_dtype == KV_FP8_E5M2 ? pa_oracle_e5m2_encode((double)q) : pa_oracle_e4m3_encode((double)q);
}

/*
 * The code depends only on the 16 input bits and the scale, so a large write
 * encodes each distinct (input, scale) once and looks the rest up: a memo of
 * encode_bf16, filled lazily, valid for one (format, scale) at a time.  It
 * changes how often the search runs, not what it returns.
 */
typedef struct {
  int kv_dtype;
  float scale;
  uint8_t code[65536];
  uint8_t done[65536];
} encode_memo;

static void memo_reset(encode_memo *m, int kv_dtype, float scale) {
  m->kv_dtype = kv_dtype;
  m->scale = scale;
  memset(m->done, 0, sizeof m->done);
}

static uint8_t memo_encode(encode_memo *m, uint16_t x) {
  if (!m->done[x]) {
    m->code[x] = encode_bf16(m->kv_dtype, x, m->scale);
    m->done[x] = 1;
  }
  return m->code[x];
}

/*
 * For each token i with slot_mapping[i] >= 0: block = slot / block_size,
 * offset = slot % block_size, and for every kv head h the cache row
 * (block, h, offset) receives enc(k[i][h][:]) (same for v).
 * enc = bit copy for bf16 and fp16 (the rows arrive in the cache's own
 * type); for E4M3 / E5M2, enc(x) = e4m3 / e5m2 of fl32(fl32(x) / scale),
 * scale being kv head h's entry of k_scales / v_scales when those are given
 * (per-head scales), else the per-tensor k_scale / v_scale.
 */
void pa_oracle_cache_write(int kv_dtype, int block_size, int num_kv_heads, int head_dim,
                           const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                           int num_tokens, float k_scale, float v_scale, const float *k_scales,
                           const float *v_scales, void *k_cache, void *v_cache) {
  encode_memo *km = NULL, *vm = NULL;
  if (kv_is_8bit(kv_dtype)) {
    /* one memo per kv head and tensor (per-head scales differ by head) */
    km = (encode_memo *)malloc(sizeof(encode_memo) * (size_t)num_kv_heads);
    vm = (encode_memo *)malloc(sizeof(encode_memo) * (size_t)num_kv_heads);
    for (int h = 0; h < num_kv_heads; ++h) {
      memo_reset(&km[h], kv_dtype, k_scales ? k_scales[h] : k_scale);
      memo_reset(&vm[h], kv_dtype, v_scales ? v_scales[h] : v_scale);
    }
  }
  for (int i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t blk = slot / block_size;
    int64_t off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      int64_t dst_row = (blk * num_kv_heads + h) * block_size + off;
      const uint16_t *ks = k + ((int64_t)i * num_kv_heads + h) * head_dim;
      const uint16_t *vs = v + ((int64_t)i * num_kv_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        if (!kv_is_8bit(kv_dtype)) {
          ((uint16_t *)k_cache)[dst_row * head_dim + d] = ks[d];
          ((uint16_t *)v_cache)[dst_row * head_dim + d] = vs[d];
        } else {
          ((uint8_t *)k_cache)[dst_row * head_dim + d] = memo_encode(&km[h], ks[d]);
          ((uint8_t *)v_cache)[dst_row * head_dim + d] = memo_encode(&vm[h], vs[d]);
        }
      }
    }
  }
  free(km);
  free(vm);
}

/* ----------------------------------------------------- one attention row */

/*
 * Attention of one query vector over the logical key range [t_begin, t_end)
 * of one sequence and one kv head:
 *   x_t = scale * sum_d q[d] K_t[d]
 *   m = max_t x_t,  l = sum_t exp(x_t - m)
 *   out = sum_t exp(x_t - m) V_t / l,   lse = m + ln l
 * An empty range gives out = 0 and lse = -inf.
 */
void pa_oracle_attend_range(int kv_dtype, int block_size, int num_kv_heads, int head_dim,
                            const uint16_t *q_vec, const void *k_cache, const void *v_cache,
                            const int32_t *table_row, int kh, int t_begin, int t_end,
                            float scale, float k_scale, float v_scale, double *out, double *lse) {
  int n = t_end - t_begin;
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n <= 0) {
    *lse = -INFINITY;
    return;
  }
  double ks = kv_is_8bit(kv_dtype) ? (double)k_scale : 1.0;
  double vs = kv_is_8bit(kv_dtype) ? (double)v_scale : 1.0;
  double *x = (double *)malloc(sizeof(double) * (size_t)n);
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    int64_t row = cache_row(table_row, block_size, num_kv_heads, kh, t_begin + j);
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d)
      dot += act_to_double(kv_dtype, q_vec[d]) * kv_elem(kv_dtype, k_cache, row, head_dim, d, ks);
    x[j] = (double)scale * dot;
    if (x[j] > m) m = x[j];
  }
  double l = 0.0;
  for (int j = 0; j < n; ++j) {
    double p = exp(x[j] - m);
    l += p;
    int64_t row = cache_row(table_row, block_size, num_kv_heads, kh, t_begin + j);
    for (int d = 0; d < head_dim; ++d)
      out[d] += p * kv_elem(kv_dtype, v_cache, row, head_dim, d, vs);
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= l;
  *lse = m + log(l);
  free(x);
}

/* ------------------------------------------------------- local attention */

/*
 * First key a query at position pos may attend ("Local-attention KV +
 * sliding-window operator -- SlidingWindowSpec and ChunkedLocalAttentionSpec"
 * of the vllm.cpp repository listing; the pages give no formula, the plain
 * readings are taken): a sliding window of W keys ending at pos starts at
 * pos - W + 1; chunked-local attention with chunks of C positions starts at
 * the query's chunk, floor(pos / C) * C.  0 disables either; with both the
 * later start applies.
 */
static int local_first_key(int pos, int window, int chunk) {
  int lo = 0;
  if (window > 0 && pos - window + 1 > lo) lo = pos - window + 1;
  if (chunk > 0 && (pos / chunk) * chunk > lo) lo = (pos / chunk) * chunk;
  return lo;
}

/* ---------------------------------------------------------------- decode */

/*
 * Decode: sequence s has one new query (q[s]) at position L_s - 1 and attends
 * every cached token [0, L_s) through its block table.  Query head h uses kv
 * head h / g with g = num_q_heads / num_kv_heads.
 *
 * With a sliding window or chunked-local attention the range starts at
 * local_first_key(L_s - 1).
 *
 * pairs: optional int32 [num_pairs][2] list of (s, h) to compute (NULL = all,
 * in (s, h) row-major order).  out: [num_pairs][head_dim], lse: [num_pairs].
 */
void pa_oracle_decode(int kv_dtype, int block_size, int num_kv_heads, int num_q_heads,
                      int head_dim, const uint16_t *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, float scale, float k_scale,
                      float v_scale, const float *k_scales, const float *v_scales, int window,
                      int chunk, const int32_t *pairs, int num_pairs, double *out, double *lse) {
  int g = num_q_heads / num_kv_heads;
  int total = pairs ? num_pairs : num_seqs * num_q_heads;
  for (int i = 0; i < total; ++i) {
    int s = pairs ? pairs[2 * i] : i / num_q_heads;
    int h = pairs ? pairs[2 * i + 1] : i % num_q_heads;
    const uint16_t *q_vec = q + ((int64_t)s * num_q_heads + h) * head_dim;
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    int L = context_lens[s];
    int lo = L > 0 ? local_first_key(L - 1, window, chunk) : 0;
    pa_oracle_attend_range(kv_dtype, block_size, num_kv_heads, head_dim, q_vec, k_cache, v_cache,
                           row, h / g, lo, L, scale, k_scales ? k_scales[h / g] : k_scale,
                           v_scales ? v_scales[h / g] : v_scale, out + (int64_t)i * head_dim, lse + i);
  }
}

/* --------------------------------------------------------------- prefill */

/*
 * Chunked prefill: sequence s owns the packed query rows
 * [query_start_loc[s], query_start_loc[s+1]); q_len = their count.  Its KV
 * already holds L_s tokens (the chunk's own K/V were written before), so query
 * i sits at position L_s - q_len + i and attends keys [0, position] (causal),
 * or [local_first_key(position), position] with local attention.
 *
 * pairs: optional int32 [num_pairs][2] list of (token row, q head) (NULL = all
 * rows x heads).  out: [num_pairs][head_dim], lse: [num_pairs].
 */
void pa_oracle_prefill(int kv_dtype, int block_size, int num_kv_heads, int num_q_heads,
                       int head_dim, const uint16_t *q, const int32_t *query_start_loc,
                       const void *k_cache, const void *v_cache, const int32_t *block_tables,
                       int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                       float scale, float k_scale, float v_scale, const float *k_scales,
                       const float *v_scales, int window, int chunk, const int32_t *pairs,
                       int num_pairs, double *out, double *lse) {
  int g = num_q_heads / num_kv_heads;
  int num_rows = query_start_loc[num_seqs];
  int total = pairs ? num_pairs : num_rows * num_q_heads;
  for (int i = 0; i < total; ++i) {
    int r = pairs ? pairs[2 * i] : i / num_q_heads;
    int h = pairs ? pairs[2 * i + 1] : i % num_q_heads;
    int s = 0;
    while (s + 1 <= num_seqs && query_start_loc[s + 1] <= r) ++s;
    int q_len = query_start_loc[s + 1] - query_start_loc[s];
    int pos = context_lens[s] - q_len + (r - query_start_loc[s]);
    const uint16_t *q_vec = q + ((int64_t)r * num_q_heads + h) * head_dim;
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    pa_oracle_attend_range(kv_dtype, block_size, num_kv_heads, head_dim, q_vec, k_cache, v_cache,
                           row, h / g, local_first_key(pos, window, chunk), pos + 1, scale,
                           k_scales ? k_scales[h / g] : k_scale, v_scales ? v_scales[h / g] : v_scale,
                           out + (int64_t)i * head_dim, lse + i);
  }
}

/* ------------------------------------------------ shared-prefix (cascade) */

/*
 * Attention of groups of queries over a shared prefix (cascade attention:
 * the pages a prefix-cache hit binds to several sequences -- "Zero-Copy Cache
 * Hits" of "1. Technical Mechanics of the Radix Cache" -- attended once for
 * all of them; the result is merged with each sequence's own suffix by the
 * log-sum-exp merge below).  Group j owns the packed query rows
 * [query_start_loc[j], query_start_loc[j+1]) and the prefix of prefix_lens[j]
 * tokens behind block_tables[j]; every query of the group attends all of it
 * (the queries come after the prefix, so no causal mask applies inside it).
 * pairs: optional (row, q head) list as in prefill.
 */
void pa_oracle_prefix(int kv_dtype, int block_size, int num_kv_heads, int num_q_heads, int head_dim,
                      const uint16_t *q, const int32_t *query_start_loc, const void *k_cache,
                      const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *prefix_lens, int num_groups, float scale, float k_scale,
                      float v_scale, const float *k_scales, const float *v_scales,
                      const int32_t *pairs, int num_pairs, double *out, double *lse) {
  int g = num_q_heads / num_kv_heads;
  int num_rows = query_start_loc[num_groups];
  int total = pairs ? num_pairs : num_rows * num_q_heads;
  for (int i = 0; i < total; ++i) {
    int r = pairs ? pairs[2 * i] : i / num_q_heads;
    int h = pairs ? pairs[2 * i + 1] : i % num_q_heads;
    int j = 0;
    while (j + 1 <= num_groups && query_start_loc[j + 1] <= r) ++j;
    const uint16_t *q_vec = q + ((int64_t)r * num_q_heads + h) * head_dim;
    const int32_t *row = block_tables + (int64_t)j * max_blocks_per_seq;
    pa_oracle_attend_range(kv_dtype, block_size, num_kv_heads, head_dim, q_vec, k_cache, v_cache,
                           row, h / g, 0, prefix_lens[j], scale, k_scales ? k_scales[h / g] : k_scale,
                           v_scales ? v_scales[h / g] : v_scale, out + (int64_t)i * head_dim, lse + i);
  }
}

/* ----------------------------------------------------------- block copies */

/*
 * Copy-on-write of whole pages: for every pair i, block dst_blocks[i] of both
 * caches receives the contents of block src_blocks[i] (all kv heads, all
 * slots), so that a sequence about to write into a page it shares with others
 * (the partly filled last page of a prefix-cache hit) gets a private copy.
 * elem_bytes: 2 for bf16 / fp16, 1 for the 8-bit formats.
 */
void pa_oracle_copy_blocks(int elem_bytes, int block_size, int num_kv_heads, int head_dim,
                           const int32_t *src_blocks, const int32_t *dst_blocks, int num_pairs,
                           void *k_cache, void *v_cache) {
  int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_dim * elem_bytes;
  for (int i = 0; i < num_pairs; ++i) {
    memcpy((char *)k_cache + dst_blocks[i] * block_bytes, (char *)k_cache + src_blocks[i] * block_bytes,
           (size_t)block_bytes);
    memcpy((char *)v_cache + dst_blocks[i] * block_bytes, (char *)v_cache + src_blocks[i] * block_bytes,
           (size_t)block_bytes);
  }
}

/* ------------------------------------------ prefix-cache page bookkeeping */

/*
 * Zero-copy cache hit ("Zero-Copy Cache Hits" of "1. Technical Mechanics of
 * the Radix Cache"): the engine binds a new sequence's block table directly
 * to the physical pages its matched prefix already occupies, and each bound
 * page gains one owner.  For every i < num_seqs, with row = seq_rows[i] and
 * the hit's pages hit_blocks[hit_start[i] .. hit_start[i+1]):
 *   block_tables[row][j] = hit_blocks[hit_start[i] + j]   for each j,
 *   refcounts[that page] += 1.
 * A page outside [0, num_blocks) is not bound (counted in *errors).
 */
void pa_oracle_bind_blocks(int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_rows,
                           const int32_t *hit_start, const int32_t *hit_blocks, int num_seqs, int32_t *refcounts,
                           int num_blocks, int32_t *errors) {
  for (int i = 0; i < num_seqs; ++i) {
    int32_t *row = block_tables + (int64_t)seq_rows[i] * max_blocks_per_seq;
    for (int j = 0; j < hit_start[i + 1] - hit_start[i]; ++j) {
      int32_t blk = hit_blocks[hit_start[i] + j];
      if (blk < 0 || blk >= num_blocks) {
        ++*errors;
        continue;
      }
      row[j] = blk;
      refcounts[blk] += 1;
    }
  }
}

/*
 * Release ("LRU Eviction": dropped entries return their memory blocks to
 * the global page pool).  Each of the first block_counts[i] pages of table
 * row seq_rows[i] loses one owner and its table entry becomes -1; a page
 * whose owner count reaches zero goes back to the pool: it is appended to
 * free_list at free_count, which grows by one.  (A finished sequence
 * releases its own row; an evicted cache entry passes its pages as a row.)
 * A page with no owner left, or outside [0, num_blocks), is left as it is
 * (counted in *errors).  The order of the free list follows the pages in
 * row-major order here; any order of the same pages is as valid.
 */
void pa_oracle_release_blocks(int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_rows,
                              const int32_t *block_counts, int num_seqs, int32_t *refcounts, int num_blocks,
                              int32_t *free_list, int32_t *free_count, int32_t *errors) {
  for (int i = 0; i < num_seqs; ++i) {
    int32_t *row = block_tables + (int64_t)seq_rows[i] * max_blocks_per_seq;
    for (int j = 0; j < block_counts[i]; ++j) {
      int32_t blk = row[j];
      if (blk < 0 || blk >= num_blocks || refcounts[blk] <= 0) {
        ++*errors;
        continue;
      }
      row[j] = -1;
      refcounts[blk] -= 1;
      if (refcounts[blk] == 0) free_list[(*free_count)++] = blk;
    }
  }
}

/* ----------------------------------------------------------------- merge */

/*
 * Merge of attention results over disjoint key ranges (log-sum-exp
 * weighting): M = max_p lse_p, w_p = exp(lse_p - M),
 * out = sum_p w_p o_p / sum_p w_p, lse = M + ln sum_p w_p.  Parts with
 * lse = -inf carry no keys and drop out; if every part is empty the result is
 * out = 0, lse = -inf.
 * part_o: [num_parts][head_dim], part_lse: [num_parts].
 */
void pa_oracle_merge(const double *part_o, const double *part_lse, int num_parts, int head_dim,
                     double *out, double *lse) {
  double M = -INFINITY;
  for (int p = 0; p < num_parts; ++p)
    if (part_lse[p] > M) M = part_lse[p];
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (M == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double wsum = 0.0;
  for (int p = 0; p < num_parts; ++p) {
    if (part_lse[p] == -INFINITY) continue;
    double w = exp(part_lse[p] - M);
    wsum += w;
    for (int d = 0; d < head_dim; ++d) out[d] += w * part_o[(int64_t)p * head_dim + d];
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= wsum;
  *lse = M + log(wsum);
}
