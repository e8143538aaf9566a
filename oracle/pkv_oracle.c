/*
 * pkv_oracle.c -- float64 CPU oracle for paged KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  The product path
 * (the CUDA library) shares nothing with it: no headers, no helpers, no
 * constants.  It is deliberately slow and obvious: every loop below is the
 * plain definition of what it computes, with no blocking, fusion or
 * reordering.
 *
 * What it computes, and where the definition comes from:
 *
 *  - oracle_kv_append: the in-place cache write of a static KV cache
 *    ("Inference part 1", brunomaga, section "KV cache": a static cache
 *    writes each new entry in place; "Inference part 2", section on the
 *    static cache and CUDA graphs, class GPTlite_StaticCache; "Efficient
 *    Inference", obvix, the in-place slice write of the KV cache), in its
 *    paged form: a slot s names row s % block_size of physical block
 *    s / block_size ("Inference part 1", section "PagedAttention: memory
 *    management for the KV cache"; "KV cache, prefill va decode",
 *    truongducdung, section 05, "Block table").
 *
 *  - oracle_paged_attention: softmax(q K^T * scale) V per sequence, query
 *    row and query head ("Inference part 1", section "Why attention
 *    matters", the attention equation), where
 *      * the keys and values of sequence b are read row by row through the
 *        block table: logical row i lives in physical block
 *        block_table[b][i / block_size], row i % block_size (section
 *        "PagedAttention" of "Inference part 1"; "Efficient Inference",
 *        the block-table diagram);
 *      * query head h reads KV head h / (Hq / Hkv): consecutive query heads
 *        share one KV head ("Inference part 1", section "Smaller KV
 *        caches: MQA, GQA and MLA", MultiHeadAttention_GQA with
 *        repeat_interleave; "Efficient Inference", gqa_forward);
 *      * with Q new query rows per sequence, query row j sees the cached
 *        rows and the new rows up to itself: row i is visible iff
 *        i <= L - Q + j, the shifted causal mask tril(diagonal = Sk - Sq)
 *        of scaled_dot_product_attention_kv_cache ("Inference part 1",
 *        section "KV cache").  Q = 1 is plain decode; Q = K + 1 is the
 *        target pass of greedy speculative verification ("Inference part
 *        2", section "Speculative decoding", generate_speculative).
 *    The softmax is the textbook two-pass form: all scores first, then
 *    their maximum, then exp(s - max) weights.  It is NOT the online
 *    recurrence the GPU path uses.
 *
 *  - oracle_tree_attention: the same attention for the Q nodes of a
 *    candidate tree, each seeing the cached rows and its own ancestors
 *    (tree attention of Medusa, "Inference part 2", section "Medusa").
 *
 *  - oracle_kv_append_fp8 / oracle_paged_attention_fp8: the same append and
 *    attention over an FP8 E4M3 cache with one scale per tensor (see the
 *    comment above oracle_e4m3_value).
 *
 * Readings where the pages are silent (each also listed in the design
 * notes): L counts every row of the sequence including the new ones; a
 * query row that sees no row at all (L - Q + j < 0, e.g. L = 0) returns a
 * zero vector; a negative slot is skipped (padding); slots and block ids
 * out of range are errors.
 *
 * Dtype codes: 0 = float32, 1 = bfloat16, 2 = float16.  Inputs of 16-bit
 * types are passed as their raw uint16 bit patterns and widened exactly to
 * double here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_SLOT -2
#define ORACLE_ERR_BLOCK -3
#define ORACLE_ERR_NOMEM -4

static int elt_size(int dtype) { return dtype == 0 ? 4 : 2; }

/* Exact widening of one stored element to double. */
static double widen(const void *base, int64_t index, int dtype) {
  if (dtype == 0) {
    float f;
    memcpy(&f, (const char *)base + index * 4, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char *)base + index * 2, 2);
  if (dtype == 1) { /* bfloat16: the high half of a float32 */
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
  /* float16: 1 sign, 5 exponent (bias 15), 10 mantissa bits */
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/*
 * oracle_kv_append: byte copy of the new rows into their slots.
 * k_new, v_new: [T, Hkv, D]; k_cache, v_cache: [NB, Hkv, bs, D] (host
 * mirrors, modified in place); slot_mapping: [T].
 */
int oracle_kv_append(void *k_cache, void *v_cache, const void *k_new,
                     const void *v_new, const int64_t *slot_mapping, int64_t T,
                     int Hkv, int D, int bs, int64_t NB, int dtype) {
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping || T < 0 ||
      Hkv <= 0 || D <= 0 || bs <= 0 || NB < 0 || dtype < 0 || dtype > 2)
    return ORACLE_ERR_ARG;
  const int64_t row_bytes = (int64_t)D * elt_size(dtype);
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token: nothing to write */
    if (slot >= NB * bs) return ORACLE_ERR_SLOT;
    int64_t block = slot / bs, offset = slot % bs;
    for (int h = 0; h < Hkv; ++h) {
      int64_t dst = ((block * Hkv + h) * bs + offset) * row_bytes;
      int64_t src = (t * Hkv + h) * row_bytes;
      memcpy((char *)k_cache + dst, (const char *)k_new + src, row_bytes);
      memcpy((char *)v_cache + dst, (const char *)v_new + src, row_bytes);
    }
  }
  return ORACLE_OK;
}

/*
 * One output row: sequence b, query row j (0..Q-1), query head h.
 * Returns ORACLE_OK or an error code; writes D doubles to out_row.
 */
static int attend_one(double *out_row, double *scores, const void *q,
                      const void *k_cache, const void *v_cache,
                      const int32_t *block_table, int max_blocks,
                      const int32_t *context_lens, int b, int j, int h, int Q,
                      int Hq, int Hkv, int D, int bs, int64_t NB, double scale,
                      int dtype) {
  const int L = context_lens[b];
  const int64_t visible = (int64_t)L - Q + 1 + j; /* rows 0 .. L-Q+j */
  const int g = h / (Hq / Hkv);                   /* KV head of query head h */
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  if (visible <= 0) return ORACLE_OK;
  if ((visible + bs - 1) / bs > max_blocks) return ORACLE_ERR_BLOCK;

  const int64_t q_base = (((int64_t)b * Q + j) * Hq + h) * D;

  /* Pass 1: every score s_i = scale * <q, k_i>. */
  for (int64_t i = 0; i < visible; ++i) {
    int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
    if (phys < 0 || phys >= NB) return ORACLE_ERR_BLOCK;
    int64_t k_base = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += widen(q, q_base + d, dtype) * widen(k_cache, k_base + d, dtype);
    scores[i] = scale * dot;
  }
  /* Their maximum. */
  double m = scores[0];
  for (int64_t i = 1; i < visible; ++i)
    if (scores[i] > m) m = scores[i];
  /* Pass 2: weights exp(s_i - m), weighted sum of the value rows. */
  double denom = 0.0;
  for (int64_t i = 0; i < visible; ++i) {
    double w = exp(scores[i] - m);
    int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
    int64_t v_base = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
    denom += w;
    for (int d = 0; d < D; ++d) out_row[d] += w * widen(v_cache, v_base + d, dtype);
  }
  for (int d = 0; d < D; ++d) out_row[d] /= denom;
  return ORACLE_OK;
}

/*
 * oracle_paged_attention.
 *   out          [B, Q, Hq, D] float64 (written)
 *   q            [B, Q, Hq, D] in `dtype`
 *   k_cache/v_cache [NB, Hkv, bs, D] in `dtype`
 *   block_table  [B, max_blocks] int32
 *   context_lens [B] int32
 *   rows, n_rows optional list of flat output-row indices ((b*Q + j)*Hq + h)
 *                to compute; rows == NULL computes all of them.  Rows not
 *                listed are left untouched.
 * OpenMP (when compiled with it) runs independent output rows in parallel;
 * each row is computed exactly as above, so the result does not depend on
 * the thread count.
 */
int oracle_paged_attention(double *out, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *block_table,
                           int max_blocks, const int32_t *context_lens, int B,
                           int Q, int Hq, int Hkv, int D, int bs, int64_t NB,
                           double scale, int dtype, const int64_t *rows,
                           int64_t n_rows) {
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens ||
      B < 0 || Q <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 ||
      bs <= 0 || max_blocks < 0 || NB < 0 || dtype < 0 || dtype > 2)
    return ORACLE_ERR_ARG;
  const int64_t total = (int64_t)B * Q * Hq;
  const int64_t count = rows ? n_rows : total;
  int64_t max_len = 1;
  for (int b = 0; b < B; ++b)
    if (context_lens[b] > max_len) max_len = context_lens[b];
  int status = ORACLE_OK;

#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
    if (!scores) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t n = 0; n < count; ++n) {
      if (!scores) continue;
      int64_t r = rows ? rows[n] : n;
      if (r < 0 || r >= total) {
#pragma omp atomic write
        status = ORACLE_ERR_ARG;
        continue;
      }
      int h = (int)(r % Hq);
      int j = (int)((r / Hq) % Q);
      int b = (int)(r / ((int64_t)Hq * Q));
      int st = attend_one(out + r * D, scores, q, k_cache, v_cache, block_table,
                          max_blocks, context_lens, b, j, h, Q, Hq, Hkv, D, bs,
                          NB, scale, dtype);
      if (st != ORACLE_OK) {
#pragma omp atomic write
        status = st;
      }
    }
    free(scores);
  }
  return status;
}

/*
 * oracle_tree_attention: attention of Q tree nodes per sequence (Medusa-style
 * tree verification, "Inference part 2", section "Medusa": every candidate
 * of the tree is verified in one pass with a mask that lets each candidate
 * attend only to its own ancestors).  The Q nodes of sequence b occupy the
 * last Q rows L - Q .. L - 1; node j sees every cached row i < L - Q, and
 * row L - Q + k exactly when bit k of tree_mask[b * mask_stride + j] is set.
 * Q <= 64.  A node that sees no row gets zeros.  Same layouts as
 * oracle_paged_attention; two-pass softmax over the visible rows.
 */
int oracle_tree_attention(double *out, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table,
                          int max_blocks, const int32_t *context_lens, int B,
                          int Q, int Hq, int Hkv, int D, int bs, int64_t NB,
                          double scale, int dtype, const uint64_t *tree_mask,
                          int64_t mask_stride) {
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens ||
      !tree_mask || B < 0 || Q <= 0 || Q > 64 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv != 0 || D <= 0 || bs <= 0 || max_blocks < 0 || NB < 0 ||
      dtype < 0 || dtype > 2)
    return ORACLE_ERR_ARG;
  int64_t max_len = 1;
  for (int b = 0; b < B; ++b)
    if (context_lens[b] > max_len) max_len = context_lens[b];
  int status = ORACLE_OK;
  const int64_t total = (int64_t)B * Q * Hq;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
    char *seen = (char *)malloc((size_t)max_len);
    if (!scores || !seen) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < total; ++r) {
      if (!scores || !seen) continue;
      const int h = (int)(r % Hq), j = (int)((r / Hq) % Q);
      const int b = (int)(r / ((int64_t)Hq * Q));
      const int L = context_lens[b];
      const int g = h / (Hq / Hkv);
      const int64_t base = (int64_t)L - Q; /* first tree row */
      const uint64_t mask = tree_mask[(int64_t)b * mask_stride + j];
      double *o = out + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (L <= 0) continue;
      if ((L + bs - 1) / bs > max_blocks) {
#pragma omp atomic write
        status = ORACLE_ERR_BLOCK;
        continue;
      }
      const int64_t q_base = (((int64_t)b * Q + j) * Hq + h) * D;
      int any = 0, bad = 0;
      double m = 0.0;
      for (int64_t i = 0; i < L; ++i) {
        /* row i is visible if cached, or if its tree node is marked */
        seen[i] = (i < base) || ((mask >> (i - base)) & 1u);
        if (!seen[i]) continue;
        int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
        if (phys < 0 || phys >= NB) { bad = 1; break; }
        int64_t k_base = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
          dot += widen(q, q_base + d, dtype) * widen(k_cache, k_base + d, dtype);
        scores[i] = scale * dot;
        if (!any || scores[i] > m) m = scores[i];
        any = 1;
      }
      if (bad) {
#pragma omp atomic write
        status = ORACLE_ERR_BLOCK;
        continue;
      }
      if (!any) continue;
      double denom = 0.0;
      for (int64_t i = 0; i < L; ++i) {
        if (!seen[i]) continue;
        double w = exp(scores[i] - m);
        int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
        int64_t v_base = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
        denom += w;
        for (int d = 0; d < D; ++d) o[d] += w * widen(v_cache, v_base + d, dtype);
      }
      for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(scores);
    free(seen);
  }
  return status;
}

/*
 * FP8 E4M3 KV cache ("Inference part 2", section "Quantization": the format
 * table gives FP8 E4M3 as 1 sign / 4 exponent / 3 mantissa bits with largest
 * value 448, used for the KV cache; section "KV cache quantization": storing
 * the cache in FP8 halves its size and the bytes read at each decode step).
 * Reading adopted where the pages leave the scheme open: one float32 scale
 * per cache tensor, code = round-to-nearest-even(x / scale) with saturation
 * at +-448, value = code * scale; the division x / scale is the float32 one.
 *
 * The decoding below is the definition of the format: exponent bias 7,
 * exponent field 0 = subnormal (m / 8 * 2^-6), all ones with mantissa 7 =
 * NaN (there is no infinity).
 */
double oracle_e4m3_value(unsigned code) {
  const int sign = (code >> 7) & 1, e = (code >> 3) & 0xf, m = code & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9); /* m/8 * 2^-6 */
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* Nearest e4m3 code of a float32 value: round to nearest, ties to the even
 * code, saturating at the largest finite magnitude (448); NaN -> 0x7f. */
unsigned oracle_e4m3_encode(float x) {
  if (x != x) return 0x7f;
  const unsigned sign = (x < 0.0f || (x == 0.0f && signbit(x))) ? 0x80u : 0u;
  const double a = fabs((double)x);
  if (a > 448.0) return sign | 0x7eu; /* saturate at the largest finite value */
  /* the 127 non-negative finite codes, in increasing value; pick the closest
     and on a tie the one whose code is even */
  unsigned best = 0;
  double best_err = a;
  for (unsigned c = 1; c <= 0x7e; ++c) {
    const double err = fabs(oracle_e4m3_value(c) - a);
    if (err < best_err || (err == best_err && (c & 1u) == 0u)) {
      best = c;
      best_err = err;
    }
  }
  return sign | best;
}

/*
 * oracle_kv_append_fp8: quantise new rows [T, Hkv, D] (float32 values, the
 * caller widens 16-bit inputs exactly) into e4m3 codes written at their slots
 * of the byte caches [NB, Hkv, bs, D].  Negative slots are skipped.
 */
int oracle_kv_append_fp8(uint8_t *k_cache, uint8_t *v_cache, const float *k_new,
                         const float *v_new, const int64_t *slot_mapping, int64_t T,
                         int Hkv, int D, int bs, int64_t NB, float k_scale,
                         float v_scale) {
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping || T < 0 ||
      Hkv <= 0 || D <= 0 || bs <= 0 || NB < 0 || !(k_scale > 0.0f) ||
      !(v_scale > 0.0f))
    return ORACLE_ERR_ARG;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= NB * bs) return ORACLE_ERR_SLOT;
    const int64_t block = slot / bs, offset = slot % bs;
    for (int h = 0; h < Hkv; ++h)
      for (int d = 0; d < D; ++d) {
        const int64_t src = (t * Hkv + h) * D + d;
        const int64_t dst = ((block * Hkv + h) * bs + offset) * D + d;
        const float kq = k_new[src] / k_scale; /* float32 division */
        const float vq = v_new[src] / v_scale;
        k_cache[dst] = (uint8_t)oracle_e4m3_encode(kq);
        v_cache[dst] = (uint8_t)oracle_e4m3_encode(vq);
      }
  }
  return ORACLE_OK;
}

/*
 * oracle_paged_attention_fp8: oracle_paged_attention over an e4m3 cache:
 * every key element is code value * k_scale and every value element code
 * value * v_scale (exact in float64); q is in q_dtype (0 f32, 1 bf16, 2 f16).
 * Output [B, Q, Hq, D] float64.  Same masking (shifted causal) and readings.
 */
int oracle_paged_attention_fp8(double *out, const void *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, const int32_t *block_table,
                               int max_blocks, const int32_t *context_lens, int B,
                               int Q, int Hq, int Hkv, int D, int bs, int64_t NB,
                               double scale, int q_dtype, double k_scale,
                               double v_scale) {
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens ||
      B < 0 || Q <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 ||
      bs <= 0 || max_blocks < 0 || NB < 0 || q_dtype < 0 || q_dtype > 2)
    return ORACLE_ERR_ARG;
  int64_t max_len = 1;
  for (int b = 0; b < B; ++b)
    if (context_lens[b] > max_len) max_len = context_lens[b];
  int status = ORACLE_OK;
  const int64_t total = (int64_t)B * Q * Hq;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
    if (!scores) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < total; ++r) {
      if (!scores) continue;
      const int h = (int)(r % Hq), j = (int)((r / Hq) % Q);
      const int b = (int)(r / ((int64_t)Hq * Q));
      const int64_t visible = (int64_t)context_lens[b] - Q + 1 + j;
      const int g = h / (Hq / Hkv);
      double *o = out + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (visible <= 0) continue;
      if ((visible + bs - 1) / bs > max_blocks) {
#pragma omp atomic write
        status = ORACLE_ERR_BLOCK;
        continue;
      }
      const int64_t q_base = (((int64_t)b * Q + j) * Hq + h) * D;
      int bad = 0;
      for (int64_t i = 0; i < visible; ++i) {
        const int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
        if (phys < 0 || phys >= NB) { bad = 1; break; }
        const int64_t kb = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
          dot += widen(q, q_base + d, q_dtype) * (oracle_e4m3_value(k_cache[kb + d]) * k_scale);
        scores[i] = scale * dot;
      }
      if (bad) {
#pragma omp atomic write
        status = ORACLE_ERR_BLOCK;
        continue;
      }
      double m = scores[0];
      for (int64_t i = 1; i < visible; ++i)
        if (scores[i] > m) m = scores[i];
      double denom = 0.0;
      for (int64_t i = 0; i < visible; ++i) {
        const double w = exp(scores[i] - m);
        const int32_t phys = block_table[(int64_t)b * max_blocks + i / bs];
        const int64_t vb = (((int64_t)phys * Hkv + g) * bs + i % bs) * D;
        denom += w;
        for (int d = 0; d < D; ++d) o[d] += w * (oracle_e4m3_value(v_cache[vb + d]) * v_scale);
      }
      for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(scores);
  }
  return status;
}

/* Number of threads the parallel region above uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
