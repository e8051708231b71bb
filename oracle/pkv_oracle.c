/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for attention over a paged
 * KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header or
 * constant with the CUDA library; the two only ever see the same seeded
 * inputs.
 *
 * What it computes, and where the pages state it:
 *   - The KV cache is cut into fixed blocks of 256 token slots (tuning guide
 *     "Nano-vLLM性能调优实战", §1.1 KV缓存块配置: kvcache_block_size = 256).
 *   - A sequence's logical blocks reach physically scattered blocks through a
 *     block table; sequences with a common prefix point at the same physical
 *     blocks (ocdem.com nano-vllm article, §2.1 "基石PagedAttention 与 vLLM
 *     的精髓").
 *   - New K/V rows are written into the cache by a store step before the
 *     attention reads it; attention runs either as prefill over a chunk or as
 *     incremental decode of one token (tuning guide §2.2 缓存复用策略:
 *     store_kvcache + flash_attn_with_kvcache + variable-length batches;
 *     intelliparadigm.com Nano-vLLM article, §7.1 执行引擎工作流).
 *
 * Paging is only addressing, so the result is the plain definition of
 * softmax attention on each sequence's gathered keys and values.  The oracle
 * therefore (1) copies bit patterns for the store, (2) gathers K/V through
 * the block table into contiguous arrays, (3) runs textbook softmax
 * attention in double precision.  No blocking, online softmax or splitting.
 *
 * Readings taken where the pages are silent:
 *   - cache layout [num_blocks][256][num_kv_heads][head_dim], bf16; token
 *     slot = block_id * 256 + offset;
 *   - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads);
 *   - context_lens count the tokens already stored in this step;
 *   - in a prefill chunk of Lq queries over a context of C tokens, query i
 *     sits at position C - Lq + i and sees keys 0 .. C - Lq + i;
 *   - slot -1 means "do not store"; an empty context gives a zero output.
 *
 * Parity pins (see tests/test_oracle.py): brute force on tiny inputs, the
 * fp64 scaled-dot-product attention of the host library in the special case
 * of contiguous blocks, closed forms (one key, zero query, equal keys, a
 * dominant key, hand-worked values), block-permutation and prefix-sharing
 * invariance, softmax rows summing to one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 256

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARG = 1,
  ORACLE_BAD_BLOCK = 2,
  ORACLE_BAD_CONTEXT = 3,
  ORACLE_BAD_CHUNK = 4,
  ORACLE_BAD_SLOT = 5,
  ORACLE_NO_MEMORY = 6,
};

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

void oracle_bf16_to_f64(const uint16_t* src, int64_t n, double* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = widen_bf16(src[i]);
}

/*
 * Store step (tuning guide §2.2, "store_kvcache"): row i of k and v is
 * copied, bit for bit, into cache slot slot_mapping[i]; slot -1 skips the
 * row.  Rows of k/v are num_kv_heads * head_dim contiguous values, row i
 * starting at i * row_stride.
 */
int oracle_store_kvcache(const uint16_t* k, const uint16_t* v, int64_t k_row_stride,
                         int64_t v_row_stride, const int32_t* slot_mapping,
                         int64_t num_tokens, uint16_t* k_cache, uint16_t* v_cache,
                         int64_t num_blocks, int32_t num_kv_heads, int32_t head_dim) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0)
    return ORACLE_BAD_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  const int64_t num_slots = num_blocks * ORACLE_BLOCK;
  for (int64_t i = 0; i < num_tokens; ++i) {
    const int64_t slot = slot_mapping[i];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) return ORACLE_BAD_SLOT;
    for (int64_t e = 0; e < row; ++e) {
      k_cache[slot * row + e] = k[i * k_row_stride + e];
      v_cache[slot * row + e] = v[i * v_row_stride + e];
    }
  }
  return ORACLE_OK;
}

/*
 * INT8 KV cache (intelliparadigm.com article §2.2, "kv_cache_dtype: int8";
 * ocdem.com article §4.1 KV Cache 量化): each (token, KV head) row of
 * head_dim values is stored as int8 codes with one binary32 scale.  The
 * pages give no formula; this is symmetric absmax quantisation:
 *   scale = max_d |x_d| / 127,  code_d = nearest(x_d / scale), ties to even,
 * both decided in binary32 (the precision the codes are decided in on the
 * GPU too), codes in [-127, 127]; an all-zero row has scale 0 and zero
 * codes.  The value a code stands for is code * scale.  Decode and prefill
 * over the INT8 cache are the same attention as over the bf16 cache, on the
 * gathered values code * scale (exact in double).  Pins
 * (tests/test_oracle_int8.py): hand-worked quantised rows, the
 * round-to-nearest bound, and, with integer rows (every scale 1), bit
 * equality with the bf16 decode and prefill; the last row of an INT8 prefill
 * chunk equals the INT8 decode of that query.
 */
void oracle_quantize_row(const uint16_t* x, int32_t n, int8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int32_t d = 0; d < n; ++d) {
    const float a = fabsf((float)widen_bf16(x[d]));
    if (a > amax) amax = a;
  }
  const float s = amax / 127.0f;
  *scale = s;
  for (int32_t d = 0; d < n; ++d) {
    long c = 0;
    if (s > 0.0f) c = lrintf((float)widen_bf16(x[d]) / s);
    if (c > 127) c = 127;
    if (c < -127) c = -127;
    codes[d] = (int8_t)c;
  }
}

/* n_rows consecutive rows of n values each, one after another. */
void oracle_quantize_rows(const uint16_t* x, int64_t n_rows, int32_t n, int8_t* codes,
                          float* scales) {
  for (int64_t r = 0; r < n_rows; ++r)
    oracle_quantize_row(x + r * n, n, codes + r * n, scales + r);
}

/*
 * Where the INT8 cache keeps the row of (slot, KV head h): the pages fix no
 * layout; each block holds its heads one after another, codes
 * [num_blocks][num_kv_heads][256][head_dim] and scales
 * [num_blocks][num_kv_heads][256], so row index
 * (block * num_kv_heads + h) * 256 + offset, slot = block * 256 + offset.
 */
static int64_t int8_row(int64_t slot, int32_t num_kv_heads, int32_t h) {
  return ((slot / ORACLE_BLOCK) * num_kv_heads + h) * ORACLE_BLOCK + slot % ORACLE_BLOCK;
}

/*
 * INT8 store: row i of k and v, head h, is quantised into cache slot
 * slot_mapping[i]: codes at row int8_row(slot, h) of k_codes and its scale
 * at the same index of k_scales (the same for v); slot -1 skips the row.
 */
int oracle_store_kvcache_int8(const uint16_t* k, const uint16_t* v, int64_t k_row_stride,
                              int64_t v_row_stride, const int32_t* slot_mapping,
                              int64_t num_tokens, int8_t* k_codes, int8_t* v_codes,
                              float* k_scales, float* v_scales, int64_t num_blocks,
                              int32_t num_kv_heads, int32_t head_dim) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0)
    return ORACLE_BAD_ARG;
  const int64_t num_slots = num_blocks * ORACLE_BLOCK;
  for (int64_t i = 0; i < num_tokens; ++i) {
    const int64_t slot = slot_mapping[i];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) return ORACLE_BAD_SLOT;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const int64_t r = int8_row(slot, num_kv_heads, h);
      oracle_quantize_row(k + i * k_row_stride + (int64_t)h * head_dim, head_dim,
                          k_codes + r * head_dim, k_scales + r);
      oracle_quantize_row(v + i * v_row_stride + (int64_t)h * head_dim, head_dim,
                          v_codes + r * head_dim, v_scales + r);
    }
  }
  return ORACLE_OK;
}

/*
 * Gather (ocdem.com article §2.1): logical token t of a sequence lives in
 * physical block block_table[t / 256] at offset t % 256.  Produces
 * contiguous K and V of shape [context_len][num_kv_heads][head_dim].
 */
int oracle_gather(const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_blocks,
                  int32_t num_kv_heads, int32_t head_dim, const int32_t* block_table,
                  int32_t max_blocks, int32_t context_len, double* K, double* V) {
  if (context_len < 0) return ORACLE_BAD_CONTEXT;
  if ((int64_t)context_len > (int64_t)max_blocks * ORACLE_BLOCK) return ORACLE_BAD_CONTEXT;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int32_t t = 0; t < context_len; ++t) {
    const int64_t block = block_table[t / ORACLE_BLOCK];
    if (block < 0 || block >= num_blocks) return ORACLE_BAD_BLOCK;
    const int64_t slot = block * ORACLE_BLOCK + t % ORACLE_BLOCK;
    for (int64_t e = 0; e < row; ++e) {
      K[(int64_t)t * row + e] = widen_bf16(k_cache[slot * row + e]);
      V[(int64_t)t * row + e] = widen_bf16(v_cache[slot * row + e]);
    }
  }
  return ORACLE_OK;
}

/*
 * Gather of an INT8 cache: as oracle_gather, each value being
 * code * scale of its (slot, KV head) row int8_row(slot, h) (exact in double).
 */
int oracle_gather_int8(const int8_t* k_codes, const int8_t* v_codes, const float* k_scales,
                       const float* v_scales, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t* block_table, int32_t max_blocks,
                       int32_t context_len, double* K, double* V) {
  if (context_len < 0) return ORACLE_BAD_CONTEXT;
  if ((int64_t)context_len > (int64_t)max_blocks * ORACLE_BLOCK) return ORACLE_BAD_CONTEXT;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int32_t t = 0; t < context_len; ++t) {
    const int64_t block = block_table[t / ORACLE_BLOCK];
    if (block < 0 || block >= num_blocks) return ORACLE_BAD_BLOCK;
    const int64_t slot = block * ORACLE_BLOCK + t % ORACLE_BLOCK;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const int64_t r = int8_row(slot, num_kv_heads, h);
      const double ks = (double)k_scales[r], vs = (double)v_scales[r];
      for (int32_t d = 0; d < head_dim; ++d) {
        K[(int64_t)t * row + (int64_t)h * head_dim + d] = (double)k_codes[r * head_dim + d] * ks;
        V[(int64_t)t * row + (int64_t)h * head_dim + d] = (double)v_codes[r * head_dim + d] * vs;
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Textbook softmax attention of one query row q[head_dim] against the first
 * n_keys gathered keys of KV head kv_head:
 *   x_t = scale * sum_d q[d] * K[t][kv_head][d]
 *   p_t = exp(x_t - max x) / sum_u exp(x_u - max x)
 *   out[d] = sum_t p_t * V[t][kv_head][d]
 * probs (may be NULL) receives p_0 .. p_{n_keys-1}.  n_keys == 0 gives zeros.
 */
void oracle_attend(const double* q, const double* K, const double* V, int32_t num_kv_heads,
                   int32_t head_dim, int32_t kv_head, int32_t n_keys, double scale,
                   double* out, double* probs) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n_keys <= 0) return;
  double* x = (double*)malloc(sizeof(double) * (size_t)n_keys);
  if (!x) return;
  double m = -INFINITY;
  for (int32_t t = 0; t < n_keys; ++t) {
    const double* k = K + (int64_t)t * row + (int64_t)kv_head * head_dim;
    double dot = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) dot += q[d] * k[d];
    x[t] = scale * dot;
    if (x[t] > m) m = x[t];
  }
  double z = 0.0;
  for (int32_t t = 0; t < n_keys; ++t) {
    x[t] = exp(x[t] - m);
    z += x[t];
  }
  for (int32_t t = 0; t < n_keys; ++t) {
    const double p = x[t] / z;
    const double* v = V + (int64_t)t * row + (int64_t)kv_head * head_dim;
    for (int32_t d = 0; d < head_dim; ++d) out[d] += p * v[d];
    if (probs) probs[t] = p;
  }
  free(x);
}

/* A (row, head) pair listed more than once in a sampled request receives
 * the same output at every position it is listed. */
static void copy_to_repeats(const int32_t* rows, int32_t n_rows, int32_t first, int32_t r,
                            int32_t h, double* out, int32_t head_dim) {
  if (!rows || first < 0) return;
  for (int32_t i = first + 1; i < n_rows; ++i)
    if (rows[2 * i] == r && rows[2 * i + 1] == h)
      memcpy(out + (int64_t)i * head_dim, out + (int64_t)first * head_dim,
             sizeof(double) * (size_t)head_dim);
}

static int check_heads(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORACLE_BAD_ARG;
  if (num_q_heads % num_kv_heads != 0) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

/*
 * Decode (intelliparadigm.com article §7.1 增量解码; tuning guide §2.2):
 * one query per sequence, q[num_seqs][num_q_heads][head_dim], attends to all
 * context_lens[s] cached tokens.  If rows != NULL only the n_rows
 * (sequence, q head) pairs listed in rows[2*i], rows[2*i+1] are computed and
 * out is [n_rows][head_dim]; otherwise out is [num_seqs][num_q_heads][head_dim].
 */
/* The cache decode reads: bf16 (k, v) or INT8 (codes and scales). */
typedef struct {
  const uint16_t* k;
  const uint16_t* v;
  const int8_t* k_codes;
  const int8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
} CacheSource;

static int gather_from(const CacheSource* c, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t* block_table, int32_t max_blocks,
                       int32_t context_len, double* K, double* V) {
  if (c->k)
    return oracle_gather(c->k, c->v, num_blocks, num_kv_heads, head_dim, block_table,
                         max_blocks, context_len, K, V);
  return oracle_gather_int8(c->k_codes, c->v_codes, c->k_scales, c->v_scales, num_blocks,
                            num_kv_heads, head_dim, block_table, max_blocks, context_len, K, V);
}

static int decode_from(const uint16_t* q, const CacheSource* cache, int64_t num_blocks,
                       const int32_t* block_tables, int32_t max_blocks,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, double scale,
                       const int32_t* rows, int32_t n_rows, double* out) {
  int rc = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (rc) return rc;
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t kv_row = (int64_t)num_kv_heads * head_dim;
  double* qrow = (double*)malloc(sizeof(double) * (size_t)head_dim);
  if (!qrow) return ORACLE_NO_MEMORY;
  for (int32_t s = 0; s < num_seqs && rc == ORACLE_OK; ++s) {
    int wanted = rows == NULL;
    for (int32_t i = 0; i < n_rows && !wanted; ++i) wanted = rows[2 * i] == s;
    if (!wanted) continue;
    const int32_t ctx = context_lens[s];
    if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks * ORACLE_BLOCK) {
      rc = ORACLE_BAD_CONTEXT;
      break;
    }
    const size_t n = (size_t)(ctx > 0 ? ctx : 1) * (size_t)kv_row;
    double* K = (double*)malloc(sizeof(double) * n);
    double* V = (double*)malloc(sizeof(double) * n);
    if (!K || !V) {
      free(K);
      free(V);
      rc = ORACLE_NO_MEMORY;
      break;
    }
    rc = gather_from(cache, num_blocks, num_kv_heads, head_dim,
                     block_tables + (int64_t)s * max_blocks, max_blocks, ctx, K, V);
    for (int32_t h = 0; h < num_q_heads && rc == ORACLE_OK; ++h) {
      double* dst = NULL;
      int32_t first = -1;
      if (rows == NULL) {
        dst = out + ((int64_t)s * num_q_heads + h) * head_dim;
      } else {
        for (int32_t i = 0; i < n_rows && first < 0; ++i)
          if (rows[2 * i] == s && rows[2 * i + 1] == h) first = i;
        if (first >= 0) dst = out + (int64_t)first * head_dim;
      }
      if (!dst) continue;
      oracle_bf16_to_f64(q + ((int64_t)s * num_q_heads + h) * head_dim, head_dim, qrow);
      oracle_attend(qrow, K, V, num_kv_heads, head_dim, h / group, ctx, scale, dst, NULL);
      copy_to_repeats(rows, n_rows, first, s, h, out, head_dim);
    }
    free(K);
    free(V);
  }
  free(qrow);
  return rc;
}

int oracle_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                  int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks,
                  const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                  int32_t num_kv_heads, int32_t head_dim, double scale,
                  const int32_t* rows, int32_t n_rows, double* out) {
  const CacheSource c = {k_cache, v_cache, NULL, NULL, NULL, NULL};
  return decode_from(q, &c, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, scale, rows, n_rows, out);
}

/* Decode over an INT8 cache (codes [num_blocks][Hkv][256][D], scales
 * [num_blocks][Hkv][256]): the same attention on the values the codes stand for. */
int oracle_decode_int8(const uint16_t* q, const int8_t* k_codes, const int8_t* v_codes,
                       const float* k_scales, const float* v_scales, int64_t num_blocks,
                       const int32_t* block_tables, int32_t max_blocks,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, double scale,
                       const int32_t* rows, int32_t n_rows, double* out) {
  const CacheSource c = {NULL, NULL, k_codes, v_codes, k_scales, v_scales};
  return decode_from(q, &c, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, scale, rows, n_rows, out);
}

/*
 * Chunked prefill (tuning guide §3.2 max_num_batched_tokens; §2.2 variable
 * length batches; intelliparadigm.com article §7.1 预填充阶段): sequence s
 * owns query rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 of
 * q[total][num_q_heads][head_dim].  With Lq queries and C = context_lens[s]
 * cached tokens (the chunk included), query i sits at position C - Lq + i
 * and attends to keys 0 .. C - Lq + i.  If rows != NULL only the listed
 * (token row, q head) pairs are computed into out[n_rows][head_dim];
 * otherwise out is [total][num_q_heads][head_dim].
 */
static int prefill_from(const uint16_t* q, const CacheSource* cache, int64_t num_blocks,
                        const int32_t* block_tables, int32_t max_blocks,
                        const int32_t* cu_seqlens_q, const int32_t* context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, double scale, const int32_t* rows, int32_t n_rows,
                        double* out) {
  int rc = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (rc) return rc;
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t kv_row = (int64_t)num_kv_heads * head_dim;
  double* qrow = (double*)malloc(sizeof(double) * (size_t)head_dim);
  if (!qrow) return ORACLE_NO_MEMORY;
  for (int32_t s = 0; s < num_seqs && rc == ORACLE_OK; ++s) {
    const int32_t t0 = cu_seqlens_q[s], t1 = cu_seqlens_q[s + 1];
    const int32_t lq = t1 - t0, ctx = context_lens[s];
    if (lq < 0 || lq > ctx) {
      rc = ORACLE_BAD_CHUNK;
      break;
    }
    if ((int64_t)ctx > (int64_t)max_blocks * ORACLE_BLOCK) {
      rc = ORACLE_BAD_CONTEXT;
      break;
    }
    int wanted = rows == NULL && lq > 0;
    for (int32_t i = 0; i < n_rows && !wanted; ++i) wanted = rows[2 * i] >= t0 && rows[2 * i] < t1;
    if (!wanted) continue;
    const size_t n = (size_t)(ctx > 0 ? ctx : 1) * (size_t)kv_row;
    double* K = (double*)malloc(sizeof(double) * n);
    double* V = (double*)malloc(sizeof(double) * n);
    if (!K || !V) {
      free(K);
      free(V);
      rc = ORACLE_NO_MEMORY;
      break;
    }
    rc = gather_from(cache, num_blocks, num_kv_heads, head_dim,
                     block_tables + (int64_t)s * max_blocks, max_blocks, ctx, K, V);
    for (int32_t tok = t0; tok < t1 && rc == ORACLE_OK; ++tok) {
      const int32_t n_keys = ctx - lq + (tok - t0) + 1;
      for (int32_t h = 0; h < num_q_heads; ++h) {
        double* dst = NULL;
        int32_t first = -1;
        if (rows == NULL) {
          dst = out + ((int64_t)tok * num_q_heads + h) * head_dim;
        } else {
          for (int32_t i = 0; i < n_rows && first < 0; ++i)
            if (rows[2 * i] == tok && rows[2 * i + 1] == h) first = i;
          if (first >= 0) dst = out + (int64_t)first * head_dim;
        }
        if (!dst) continue;
        oracle_bf16_to_f64(q + ((int64_t)tok * num_q_heads + h) * head_dim, head_dim, qrow);
        oracle_attend(qrow, K, V, num_kv_heads, head_dim, h / group, n_keys, scale, dst, NULL);
        copy_to_repeats(rows, n_rows, first, tok, h, out, head_dim);
      }
    }
    free(K);
    free(V);
  }
  free(qrow);
  return rc;
}

int oracle_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                   int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks,
                   const int32_t* cu_seqlens_q, const int32_t* context_lens, int32_t num_seqs,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, double scale,
                   const int32_t* rows, int32_t n_rows, double* out) {
  const CacheSource c = {k_cache, v_cache, NULL, NULL, NULL, NULL};
  return prefill_from(q, &c, num_blocks, block_tables, max_blocks, cu_seqlens_q, context_lens,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, scale, rows, n_rows, out);
}

/* Chunked prefill over an INT8 cache (layout as for oracle_decode_int8): the
 * same causal attention on the values code * scale the codes stand for. */
int oracle_prefill_int8(const uint16_t* q, const int8_t* k_codes, const int8_t* v_codes,
                        const float* k_scales, const float* v_scales, int64_t num_blocks,
                        const int32_t* block_tables, int32_t max_blocks,
                        const int32_t* cu_seqlens_q, const int32_t* context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, double scale, const int32_t* rows, int32_t n_rows,
                        double* out) {
  const CacheSource c = {NULL, NULL, k_codes, v_codes, k_scales, v_scales};
  return prefill_from(q, &c, num_blocks, block_tables, max_blocks, cu_seqlens_q, context_lens,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, scale, rows, n_rows, out);
}
