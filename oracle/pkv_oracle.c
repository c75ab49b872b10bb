/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE, not part of the library.
 *
 * A plain, slow, FP64 CPU statement of what paged KV decode attention
 * computes.  It exists only to check the CUDA path: nothing in the library
 * links, imports or calls it.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load it.  It shares no code
 * with the CUDA path.
 *
 * What it follows, on the web textbook page "Chapter 8: Inference
 * Optimization" (clxhxhhr.top/posts/4341):
 *   - §8.1.1: in a decode step the model feeds the new token, reads the
 *     request's context KV and stores the new token's K and V;
 *   - §8.3.1 and Fig. 8-10: KV lives in fixed-size physical blocks; the
 *     request's block table maps logical block j (tokens j*p .. j*p+p-1) to a
 *     physical block, and attention finds each token's KV through it;
 *   - §8.3.1 worked example, Fig. 8-13: several block tables may reference
 *     the same physical block (a common prefix stored once);
 *   - §8.2.3, Fig. 8-8/8-9: of c new tokens after h cached ones, new token j
 *     (1-based) attends to the first h + j tokens.
 * The attention itself is the textbook definition out = softmax(scale*q.K^T) V
 * over the visible keys, evaluated directly in double precision: every logit,
 * then the maximum, then exp(s - max), their sum, and the weighted sum of V.
 * No blocking, no online rescaling, no reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* BF16 is the upper half of an IEEE binary32. */
static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Index of element d of token `off` of KV head `kvh` in physical block `blk`,
 * for the pool layout [num_blocks][num_kv_heads][block_size][head_dim]. */
static int64_t cache_index(int64_t blk, int32_t kvh, int32_t off, int32_t d, int32_t num_kv_heads,
                           int32_t block_size, int32_t head_dim) {
  return ((blk * num_kv_heads + kvh) * block_size + off) * (int64_t)head_dim + d;
}

/* Query i (0-based) of a request whose cache holds ctx tokens, q_len of them
 * new this step, sits at position ctx - q_len + i and sees key positions
 * 0 .. ctx - q_len + i (causal within the chunk; plain decode when q_len=1). */
static int key_visible(int64_t t, int32_t ctx, int32_t q_len, int32_t i) {
  return t < ctx && t <= (int64_t)ctx - q_len + i;
}

/* Store each new token's K and V in its slot: physical block slot / p,
 * offset slot % p.  Negative slots are padding and skipped; so are slots past
 * the pool. */
void oracle_kv_append(uint16_t* k_cache, uint16_t* v_cache, int32_t num_blocks, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_dim, const int64_t* slot_mapping,
                      const uint16_t* k_new, const uint16_t* v_new, int32_t num_tokens) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
    int64_t blk = slot / block_size;
    int32_t off = (int32_t)(slot % block_size);
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int32_t d = 0; d < head_dim; ++d) {
        int64_t dst = cache_index(blk, h, off, d, num_kv_heads, block_size, head_dim);
        int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
        k_cache[dst] = k_new[src];
        v_cache[dst] = v_new[src];
      }
    }
  }
}

/* Number of (query, key) pairs the causal rule admits over a batch. */
int64_t oracle_visible_pairs(const int32_t* context_lens, int32_t num_seqs, int32_t q_len) {
  int64_t n = 0;
  for (int32_t r = 0; r < num_seqs; ++r)
    for (int32_t i = 0; i < q_len; ++i)
      for (int64_t t = 0; t < context_lens[r]; ++t) n += key_visible(t, context_lens[r], q_len, i);
  return n;
}

/*
 * out     : [n_sel][q_len][num_q_heads][head_dim] doubles, n_sel = num_ids when
 *           seq_ids != NULL (rows seq_ids[0..num_ids)), else num_seqs.
 * out_lse : same rows without head_dim (natural log); may be NULL.
 * A query with no visible key gets zeros and lse = -inf.
 * Returns 0, or -1 when a table entry that must be read lies outside the pool.
 */
int oracle_paged_attention(double* out, double* out_lse, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                           int32_t q_len, int32_t num_q_heads, double scale, const int32_t* seq_ids,
                           int32_t num_ids, int32_t num_threads) {
  int32_t n_sel = seq_ids ? num_ids : num_seqs;
  int32_t group = num_q_heads / num_kv_heads; /* query heads per KV head */
  int64_t n_rows = (int64_t)n_sel * q_len * num_q_heads;
  int bad = 0;

  for (int32_t s = 0; s < n_sel; ++s) {
    int32_t r = seq_ids ? seq_ids[s] : s;
    int32_t ctx = context_lens[r];
    for (int64_t j = 0; j * block_size < ctx && !bad; ++j) {
      if (j >= max_blocks_per_seq) {
        bad = 1;
        break;
      }
      int32_t blk = block_tables[(int64_t)r * max_blocks_per_seq + j];
      if (blk < 0 || blk >= num_blocks) bad = 1;
    }
  }
  if (bad) return -1;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t row = 0; row < n_rows; ++row) {
    int32_t h = (int32_t)(row % num_q_heads);
    int32_t i = (int32_t)((row / num_q_heads) % q_len);
    int32_t s = (int32_t)(row / ((int64_t)num_q_heads * q_len));
    int32_t r = seq_ids ? seq_ids[s] : s;
    int32_t ctx = context_lens[r];
    int32_t kvh = h / group;
    const uint16_t* qv = q + (((int64_t)r * q_len + i) * num_q_heads + h) * head_dim;
    double* o = out + row * head_dim;
    for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;

    double* logit = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    double m = -INFINITY;
    for (int64_t t = 0; t < ctx; ++t) {
      if (!key_visible(t, ctx, q_len, i)) continue;
      int64_t blk = block_tables[(int64_t)r * max_blocks_per_seq + t / block_size];
      int32_t off = (int32_t)(t % block_size);
      double dot = 0.0;
      for (int32_t d = 0; d < head_dim; ++d)
        dot += bf16_value(qv[d]) *
               bf16_value(k_cache[cache_index(blk, kvh, off, d, num_kv_heads, block_size, head_dim)]);
      logit[t] = scale * dot;
      if (logit[t] > m) m = logit[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < ctx; ++t) {
      if (!key_visible(t, ctx, q_len, i)) continue;
      denom += exp(logit[t] - m);
    }
    for (int64_t t = 0; t < ctx; ++t) {
      if (!key_visible(t, ctx, q_len, i)) continue;
      int64_t blk = block_tables[(int64_t)r * max_blocks_per_seq + t / block_size];
      int32_t off = (int32_t)(t % block_size);
      double w = exp(logit[t] - m) / denom;
      for (int32_t d = 0; d < head_dim; ++d)
        o[d] += w * bf16_value(
                        v_cache[cache_index(blk, kvh, off, d, num_kv_heads, block_size, head_dim)]);
    }
    if (out_lse) out_lse[row] = denom > 0.0 ? m + log(denom) : -INFINITY;
    free(logit);
  }
  return 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int32_t oracle_max_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * q8_0 KV ("Chapter 8: Inference Optimization" §8.4.2, Fig. 8-23): every 32
 * consecutive values of a token's head vector share one 2-byte scale and are
 * stored as 8-bit codes, 34 bytes per 32 values.  The pages fix the storage;
 * the rounding is the plain symmetric one: d = max|x| / 127 in FP32, code =
 * round-half-away-from-zero(x * (1/d)), scale stored as FP16 (round to
 * nearest even); value = fp16(d) * code.  The integer decisions are taken in
 * FP32 exactly as written (the build disables contraction into FMA).
 * Tile of one (block, kv head): codes int8 [16][128] then scales fp16 [16][4].
 * --------------------------------------------------------------------------- */
#define Q8_TILE_BYTES 2176

static float bf16_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* 32 BF16 values -> 32 codes and the FP16 bit pattern of the scale. */
void oracle_quantize_q8_0_group(const uint16_t* x, int8_t* codes, uint16_t* scale_bits) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(bf16_float(x[i]));
    if (a > amax) amax = a;
  }
  float d = amax / 127.0f;
  float id = d != 0.0f ? 1.0f / d : 0.0f;
  for (int i = 0; i < 32; ++i) codes[i] = (int8_t)roundf(bf16_float(x[i]) * id);
  _Float16 h = (_Float16)d;
  memcpy(scale_bits, &h, sizeof h);
}

static double fp16_value(uint16_t bits) {
  _Float16 h;
  memcpy(&h, &bits, sizeof h);
  return (double)(float)h;
}

/* Store each new token's K and V in its slot of q8_0 pools
 * [num_blocks][num_kv_heads][Q8_TILE_BYTES]; same slot rules as
 * oracle_kv_append. */
void oracle_kv_append_q8_0(uint8_t* k_cache, uint8_t* v_cache, int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, const int64_t* slot_mapping, const uint16_t* k_new,
                           const uint16_t* v_new, int32_t num_tokens) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
    int64_t blk = slot / block_size;
    int32_t off = (int32_t)(slot % block_size);
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      for (int which = 0; which < 2; ++which) {
        uint8_t* tile = (which ? v_cache : k_cache) + (blk * num_kv_heads + h) * (int64_t)Q8_TILE_BYTES;
        const uint16_t* src = (which ? v_new : k_new) + ((int64_t)t * num_kv_heads + h) * 128;
        for (int g = 0; g < 4; ++g) {
          uint16_t sb;
          oracle_quantize_q8_0_group(src + 32 * g, (int8_t*)(tile + off * 128 + 32 * g), &sb);
          memcpy(tile + 2048 + (off * 4 + g) * 2, &sb, 2);
        }
      }
    }
  }
}

/* Dequantize q8_0 pools into double pools [num_blocks][num_kv_heads][block_size][128]. */
void oracle_dequantize_q8_0(const uint8_t* cache, double* out, int32_t num_blocks, int32_t num_kv_heads,
                            int32_t block_size) {
  for (int64_t bh = 0; bh < (int64_t)num_blocks * num_kv_heads; ++bh) {
    const uint8_t* tile = cache + bh * Q8_TILE_BYTES;
    for (int32_t t = 0; t < block_size; ++t)
      for (int32_t d = 0; d < 128; ++d) {
        uint16_t sb;
        memcpy(&sb, tile + 2048 + (t * 4 + d / 32) * 2, 2);
        out[(bh * block_size + t) * 128 + d] = fp16_value(sb) * (double)(int8_t)tile[t * 128 + d];
      }
  }
}

/* Attention over double pools (e.g. dequantized q8_0 values); otherwise
 * exactly oracle_paged_attention. */
int oracle_paged_attention_f64(double* out, double* out_lse, const uint16_t* q, const double* k_cache,
                               const double* v_cache, int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                               double scale, int32_t num_threads) {
  int32_t group = num_q_heads / num_kv_heads;
  int64_t n_rows = (int64_t)num_seqs * q_len * num_q_heads;
  for (int32_t r = 0; r < num_seqs; ++r)
    for (int64_t j = 0; j * block_size < context_lens[r]; ++j) {
      if (j >= max_blocks_per_seq) return -1;
      int32_t blk = block_tables[(int64_t)r * max_blocks_per_seq + j];
      if (blk < 0 || blk >= num_blocks) return -1;
    }
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t row = 0; row < n_rows; ++row) {
    int32_t h = (int32_t)(row % num_q_heads);
    int32_t i = (int32_t)((row / num_q_heads) % q_len);
    int32_t r = (int32_t)(row / ((int64_t)num_q_heads * q_len));
    int32_t ctx = context_lens[r];
    int32_t kvh = h / group;
    const uint16_t* qv = q + (((int64_t)r * q_len + i) * num_q_heads + h) * head_dim;
    double* o = out + row * head_dim;
    for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
    double* logit = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    double m = -INFINITY;
    for (int64_t t = 0; t < ctx; ++t) {
      if (!key_visible(t, ctx, q_len, i)) continue;
      int64_t blk = block_tables[(int64_t)r * max_blocks_per_seq + t / block_size];
      int32_t off = (int32_t)(t % block_size);
      double dot = 0.0;
      for (int32_t d = 0; d < head_dim; ++d)
        dot += bf16_value(qv[d]) * k_cache[cache_index(blk, kvh, off, d, num_kv_heads, block_size, head_dim)];
      logit[t] = scale * dot;
      if (logit[t] > m) m = logit[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < ctx; ++t)
      if (key_visible(t, ctx, q_len, i)) denom += exp(logit[t] - m);
    for (int64_t t = 0; t < ctx; ++t) {
      if (!key_visible(t, ctx, q_len, i)) continue;
      int64_t blk = block_tables[(int64_t)r * max_blocks_per_seq + t / block_size];
      int32_t off = (int32_t)(t % block_size);
      double w = exp(logit[t] - m) / denom;
      for (int32_t d = 0; d < head_dim; ++d)
        o[d] += w * v_cache[cache_index(blk, kvh, off, d, num_kv_heads, block_size, head_dim)];
    }
    if (out_lse) out_lse[row] = denom > 0.0 ? m + log(denom) : -INFINITY;
    free(logit);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * FP8 KV ("Chapter 8: Inference Optimization" §8.4.4: K and V stored in FP8,
 * the query kept in BF16).  The pages do not fix the FP8 variant; this is the
 * plain reading: OCP E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; subnormals below 2^-6; no infinities; magnitudes up to 448), each
 * BF16 value rounded to the nearest E4M3 value, ties to even mantissa, finite
 * values beyond 448 saturated to +-448, no scale.  Tile of one (block, kv
 * head): E4M3 codes [16][128], 2048 bytes.
 * --------------------------------------------------------------------------- */
#define FP8_TILE_BYTES 2048

/* Value of an E4M3 code (finite codes only; 0x7F / 0xFF are NaN). */
double oracle_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest E4M3 code of a finite value (round half to even, saturating). */
uint8_t oracle_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E; /* 448 = 1.75 * 2^8 */
  /* magnitudes are ordered like their codes 0x00 .. 0x7E: bisect */
  int lo = 0, hi = 0x7E;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_value((uint8_t)mid) <= a) lo = mid;
    else hi = mid;
  }
  double vlo = oracle_e4m3_value((uint8_t)lo), vhi = oracle_e4m3_value((uint8_t)hi);
  int pick;
  if (a - vlo < vhi - a) pick = lo;
  else if (a - vlo > vhi - a) pick = hi;
  else pick = (lo & 1) ? hi : lo; /* tie: the even code (even mantissa) */
  if (a == vhi) pick = hi;
  return sign | (uint8_t)pick;
}

/* Store each new token's K and V in its slot of E4M3 pools
 * [num_blocks][num_kv_heads][16][128]; same slot rules as oracle_kv_append. */
void oracle_kv_append_fp8(uint8_t* k_cache, uint8_t* v_cache, int32_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, const int64_t* slot_mapping, const uint16_t* k_new,
                          const uint16_t* v_new, int32_t num_tokens) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
    int64_t blk = slot / block_size;
    int32_t off = (int32_t)(slot % block_size);
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t d = 0; d < 128; ++d) {
        int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * 128 + d;
        int64_t src = ((int64_t)t * num_kv_heads + h) * 128 + d;
        k_cache[dst] = oracle_e4m3_encode(bf16_value(k_new[src]));
        v_cache[dst] = oracle_e4m3_encode(bf16_value(v_new[src]));
      }
  }
}

/* E4M3 pool -> double pool of the same shape. */
void oracle_dequantize_fp8(const uint8_t* cache, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(cache[i]);
}
