/*
 * Oracle for the paged-attention decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously correct CPU
 * statement of what the GPU library computes, used by the tests, by the
 * smoke check and by the benchmark's CPU-baseline leg.  The product never
 * calls it, links it or falls back to it, and it shares no code with the
 * GPU library.
 *
 * Sources (page title and section):
 *   [P1] "深入解析LLM推理引擎：从PagedAttention到调度优化"
 *   [P2] "vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量"
 *   [P3] "vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制"
 *
 * Arithmetic is IEEE binary64 throughout; fp16 inputs are widened exactly
 * and the attention output is rounded once to fp16 (round to nearest even).
 *
 * Cache layout (per layer): key_cache, value_cache are fp16
 * [num_blocks][num_heads][block_size][head_dim]; block_tables int32
 * [num_seqs][max_blocks]; context_lens int32 [num_seqs].  fp16 values are
 * passed as their uint16 bit patterns.
 *
 * Every function returns 0 on success, or a negative number when an index
 * in its input falls outside the arrays it was given (then the output is
 * not meaningful).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary64, from the format's definition:            */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                 */

double oracle_half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. */
uint16_t oracle_double_to_half(double x) {
  const uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00);
  const double a = fabs(x);
  /* 65504 is the largest finite half; the midpoint to 2^16 rounds to even,
   * which is the (infinite) next binade. */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
  if (a < 0x1p-14) {
    /* Subnormal range: the representable step is 2^-24. */
    const double r = nearbyint(a * 0x1p24);  /* exact scaling, RNE rounding */
    return (uint16_t)(sign | (uint16_t)r);   /* r == 1024 is the smallest normal */
  }
  int e2;
  frexp(a, &e2);                             /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;                            /* a in [2^E, 2^(E+1)) */
  double r = nearbyint(ldexp(a, 10 - E));    /* significand in units of 2^(E-10) */
  if (r == 2048.0) { r = 1024.0; E += 1; }
  if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | ((E + 15) << 10) | ((int)r - 1024));
}

void oracle_half_to_double_array(double* out, const uint16_t* in, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(in[i]);
}

void oracle_double_to_half_array(uint16_t* out, const double* in, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_double_to_half(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Paged address map [P2 §2.3]: logical token i of a sequence lives in      */
/* physical block BlockTable[i div B] at offset i mod B.  The slot of a     */
/* token is physical_block * B + offset [P1 §3.2, worked block-table         */
/* example].                                                                 */

int oracle_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                        const int32_t* token_seq, const int32_t* token_pos, int num_tokens,
                        int num_seqs, int block_size, int num_blocks) {
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int s = token_seq[t];
    const int pos = token_pos[t];
    if (s < 0) { slots[t] = -1; continue; }          /* padding token */
    if (s >= num_seqs || pos < 0 || pos / block_size >= max_blocks) { slots[t] = -1; bad = 1; continue; }
    const int phys = block_tables[(size_t)s * max_blocks + pos / block_size];
    if (phys < 0 || phys >= num_blocks) { slots[t] = -1; bad = 1; continue; }
    slots[t] = (int64_t)phys * block_size + pos % block_size;
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Cache write: token t's key/value vectors for every head go to the slot   */
/* the block manager assigned [P1 §3.2: a block fills token by token, a new */
/* block is taken when the last one is full].  slot < 0 marks a padding     */
/* token and is skipped.                                                     */

int oracle_reshape_and_cache(uint16_t* key_cache, uint16_t* value_cache, const uint16_t* key,
                             const uint16_t* value, const int64_t* slot_mapping, int num_tokens,
                             int num_heads, int head_dim, int block_size, int num_blocks) {
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size;
    const int64_t off = slot % block_size;
    if (blk >= num_blocks) { bad = 1; continue; }
    for (int h = 0; h < num_heads; ++h) {
      for (int d = 0; d < head_dim; ++d) {
        const size_t src = ((size_t)t * num_heads + h) * head_dim + d;
        const size_t dst = (((size_t)blk * num_heads + h) * block_size + off) * head_dim + d;
        key_cache[dst] = key[src];
        value_cache[dst] = value[src];
      }
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Copy-on-write block copy [P3 §2.3]: for each (src, dst) pair, in every   */
/* layer, the destination block receives the source block's keys and        */
/* values for all heads.  key_caches / value_caches hold num_layers         */
/* pointers.                                                                 */

int oracle_copy_blocks(uint16_t** key_caches, uint16_t** value_caches, int num_layers,
                       const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim,
                       int block_size, int num_blocks) {
  const size_t blk_elems = (size_t)num_heads * block_size * head_dim;
  int bad = 0;
  for (int p = 0; p < num_pairs; ++p) {
    const int64_t src = block_mapping[2 * p];
    const int64_t dst = block_mapping[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { bad = 1; continue; }
    for (int l = 0; l < num_layers; ++l) {
      for (size_t e = 0; e < blk_elems; ++e) {
        key_caches[l][(size_t)dst * blk_elems + e] = key_caches[l][(size_t)src * blk_elems + e];
        value_caches[l][(size_t)dst * blk_elems + e] = value_caches[l][(size_t)src * blk_elems + e];
      }
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Block swap between two pools ["【硬核】啃透vLLM源码" §三: when GPU memory   */
/* runs short the scheduler moves blocks to CPU memory and back              */
/* (blocks_to_swap_out / blocks_to_swap_in); "vLLM推理加速深度解读" §4.3     */
/* preemption]: for each pair (src, dst) and each of num_caches caches,      */
/* block dst of the destination pool receives block src of the source pool,  */
/* byte for byte (block_bytes bytes: all heads of one block of one layer's   */
/* keys or values).  Either pool may be the host's or the device's.          */

int oracle_swap_blocks(uint8_t** dst_caches, uint8_t** src_caches, int num_caches,
                       const int64_t* block_mapping, int num_pairs, size_t block_bytes,
                       int64_t src_num_blocks, int64_t dst_num_blocks) {
  int bad = 0;
  for (int p = 0; p < num_pairs; ++p) {
    const int64_t src = block_mapping[2 * p];
    const int64_t dst = block_mapping[2 * p + 1];
    if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) { bad = 1; continue; }
    for (int c = 0; c < num_caches; ++c)
      for (size_t e = 0; e < block_bytes; ++e)
        dst_caches[c][(size_t)dst * block_bytes + e] = src_caches[c][(size_t)src * block_bytes + e];
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over the paged cache [P2 §2.1, §2.3]:                   */
/*   out[s,h] = softmax(q[s,h] . K_paged^T * scale) V_paged                  */
/* with K_paged[i] = key_cache[bt[s][i div B]][h][i mod B] for i < c_s.      */
/* The softmax subtracts the maximum logit before exponentiating, which     */
/* leaves its value unchanged.  c_s == 0 gives a zero row.                   */
/* out16 (fp16 bits) and/or out64 (unrounded) may be NULL.                   */

int oracle_decode(uint16_t* out16, double* out64, const uint16_t* query,
                  const uint16_t* key_cache, const uint16_t* value_cache,
                  const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                  int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                  double scale) {
  int bad = 0;
  const long pairs = (long)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long sh = 0; sh < pairs; ++sh) {
    const int s = (int)(sh / num_heads);
    const int h = (int)(sh % num_heads);
    const int c = context_lens[s];
    double* acc = (double*)calloc((size_t)head_dim, sizeof(double));
    double* x = (double*)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    int ok = (c >= 0) && (c <= max_blocks * block_size);
    for (int d = 0; d < head_dim; ++d)
      qd[d] = oracle_half_to_double(query[((size_t)s * num_heads + h) * head_dim + d]);

    /* Logits x_i = (q . K_i) * scale. */
    for (int i = 0; ok && i < c; ++i) {
      const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
      if (phys < 0 || phys >= num_blocks) { ok = 0; break; }
      const uint16_t* k =
          key_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d) dot += qd[d] * oracle_half_to_double(k[d]);
      x[i] = dot * scale;
    }

    double denom = 0.0;
    if (ok && c > 0) {
      double m = x[0];
      for (int i = 1; i < c; ++i) if (x[i] > m) m = x[i];
      for (int i = 0; i < c; ++i) {
        const double w = exp(x[i] - m);
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        const uint16_t* v =
            value_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        denom += w;
        for (int d = 0; d < head_dim; ++d) acc[d] += w * oracle_half_to_double(v[d]);
      }
    }
    if (!ok) bad |= 1;

    for (int d = 0; d < head_dim; ++d) {
      const double o = (ok && c > 0) ? acc[d] / denom : 0.0;
      const size_t idx = ((size_t)s * num_heads + h) * head_dim + d;
      if (out64) out64[idx] = o;
      if (out16) out16[idx] = oracle_double_to_half(o);
    }
    free(acc);
    free(x);
    free(qd);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Multi-query paged attention: a chunk of new query tokens per sequence    */
/* (chunked prefill; decode is the one-token case; prefill and decode        */
/* sequences share one batch) ["vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" */
/* §4.3: prefill and decode in the same batch; "深入解析LLM推理引擎：从PagedAttention  */
/* 到调度优化" §3.3: attention reads K/V through the block table].           */
/* Sequence s has q_len = query_start[s+1] - query_start[s] new tokens, the  */
/* last q_len of its context_lens[s] tokens (their K/V already written);     */
/* new token j sits at position p = c_s - q_len + j and attends causally to  */
/* positions 0..p:                                                            */
/*   out[query_start[s]+j, h] = softmax_i<=p(scale q.K_i) V.                 */
/* query / out: [total_query_tokens][num_heads][head_dim].                    */

int oracle_prefill(uint16_t* out16, double* out64, const uint16_t* query,
                   const uint16_t* key_cache, const uint16_t* value_cache,
                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                   const int32_t* query_start, int num_seqs, int num_heads, int head_dim,
                   int block_size, int num_blocks, double scale) {
  int bad = 0;
  const long pairs = (long)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long sh = 0; sh < pairs; ++sh) {
    const int s = (int)(sh / num_heads);
    const int h = (int)(sh % num_heads);
    const int c = context_lens[s];
    const int q0 = query_start[s];
    const int q_len = query_start[s + 1] - q0;
    int ok = (c >= 0) && (c <= max_blocks * block_size) && (q_len >= 0) && (q_len <= c);
    double* x = (double*)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim);
    for (int j = 0; ok && j < q_len; ++j) {
      const int p = c - q_len + j;
      const size_t row = ((size_t)(q0 + j) * num_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) qd[d] = oracle_half_to_double(query[row + d]);
      for (int i = 0; ok && i <= p; ++i) {
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        if (phys < 0 || phys >= num_blocks) { ok = 0; break; }
        const uint16_t* k =
            key_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qd[d] * oracle_half_to_double(k[d]);
        x[i] = dot * scale;
      }
      if (!ok) break;
      double m = x[0];
      for (int i = 1; i <= p; ++i) if (x[i] > m) m = x[i];
      double denom = 0.0;
      for (int d = 0; d < head_dim; ++d) acc[d] = 0.0;
      for (int i = 0; i <= p; ++i) {
        const double w = exp(x[i] - m);
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        const uint16_t* v =
            value_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        denom += w;
        for (int d = 0; d < head_dim; ++d) acc[d] += w * oracle_half_to_double(v[d]);
      }
      for (int d = 0; d < head_dim; ++d) {
        const double o = acc[d] / denom;
        if (out64) out64[row + d] = o;
        if (out16) out16[row + d] = oracle_double_to_half(o);
      }
    }
    if (!ok) bad |= 1;
    free(x);
    free(qd);
    free(acc);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV cache ["vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §3.3 names */
/* FP8 support; the format and scaling are not given there].  Reading taken:  */
/* OCP FP8 E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3 fraction    */
/* bits, no infinities, S.1111.111 is NaN, largest finite 448), one scale per */
/* cache tensor: stored = E4M3(x / scale) with x / scale evaluated in IEEE    */
/* binary32 and rounded to nearest even, saturating to +-448; the value a     */
/* code stands for is E4M3(code) * scale.                                     */

double oracle_e4m3_to_double(uint8_t c) {
  const int sign = (c >> 7) & 1;
  const int e = (c >> 3) & 0xf;
  const int f = c & 7;
  double v;
  if (e == 15 && f == 7) return NAN;
  if (e == 0) v = ldexp((double)f, -9);           /* subnormal: f/8 * 2^-6 */
  else v = ldexp((double)(8 + f), e - 10);         /* (1 + f/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* Nearest E4M3 code to x (ties to even), saturating at +-448; NaN -> 0x7f. */
uint8_t oracle_double_to_e4m3(double x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return 0x7f;
  const double a = fabs(x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  if (a < 0x1p-6) {
    const double r = nearbyint(a * 0x1p9);   /* subnormal step 2^-9 */
    return (uint8_t)(sign | (uint8_t)r);      /* r == 8 is the smallest normal */
  }
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;                             /* a in [2^E, 2^(E+1)) */
  double r = nearbyint(ldexp(a, 3 - E));      /* significand in units of 2^(E-3) */
  if (r == 16.0) { r = 8.0; E += 1; }
  if (E + 7 > 15 || (E + 7 == 15 && r - 8 > 6)) return (uint8_t)(sign | 0x7e);
  return (uint8_t)(sign | ((E + 7) << 3) | ((int)r - 8));
}

void oracle_e4m3_to_double_array(double* out, const uint8_t* in, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(in[i]);
}

void oracle_double_to_e4m3_array(uint8_t* out, const double* in, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_double_to_e4m3(in[i]);
}

/* Quantised code of an fp16 value under a scale: E4M3(fl32(x / scale)). */
static uint8_t quantize_e4m3(uint16_t h, float scale) {
  const float x = (float)oracle_half_to_double(h);   /* exact */
  const float y = x / scale;                          /* binary32 division, round to nearest */
  return oracle_double_to_e4m3((double)y);
}

/* Elementwise quantisation of n fp16 values (a whole cache, layout kept).
   Elements are independent; the loop is split over threads. */
void oracle_quantize_e4m3_array(uint8_t* out, const uint16_t* in, size_t n, float scale) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = quantize_e4m3(in[i], scale);
}

/* Cache write into FP8 caches (same slots as oracle_reshape_and_cache). */
int oracle_reshape_and_cache_fp8(uint8_t* key_cache, uint8_t* value_cache, const uint16_t* key,
                                 const uint16_t* value, const int64_t* slot_mapping,
                                 int num_tokens, int num_heads, int head_dim, int block_size,
                                 int num_blocks, float k_scale, float v_scale) {
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size;
    const int64_t off = slot % block_size;
    if (blk >= num_blocks) { bad = 1; continue; }
    for (int h = 0; h < num_heads; ++h) {
      for (int d = 0; d < head_dim; ++d) {
        const size_t src = ((size_t)t * num_heads + h) * head_dim + d;
        const size_t dst = (((size_t)blk * num_heads + h) * block_size + off) * head_dim + d;
        key_cache[dst] = quantize_e4m3(key[src], k_scale);
        value_cache[dst] = quantize_e4m3(value[src], v_scale);
      }
    }
  }
  return bad ? -1 : 0;
}

/* Decode over FP8 caches: the same attention on the dequantised values
 * K_i = E4M3(code) * k_scale, V_i = E4M3(code) * v_scale (exact in binary64). */
int oracle_decode_fp8(uint16_t* out16, double* out64, const uint16_t* query,
                      const uint8_t* key_cache, const uint8_t* value_cache,
                      const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                      int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                      double scale, double k_scale, double v_scale) {
  int bad = 0;
  const long pairs = (long)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long sh = 0; sh < pairs; ++sh) {
    const int s = (int)(sh / num_heads);
    const int h = (int)(sh % num_heads);
    const int c = context_lens[s];
    double* acc = (double*)calloc((size_t)head_dim, sizeof(double));
    double* x = (double*)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    int ok = (c >= 0) && (c <= max_blocks * block_size);
    for (int d = 0; d < head_dim; ++d)
      qd[d] = oracle_half_to_double(query[((size_t)s * num_heads + h) * head_dim + d]);
    for (int i = 0; ok && i < c; ++i) {
      const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
      if (phys < 0 || phys >= num_blocks) { ok = 0; break; }
      const uint8_t* k =
          key_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d) dot += qd[d] * (oracle_e4m3_to_double(k[d]) * k_scale);
      x[i] = dot * scale;
    }
    double denom = 0.0;
    if (ok && c > 0) {
      double m = x[0];
      for (int i = 1; i < c; ++i) if (x[i] > m) m = x[i];
      for (int i = 0; i < c; ++i) {
        const double w = exp(x[i] - m);
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        const uint8_t* v =
            value_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        denom += w;
        for (int d = 0; d < head_dim; ++d) acc[d] += w * (oracle_e4m3_to_double(v[d]) * v_scale);
      }
    }
    if (!ok) bad |= 1;
    for (int d = 0; d < head_dim; ++d) {
      const double o = (ok && c > 0) ? acc[d] / denom : 0.0;
      const size_t idx = ((size_t)s * num_heads + h) * head_dim + d;
      if (out64) out64[idx] = o;
      if (out16) out16[idx] = oracle_double_to_half(o);
    }
    free(acc);
    free(x);
    free(qd);
  }
  return bad ? -1 : 0;
}

/* Multi-query paged attention over FP8 caches: the causal attention of
 * oracle_prefill on the dequantised values K_i = E4M3(code) * k_scale,
 * V_i = E4M3(code) * v_scale (exact in binary64).  Returns -1 on the same
 * bad inputs as oracle_prefill. */
int oracle_prefill_fp8(uint16_t* out16, double* out64, const uint16_t* query,
                       const uint8_t* key_cache, const uint8_t* value_cache,
                       const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       const int32_t* query_start, int num_seqs, int num_heads, int head_dim,
                       int block_size, int num_blocks, double scale, double k_scale,
                       double v_scale) {
  int bad = 0;
  const long pairs = (long)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long sh = 0; sh < pairs; ++sh) {
    const int s = (int)(sh / num_heads);
    const int h = (int)(sh % num_heads);
    const int c = context_lens[s];
    const int q0 = query_start[s];
    const int q_len = query_start[s + 1] - q0;
    int ok = (c >= 0) && (c <= max_blocks * block_size) && (q_len >= 0) && (q_len <= c);
    double* x = (double*)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim);
    for (int j = 0; ok && j < q_len; ++j) {
      const int p = c - q_len + j; /* position of new token j: it sees keys 0..p */
      const size_t row = ((size_t)(q0 + j) * num_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) qd[d] = oracle_half_to_double(query[row + d]);
      for (int i = 0; ok && i <= p; ++i) {
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        if (phys < 0 || phys >= num_blocks) { ok = 0; break; }
        const uint8_t* k =
            key_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qd[d] * (oracle_e4m3_to_double(k[d]) * k_scale);
        x[i] = dot * scale;
      }
      if (!ok) break;
      double m = x[0];
      for (int i = 1; i <= p; ++i) if (x[i] > m) m = x[i];
      double denom = 0.0;
      for (int d = 0; d < head_dim; ++d) acc[d] = 0.0;
      for (int i = 0; i <= p; ++i) {
        const double w = exp(x[i] - m);
        const int phys = block_tables[(size_t)s * max_blocks + i / block_size];
        const uint8_t* v =
            value_cache + (((size_t)phys * num_heads + h) * block_size + i % block_size) * head_dim;
        denom += w;
        for (int d = 0; d < head_dim; ++d) acc[d] += w * (oracle_e4m3_to_double(v[d]) * v_scale);
      }
      for (int d = 0; d < head_dim; ++d) {
        const double o = acc[d] / denom;
        if (out64) out64[row + d] = o;
        if (out16) out16[row + d] = oracle_double_to_half(o);
      }
    }
    if (!ok) bad |= 1;
    free(x);
    free(qd);
    free(acc);
  }
  return bad ? -1 : 0;
}

/* Threads the parallel loops use (OpenMP's maximum, 1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Sets the threads later parallel loops use (n >= 1; no effect without OpenMP). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
