/*
 * oracle.c -- plain, slow fp64 CPU oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline arm load
 * this library. It shares no code, header or constant with the CUDA library, and it never calls it.
 *
 * What it computes, and where the source pages say so:
 *
 *  [P1] "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), section "vLLM是什么？":
 *       the KV cache is cut into fixed-size blocks; a block table maps each sequence's logical
 *       blocks to physical blocks, so one sequence's keys and values sit in blocks that need not
 *       be contiguous; the attention kernel fetches each block separately; KV can be shared within
 *       and across requests.
 *  [P3] "nano-vllm 深度分析报告", table "可复用的模式与技巧", row "slot_mapping -1 padding":
 *       positions padded for CUDA graphs carry slot -1 and the cache-store kernel skips them;
 *       section "创新之处": prefix-cache hits reuse physical blocks.
 *
 * Paging changes where bytes live, not the arithmetic: attention over a paged cache is ordinary
 * softmax attention over the sequence's keys and values laid end to end. So this oracle first
 * materialises each sequence's contiguous K and V by walking its block table, then applies the
 * textbook formula  o = sum_j w_j v_j / sum_j w_j,  w_j = exp(s_j - max s),  s_j = scale * q.k_j
 * in double precision (bf16 -> double is exact).
 *
 * Readings where the pages are silent (the design notes list them all):
 *  - slot = physical_block * block_size + offset; the row it names is (slot / BS, slot % BS).
 *  - exactly -1 is padding; any other negative or out-of-range slot is invalid: it is skipped
 *    and counted.
 *  - grouped-query attention: query head h reads kv head h / (Hq / Hkv).
 *  - decode attends over context_lens[b] tokens (the newest token has already been stored);
 *    a sequence with context 0 (a padded batch entry) produces zeros.
 *  - prefill is causal and aligned to the end: new query i of a sequence with q_len new tokens
 *    and k_len keys sees keys 0 .. k_len - q_len + i. Keys below k_len - q_len are the cached
 *    prefix (read through the block table); the rest are the new tokens themselves.
 *
 * Layouts: caches [num_blocks, block_size, Hkv, D]; q [rows, Hq, D]; k/v new rows [rows, Hkv, D];
 * bf16 values are passed as their uint16 bit patterns; outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------------------------------------
 * KV store [P3 slot_mapping -1 padding; P1 fixed-size blocks].
 * For each token t: s = slot_mapping[t]; s == -1 is skipped; otherwise the token's K row and V row
 * (Hkv * D values each) are copied bit for bit to block s / BS, offset s % BS of the caches.
 * Returns the number of invalid slots (skipped).
 * ------------------------------------------------------------------------------------------- */
int64_t oracle_kv_store(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                        int64_t num_tokens, int32_t num_blocks, int32_t block_size,
                        int32_t num_kv_heads, int32_t head_dim, uint16_t *k_cache,
                        uint16_t *v_cache) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  int64_t invalid = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s == -1) continue;
    if (s < 0 || s >= (int64_t)num_blocks * block_size) {
      ++invalid;
      continue;
    }
    const int64_t block = s / block_size;
    const int64_t offset = s % block_size;
    const int64_t dst = (block * block_size + offset) * row;
    memcpy(k_cache + dst, k + t * row, (size_t)row * sizeof(uint16_t));
    memcpy(v_cache + dst, v + t * row, (size_t)row * sizeof(uint16_t));
  }
  return invalid;
}

/* ---------------------------------------------------------------------------------------------
 * Materialise [P1 block table]: out[p][d] = cache[bt_row[p / BS], p % BS, kv_head, d] for p < len,
 * as doubles. Returns -1 if the walk meets a block id outside [0, num_blocks), else 0.
 * ------------------------------------------------------------------------------------------- */
int oracle_gather_head(const uint16_t *cache, int32_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, const int32_t *bt_row, int32_t len,
                       int32_t kv_head, double *out) {
  for (int32_t p = 0; p < len; ++p) {
    const int64_t block = bt_row[p / block_size];
    const int64_t offset = p % block_size;
    if (block < 0 || block >= num_blocks) return -1;
    const uint16_t *src =
        cache + ((block * block_size + offset) * num_kv_heads + kv_head) * (int64_t)head_dim;
    for (int32_t d = 0; d < head_dim; ++d) out[(int64_t)p * head_dim + d] = bf16_to_double(src[d]);
  }
  return 0;
}

/* Softmax attention of one query row over n keys (the textbook definition).
 * q: head_dim doubles; K, V: n x head_dim doubles; out: head_dim doubles; s: n doubles scratch. */
static void attend_one(const double *q, const double *K, const double *V, int64_t n,
                       int32_t head_dim, double scale, double *s, double *out) {
  if (n <= 0) {
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) dot += q[d] * K[j * head_dim + d];
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double den = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    s[j] = exp(s[j] - m);
    den += s[j];
  }
  for (int32_t d = 0; d < head_dim; ++d) {
    double num = 0.0;
    for (int64_t j = 0; j < n; ++j) num += s[j] * V[j * head_dim + d];
    out[d] = num / den;
  }
}

/* ---------------------------------------------------------------------------------------------
 * Paged decode [P1 PagedAttention]: for sequence b and query head h (kv head g = h / G),
 * out[b][h] = softmax(scale * q[b][h] . K_b^T) V_b over the context_lens[b] cached tokens, where
 * K_b, V_b are materialised through block_tables[b]. Work is split over (sequence, kv head) units.
 * Returns 0, or -1 if a block table walk leaves the pool (that unit's outputs are then NaN).
 * ------------------------------------------------------------------------------------------- */
int oracle_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                        int32_t head_dim, const int32_t *block_tables, int32_t max_blocks,
                        const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                        double scale, double *out, int32_t num_threads) {
  const int32_t G = num_q_heads / num_kv_heads;
  const int64_t units = (int64_t)num_seqs * num_kv_heads;
  int status = 0;
  if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(min : status)
  for (int64_t u = 0; u < units; ++u) {
    const int32_t b = (int32_t)(u / num_kv_heads);
    const int32_t g = (int32_t)(u % num_kv_heads);
    const int32_t ctx = context_lens[b];
    const int64_t n = ctx > 0 ? ctx : 0;
    double *K = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
    double *V = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(n + 1));
    double *qh = (double *)malloc(sizeof(double) * (size_t)head_dim);
    const int32_t *bt_row = block_tables + (int64_t)b * max_blocks;
    int bad = 0;
    if (n > 0) {
      bad |= oracle_gather_head(k_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,
                                (int32_t)n, g, K);
      bad |= oracle_gather_head(v_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,
                                (int32_t)n, g, V);
    }
    for (int32_t h = g * G; h < (g + 1) * G; ++h) {
      double *o = out + ((int64_t)b * num_q_heads + h) * head_dim;
      if (bad) {
        for (int32_t d = 0; d < head_dim; ++d) o[d] = NAN;
        continue;
      }
      const uint16_t *qsrc = q + ((int64_t)b * num_q_heads + h) * head_dim;
      for (int32_t d = 0; d < head_dim; ++d) qh[d] = bf16_to_double(qsrc[d]);
      attend_one(qh, K, V, n, head_dim, scale, s, o);
    }
    if (bad) status = -1;
    free(K);
    free(V);
    free(s);
    free(qh);
  }
  return status;
}

/* ---------------------------------------------------------------------------------------------
 * Varlen paged causal prefill [P1 PagedAttention; P3 prefix-cache hits share blocks].
 * Sequence b has q_len = cu_q[b+1] - cu_q[b] new tokens (rows cu_q[b] .. of q, k, v) and
 * k_len = cu_k[b+1] - cu_k[b] keys; P = k_len - q_len keys form the cached prefix, read through
 * block_tables[b] (block_tables may be NULL only when every P is 0). Key j < P is prefix position
 * j; key j >= P is new token j - P. New query i attends keys 0 .. P + i.
 * Returns 0, -1 if a block walk leaves the pool, -2 if some k_len < q_len or a prefix has no table.
 * ------------------------------------------------------------------------------------------- */
int oracle_paged_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         int32_t num_seqs, const int32_t *block_tables, int32_t max_blocks,
                         const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                         int32_t num_q_heads, double scale, double *out, int32_t num_threads) {
  const int32_t G = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    const int32_t k_len = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
    if (q_len < 0 || k_len < q_len) return -2;
    if (k_len > q_len && block_tables == NULL) return -2;
  }
  const int64_t units = (int64_t)num_seqs * num_kv_heads;
  int status = 0;
  if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(min : status)
  for (int64_t u = 0; u < units; ++u) {
    const int32_t b = (int32_t)(u / num_kv_heads);
    const int32_t g = (int32_t)(u % num_kv_heads);
    const int64_t row0 = cu_seqlens_q[b];
    const int32_t q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    const int32_t k_len = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
    const int32_t P = k_len - q_len;
    double *K = (double *)malloc(sizeof(double) * (size_t)((int64_t)k_len * head_dim + 1));
    double *V = (double *)malloc(sizeof(double) * (size_t)((int64_t)k_len * head_dim + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(k_len + 1));
    double *qh = (double *)malloc(sizeof(double) * (size_t)head_dim);
    int bad = 0;
    if (P > 0) {
      const int32_t *bt_row = block_tables + (int64_t)b * max_blocks;
      bad |= oracle_gather_head(k_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,
                                P, g, K);
      bad |= oracle_gather_head(v_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,
                                P, g, V);
    }
    for (int32_t j = P; j < k_len; ++j) {
      const int64_t src = ((row0 + (j - P)) * num_kv_heads + g) * (int64_t)head_dim;
      for (int32_t d = 0; d < head_dim; ++d) {
        K[(int64_t)j * head_dim + d] = bf16_to_double(k[src + d]);
        V[(int64_t)j * head_dim + d] = bf16_to_double(v[src + d]);
      }
    }
    for (int32_t i = 0; i < q_len; ++i) {
      for (int32_t h = g * G; h < (g + 1) * G; ++h) {
        double *o = out + ((row0 + i) * num_q_heads + h) * head_dim;
        if (bad) {
          for (int32_t d = 0; d < head_dim; ++d) o[d] = NAN;
          continue;
        }
        const uint16_t *qsrc = q + ((row0 + i) * num_q_heads + h) * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) qh[d] = bf16_to_double(qsrc[d]);
        attend_one(qh, K, V, (int64_t)P + i + 1, head_dim, scale, s, o);
      }
    }
    if (bad) status = -1;
    free(K);
    free(V);
    free(s);
    free(qh);
  }
  return status;
}

/* ---------------------------------------------------------------------------------------------
 * Whole-block moves ["nano-vllm 深度分析报告", section "解法哲学": swap (CPU offload) and
 * copy-on-write act on whole physical blocks]. block_elems = block_size * Hkv * D values.
 * Each returns the number of entries skipped because a block id was outside [0, num_blocks).
 * ------------------------------------------------------------------------------------------- */
int32_t oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                           int64_t block_elems, const int32_t *pairs, int32_t n) {
  int32_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      ++bad;
      continue;
    }
    memcpy(k_cache + dst * block_elems, k_cache + src * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
    memcpy(v_cache + dst * block_elems, v_cache + src * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
  }
  return bad;
}

int32_t oracle_gather_blocks(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks,
                             int64_t block_elems, const int32_t *ids, int32_t n, uint16_t *out_k,
                             uint16_t *out_v) {
  int32_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t blk = ids[i];
    if (blk < 0 || blk >= num_blocks) {
      ++bad;
      continue;
    }
    memcpy(out_k + i * block_elems, k_cache + blk * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
    memcpy(out_v + i * block_elems, v_cache + blk * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
  }
  return bad;
}

int32_t oracle_scatter_blocks(const uint16_t *in_k, const uint16_t *in_v, const int32_t *ids,
                              int32_t n, uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                              int64_t block_elems) {
  int32_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t blk = ids[i];
    if (blk < 0 || blk >= num_blocks) {
      ++bad;
      continue;
    }
    memcpy(k_cache + blk * block_elems, in_k + i * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
    memcpy(v_cache + blk * block_elems, in_v + i * block_elems,
           (size_t)block_elems * sizeof(uint16_t));
  }
  return bad;
}

/* ---------------------------------------------------------------------------------------------
 * Chained block hashes for prefix caching ["nano-vllm 深度分析报告", section "创新之处" and table
 * "可复用的模式与技巧": each full block is content-addressed by an xxhash64 that includes the hash
 * of the blocks before it, so equal hashes mean equal token prefixes, not just equal blocks].
 * Reading: block i of a sequence hashes the byte string
 *     [8-byte little-endian hash of block i-1, omitted for block 0] ++ [its block_size token ids
 *      as 4-byte little-endian integers]
 * with XXH64, seed 0. Only full blocks are hashed.
 *
 * XXH64 below follows the published xxHash specification (64-bit variant): four 64-bit lanes
 * over 32-byte stripes, lane merge, length, 8/4/1-byte tail steps, final avalanche.
 * ------------------------------------------------------------------------------------------- */
static const uint64_t XXP1 = 0x9E3779B185EBCA87ull, XXP2 = 0xC2B2AE3D27D4EB4Full,
                      XXP3 = 0x165667B19E3779F9ull, XXP4 = 0x85EBCA77C2B2AE63ull,
                      XXP5 = 0x27D4EB2F165667C5ull;

static uint64_t rotl64(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

static uint64_t read_le64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

static uint32_t read_le32(const uint8_t *p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static uint64_t xx_round(uint64_t acc, uint64_t lane) {
  acc += lane * XXP2;
  acc = rotl64(acc, 31);
  return acc * XXP1;
}

uint64_t oracle_xxh64(const uint8_t *data, int64_t len, uint64_t seed) {
  const uint8_t *p = data;
  const uint8_t *end = data + len;
  uint64_t acc;
  if (len >= 32) {
    uint64_t v1 = seed + XXP1 + XXP2, v2 = seed + XXP2, v3 = seed, v4 = seed - XXP1;
    while (end - p >= 32) {
      v1 = xx_round(v1, read_le64(p));
      v2 = xx_round(v2, read_le64(p + 8));
      v3 = xx_round(v3, read_le64(p + 16));
      v4 = xx_round(v4, read_le64(p + 24));
      p += 32;
    }
    acc = rotl64(v1, 1) + rotl64(v2, 7) + rotl64(v3, 12) + rotl64(v4, 18);
    const uint64_t lanes[4] = {v1, v2, v3, v4};
    for (int i = 0; i < 4; ++i) {
      acc ^= xx_round(0, lanes[i]);
      acc = acc * XXP1 + XXP4;
    }
  } else {
    acc = seed + XXP5;
  }
  acc += (uint64_t)len;
  while (end - p >= 8) {
    acc ^= xx_round(0, read_le64(p));
    acc = rotl64(acc, 27) * XXP1 + XXP4;
    p += 8;
  }
  if (end - p >= 4) {
    acc ^= (uint64_t)read_le32(p) * XXP1;
    acc = rotl64(acc, 23) * XXP2 + XXP3;
    p += 4;
  }
  while (p < end) {
    acc ^= (uint64_t)(*p) * XXP5;
    acc = rotl64(acc, 11) * XXP1;
    ++p;
  }
  acc ^= acc >> 33;
  acc *= XXP2;
  acc ^= acc >> 29;
  acc *= XXP3;
  acc ^= acc >> 32;
  return acc;
}

/* Hashes of the full blocks of each sequence: out[b * max_blocks + i] for i < len_b / block_size
 * (tokens of sequence b are token_ids[cu_seqlens[b] .. cu_seqlens[b+1])). Returns the number of
 * sequences with more full blocks than max_blocks (their extra blocks are not hashed). */
int32_t oracle_block_hashes(const int32_t *token_ids, const int32_t *cu_seqlens, int32_t num_seqs,
                            int32_t block_size, int32_t max_blocks, uint64_t *out) {
  int32_t clamped = 0;
  uint8_t *buf = (uint8_t *)malloc(8 + 4 * (size_t)block_size);
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t len = cu_seqlens[b + 1] - cu_seqlens[b];
    int32_t nfull = len / block_size;
    if (nfull > max_blocks) {
      ++clamped;
      nfull = max_blocks;
    }
    uint64_t parent = 0;
    for (int32_t i = 0; i < nfull; ++i) {
      size_t n = 0;
      if (i > 0)
        for (int k = 0; k < 8; ++k) buf[n++] = (uint8_t)(parent >> (8 * k));
      const int32_t *tok = token_ids + cu_seqlens[b] + (int64_t)i * block_size;
      for (int32_t t = 0; t < block_size; ++t)
        for (int k = 0; k < 4; ++k) buf[n++] = (uint8_t)((uint32_t)tok[t] >> (8 * k));
      parent = oracle_xxh64(buf, (int64_t)n, 0);
      out[(int64_t)b * max_blocks + i] = parent;
    }
  }
  free(buf);
  return clamped;
}
