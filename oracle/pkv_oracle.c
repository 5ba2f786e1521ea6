/*
 * pkv_oracle.c -- plain, slow fp64 CPU oracle for the paged-KV attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code, header,
 * table or helper with the CUDA library; the only thing both sides share is
 * the seeded input generator, which holds none of this arithmetic.
 *
 * What it computes follows nano-vllm as described on the page
 * "13. 读一个最小推理引擎：nano-vllm" (commit bb823b3):
 *   - the per-layer cache is (num_blocks, block_size, num_kv_heads, head_dim)
 *     ("第五站：执行准备与 KV 容量", KV-capacity paragraph);
 *   - the KV write copies each token's whole K row and V row
 *     (num_kv_heads * head_dim contiguous elements) to offset slot * row in the
 *     cache and skips slot -1 ("第六站：注意力层", the store kernel);
 *   - logical position p of a sequence lives at physical slot
 *     block_table[p / bs] * bs + p % bs ("第五站", slot mapping);
 *   - attention is causal softmax attention over the cached context, read
 *     through the block table, for varlen prefill starting at
 *     num_cached_tokens and for one-token decode ("第二站" num_cached_tokens,
 *     "第六站" FlashAttention calls).
 * Readings where the page is silent (all listed in the design notes):
 *   - GQA: query head h uses kv head h / (Hq / Hkv);
 *   - a prefill sequence with L keys and n queries places query j at absolute
 *     position L - n + j (bottom-right causal alignment), so it sees keys
 *     0 .. L - n + j;
 *   - a decode row with context length 0 (graph padding) yields zeros;
 *   - scale multiplies the raw dot product before the softmax.
 *
 * Every value is computed in IEEE double.  bf16 inputs (passed as raw uint16
 * bit patterns) widen to double exactly.  No blocking, no online softmax, no
 * reordering: scores are computed, the maximum subtracted, exponentiated,
 * normalised by their sum and used to weight V, in that order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_RANGE (-2)
#define ORACLE_ERR_NOMEM (-3)

static double widen_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int pkv_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void pkv_oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * KV write.  For token i in order: s = slot_mapping[i]; s == -1 means a
 * padding row and is skipped; otherwise the token's K row and V row
 * (row_elems = num_kv_heads * head_dim elements) are copied to cache
 * offset s * row_elems.  Tokens are applied in index order.
 */
int pkv_oracle_kv_cache_write(const uint16_t* k, int64_t k_token_stride, const uint16_t* v,
                              int64_t v_token_stride, const int32_t* slot_mapping,
                              int64_t num_tokens, uint16_t* k_cache, uint16_t* v_cache,
                              int64_t num_slots, int64_t row_elems) {
  if (num_tokens < 0 || row_elems <= 0 || num_slots < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t s = slot_mapping[i];
    if (s == -1) continue;
    if (s < 0 || s >= num_slots) return ORACLE_ERR_RANGE;
  }
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t s = slot_mapping[i];
    if (s == -1) continue;
    for (int64_t e = 0; e < row_elems; ++e) {
      k_cache[s * row_elems + e] = k[i * k_token_stride + e];
      v_cache[s * row_elems + e] = v[i * v_token_stride + e];
    }
  }
  return ORACLE_OK;
}

/* Physical slot of logical position p through one sequence's block table. */
static int64_t slot_of(const int32_t* table, int64_t p, int64_t bs) {
  return (int64_t)table[p / bs] * bs + p % bs;
}

/*
 * One attention output row for one query head: the query attends to logical
 * keys 0 .. n_keys-1 of one sequence, kv head g.  `w` is scratch of n_keys
 * doubles.  Writes head_dim doubles to `out`.
 */
static void attend_row(const uint16_t* qrow, const uint16_t* k_cache, const uint16_t* v_cache,
                       const int32_t* table, int64_t n_keys, int64_t bs, int64_t hkv,
                       int64_t hd, int64_t g, double scale, double* w, double* out) {
  double m = -INFINITY;
  for (int64_t t = 0; t < n_keys; ++t) {
    const int64_t base = (slot_of(table, t, bs) * hkv + g) * hd;
    double dot = 0.0;
    for (int64_t d = 0; d < hd; ++d) dot += widen_bf16(qrow[d]) * widen_bf16(k_cache[base + d]);
    w[t] = scale * dot;
    if (w[t] > m) m = w[t];
  }
  double denom = 0.0;
  for (int64_t t = 0; t < n_keys; ++t) {
    w[t] = exp(w[t] - m);
    denom += w[t];
  }
  for (int64_t d = 0; d < hd; ++d) out[d] = 0.0;
  for (int64_t t = 0; t < n_keys; ++t) {
    const int64_t base = (slot_of(table, t, bs) * hkv + g) * hd;
    const double p = w[t] / denom;
    for (int64_t d = 0; d < hd; ++d) out[d] += p * widen_bf16(v_cache[base + d]);
  }
}

static int check_table(const int32_t* table, int64_t n_keys, int64_t bs, int64_t num_blocks) {
  const int64_t nb = (n_keys + bs - 1) / bs;
  for (int64_t i = 0; i < nb; ++i)
    if (table[i] < 0 || table[i] >= num_blocks) return ORACLE_ERR_RANGE;
  return ORACLE_OK;
}

/*
 * Decode: one query token per sequence.  out[b, h, :] is the softmax
 * attention of q[b, h, :] over the first context_lens[b] tokens of sequence
 * b (the newly written token included).  context_lens[b] == 0 gives zeros.
 * q is [batch, hq, hd]; out is [batch, hq, hd] doubles.
 */
int pkv_oracle_paged_attn_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                 const int32_t* context_lens, const int32_t* block_tables,
                                 int64_t max_blocks_per_seq, int64_t batch, int64_t hq, int64_t hkv,
                                 int64_t hd, int64_t bs, int64_t num_blocks, double scale,
                                 double* out) {
  if (batch < 0 || hq <= 0 || hkv <= 0 || hd <= 0 || bs <= 0 || hq % hkv) return ORACLE_ERR_ARG;
  int64_t max_len = 0;
  for (int64_t b = 0; b < batch; ++b) {
    const int64_t L = context_lens[b];
    if (L < 0 || L > max_blocks_per_seq * bs) return ORACLE_ERR_RANGE;
    if (check_table(block_tables + b * max_blocks_per_seq, L, bs, num_blocks)) return ORACLE_ERR_RANGE;
    if (L > max_len) max_len = L;
  }
  const int64_t group = hq / hkv;
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!w) {
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < batch * hq; ++bh) {
      const int64_t b = bh / hq, h = bh % hq;
      double* o = out + bh * hd;
      const int64_t L = context_lens[b];
      if (L == 0 || !w) {
        for (int64_t d = 0; d < hd; ++d) o[d] = 0.0;
        continue;
      }
      attend_row(q + bh * hd, k_cache, v_cache, block_tables + b * max_blocks_per_seq, L, bs, hkv,
                 hd, h / group, scale, w, o);
    }
    free(w);
  }
  return err;
}

/*
 * Varlen prefill.  Sequence i owns query rows cu_seqlens_q[i] ..
 * cu_seqlens_q[i+1]-1 (n_i rows) and L_i = cu_seqlens_k[i+1]-cu_seqlens_k[i]
 * keys in the cache; c_i = L_i - n_i must be >= 0.  Query row j of sequence i
 * sees keys 0 .. c_i + j.  q is [total_q, hq, hd]; out is [total_q, hq, hd]
 * doubles.
 *
 * If `rows` is non-NULL only the n_rows listed global query rows are computed
 * (for large inputs); other rows of `out` are left untouched.
 */
int pkv_oracle_paged_attn_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  const int32_t* block_tables, int64_t max_blocks_per_seq,
                                  int64_t num_seqs, int64_t hq, int64_t hkv, int64_t hd, int64_t bs,
                                  int64_t num_blocks, double scale, const int64_t* rows,
                                  int64_t n_rows, double* out) {
  if (num_seqs < 0 || hq <= 0 || hkv <= 0 || hd <= 0 || bs <= 0 || hq % hkv) return ORACLE_ERR_ARG;
  if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0) return ORACLE_ERR_ARG;
  int64_t max_len = 0;
  for (int64_t i = 0; i < num_seqs; ++i) {
    const int64_t n = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    const int64_t L = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
    if (n < 0 || L < n || L > max_blocks_per_seq * bs) return ORACLE_ERR_RANGE;
    if (check_table(block_tables + i * max_blocks_per_seq, L, bs, num_blocks)) return ORACLE_ERR_RANGE;
    if (L > max_len) max_len = L;
  }
  const int64_t total_q = cu_seqlens_q[num_seqs];
  const int64_t count = rows ? n_rows : total_q;
  for (int64_t r = 0; r < count; ++r) {
    const int64_t row = rows ? rows[r] : r;
    if (row < 0 || row >= total_q) return ORACLE_ERR_RANGE;
  }
  const int64_t group = hq / hkv;
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!w) {
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < count * hq; ++rh) {
      const int64_t row = rows ? rows[rh / hq] : rh / hq;
      const int64_t h = rh % hq;
      if (!w) continue;
      /* the sequence that owns this query row */
      int64_t i = 0;
      while (cu_seqlens_q[i + 1] <= row) ++i;
      const int64_t n = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
      const int64_t L = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
      const int64_t j = row - cu_seqlens_q[i];
      const int64_t n_keys = (L - n) + j + 1;
      attend_row(q + (row * hq + h) * hd, k_cache, v_cache, block_tables + i * max_blocks_per_seq,
                 n_keys, bs, hkv, hd, h / group, scale, w, out + (row * hq + h) * hd);
    }
    free(w);
  }
  return err;
}

/*
 * Exponential-race sampler (page section "其余部分": temperature-only
 * sampling; the probabilities are divided by exponentially distributed
 * random numbers and the largest quotient wins, which samples each token with
 * its probability; temperature 0 is not allowed).
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC 2011), a counter-based generator.  For row
 * b and token i the 32-bit word is output word (i % 4) of
 * Philox(counter = {i / 4, b, offset_lo, offset_hi}, key = {seed_lo, seed_hi});
 * U = ((word >> 9) + 0.5) / 2^23 lies strictly inside (0, 1) and
 * E = -ln(U) ~ Exp(1).
 *
 * Steps, per row, in double: p = softmax(logits / T) (maximum subtracted),
 * E_i from the generator, token = the first i maximising p_i / E_i.
 * T must be finite and > 0; otherwise the row's token is -1.
 */
static uint32_t mulhi32(uint32_t a, uint32_t b) { return (uint32_t)(((uint64_t)a * b) >> 32); }

void pkv_oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k[0] += 0x9E3779B9u;
      k[1] += 0xBB67AE85u;
    }
    const uint32_t hi0 = mulhi32(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
    const uint32_t hi1 = mulhi32(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k[0], n1 = lo1, n2 = hi0 ^ c[3] ^ k[1], n3 = lo0;
    c[0] = n0;
    c[1] = n1;
    c[2] = n2;
    c[3] = n3;
  }
  out[0] = c[0];
  out[1] = c[1];
  out[2] = c[2];
  out[3] = c[3];
}

/* The uniform U in (0, 1) of row b, token i. */
double pkv_oracle_uniform(int64_t b, int64_t i, uint64_t seed, uint64_t offset) {
  const uint32_t ctr[4] = {(uint32_t)(i / 4), (uint32_t)b, (uint32_t)offset, (uint32_t)(offset >> 32)};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  pkv_oracle_philox4x32_10(ctr, key, w);
  return ((double)(w[i % 4] >> 9) + 0.5) / 8388608.0;
}

/*
 * logits [batch, vocab] float32 (row stride in elements), temperatures
 * [batch]; writes tokens [batch] and, if `scores` is not NULL, the log-space
 * score log(p_i) - log(E_i) of every token (for near-tie checks).
 */
int pkv_oracle_sample(const float* logits, int64_t row_stride, const float* temperatures, int64_t batch,
                      int64_t vocab, uint64_t seed, uint64_t offset, int32_t* tokens, double* scores) {
  if (batch < 0 || vocab <= 0 || row_stride < vocab) return ORACLE_ERR_ARG;
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
    if (!p) {
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b) {
      const double T = temperatures[b];
      if (!p || !(T > 0.0) || !isfinite(T)) {
        tokens[b] = -1;
        continue;
      }
      const float* l = logits + b * row_stride;
      double m = -INFINITY;
      for (int64_t i = 0; i < vocab; ++i)
        if ((double)l[i] / T > m) m = (double)l[i] / T;
      double sum = 0.0;
      for (int64_t i = 0; i < vocab; ++i) {
        p[i] = exp((double)l[i] / T - m);
        sum += p[i];
      }
      int64_t best = 0;
      double best_q = -1.0;
      for (int64_t i = 0; i < vocab; ++i) {
        const double E = -log(pkv_oracle_uniform(b, i, seed, offset));
        const double q = (p[i] / sum) / E;
        if (q > best_q) {
          best_q = q;
          best = i;
        }
        if (scores) scores[b * vocab + i] = log(p[i] / sum) - log(E);
      }
      tokens[b] = (int32_t)best;
    }
    free(p);
  }
  return err;
}
