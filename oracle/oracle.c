/*
 * oracle.c -- plain fp64 CPU oracle for unified paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it reads the same stored input values (fp32 or bf16 bit
 * patterns) and widens them to double itself.
 *
 * What it computes follows the definition on the pages, written out with no
 * blocking, fusion or reordering:
 *
 *   "vLLM Triton attention backend deep dive", section "Technical
 *   implementation of paged attention": the KV cache is paged; the kernel
 *   walks the query tokens, the query/KV heads and the pages of the cache to
 *   form attention scores.  Section "Q-block optimisation": several query heads
 *   share one KV head (GQA).
 *
 *   "vLLM AMD ROCm attention backend optimisation", section "Mixed inference
 *   workload challenge": one continuous batch holds prefill, extend (more
 *   prompt tokens on a partly built cache) and decode (one token) requests.
 *
 *   Same page, section "AITER MLA backend / hybrid processing strategy": the
 *   absorbed MLA decode works directly on the 576-wide compressed latent.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - query i of request s sits at absolute position prefix_s + i, where
 *     prefix_s = seq_len_s - q_len_s; it sees positions 0..prefix_s+i
 *     (bottom-right causal alignment);
 *   - the new tokens' K/V are already in the cache (seq_len includes them);
 *   - head h reads KV head floor(h / G), G = num_heads / num_kv_heads;
 *   - absorbed MLA: the value of a cached latent row is its first
 *     kv_lora_rank entries; the trailing rope entries only enter the score;
 *   - model variants ("vLLM Triton attention backend deep dive", section
 *     "Usage scenarios": ALiBi sqrt, sink tokens, GPT-OSS behaviour), which
 *     the pages name but do not define:
 *       sliding window W (GPT-OSS local attention): the query at position i
 *       sees only the W most recent positions, i - W < j <= i;
 *       ALiBi (linear biases, one slope m_h per head, slopes supplied by
 *       the caller): score_ij += -m_h * (i - j);
 *       ALiBi sqrt: score_ij += -m_h * sqrt(i - j).
 *
 * Softmax is the two-pass textbook form: max, then exp(s - max) / sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_BAD_ARGS 1
#define OR_BAD_METADATA 2
#define OR_NO_MEMORY 3

#define OR_F32 0
#define OR_BF16 1

/* Widen one stored element to double.  bf16 is the upper half of an IEEE
 * binary32, so the widening is exact. */
static double widen(const void *base, int dtype, size_t idx) {
  if (dtype == OR_F32) return (double)((const float *)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Physical cache row of logical KV position j of request s, through the
 * request's block table: page = table[s][j / bs], slot = j mod bs.
 * Returns -1 when the page id is outside the pool. */
static long long cache_row(const int32_t *block_table, int max_blocks_per_seq,
                           int num_blocks, int block_size, int s, long long j) {
  long long logical_page = j / block_size;
  if (logical_page >= max_blocks_per_seq) return -1;
  int32_t page = block_table[(size_t)s * max_blocks_per_seq + logical_page];
  if (page < 0 || page >= num_blocks) return -1;
  return (long long)page * block_size + (j % block_size);
}

/* Attention for one query row over the visible KV positions in
 * [kv_begin, kv_end) of request s.
 *   score_j = scale * sum_d q[d] * K_j[d] + bias_j (d < dk)
 *   bias_j  = -slope * (qpos - j), or -slope * sqrt(qpos - j) with bias_sqrt
 *             (ALiBi; slope 0 adds -0.0, which changes no score)
 *   p_j     = exp(score_j - max) / sum exp(score - max)
 *   out[e]  = sum_j p_j * V_j[e]                   (e < dv)
 * K_j[d] = kc[row_j*kstride + koff + d], V_j[e] = vc[row_j*vstride + voff + e].
 * Writes *lse = max + log(sum) (natural log); an empty range gives
 * out = 0 and lse = -inf.  `scores` has room for kv_end - kv_begin values. */
static int attend_row(const double *qrow, int dk, int dv,
                      const void *kc, const void *vc, int dtype,
                      size_t kstride, size_t koff, size_t vstride, size_t voff,
                      const int32_t *block_table, int max_blocks_per_seq,
                      int num_blocks, int block_size, int s,
                      long long kv_begin, long long kv_end, double scale,
                      double slope, int bias_sqrt, long long qpos,
                      double *scores, double *out, double *lse) {
  long long n = kv_end - kv_begin;
  for (int e = 0; e < dv; ++e) out[e] = 0.0;
  if (n <= 0) {
    *lse = -INFINITY;
    return OR_OK;
  }
  double mx = -INFINITY;
  for (long long t = 0; t < n; ++t) {
    long long row = cache_row(block_table, max_blocks_per_seq, num_blocks,
                              block_size, s, kv_begin + t);
    if (row < 0) return OR_BAD_METADATA;
    double acc = 0.0;
    for (int d = 0; d < dk; ++d)
      acc += qrow[d] * widen(kc, dtype, (size_t)row * kstride + koff + d);
    const double dist = (double)(qpos - (kv_begin + t));
    const double bias = bias_sqrt ? -slope * sqrt(dist) : -slope * dist;
    scores[t] = scale * acc + bias;
    if (scores[t] > mx) mx = scores[t];
  }
  double denom = 0.0;
  for (long long t = 0; t < n; ++t) {
    scores[t] = exp(scores[t] - mx);
    denom += scores[t];
  }
  for (long long t = 0; t < n; ++t) {
    long long row = cache_row(block_table, max_blocks_per_seq, num_blocks,
                              block_size, s, kv_begin + t);
    double p = scores[t] / denom;
    for (int e = 0; e < dv; ++e)
      out[e] += p * widen(vc, dtype, (size_t)row * vstride + voff + e);
  }
  *lse = mx + log(denom);
  return OR_OK;
}

/* Request index of every query token, from query_start_loc. */
static int token_owner(const int32_t *qsl, int num_seqs, int num_tokens,
                       int32_t *owner) {
  if (qsl[0] != 0 || qsl[num_seqs] != num_tokens) return OR_BAD_METADATA;
  for (int s = 0; s < num_seqs; ++s) {
    if (qsl[s + 1] < qsl[s]) return OR_BAD_METADATA;
    for (int t = qsl[s]; t < qsl[s + 1]; ++t) owner[t] = s;
  }
  return OR_OK;
}

/*
 * Unified paged attention over a mixed batch, restricted to the KV window
 * [kv_begin, kv_end) of every request (kv_begin = 0, kv_end = INT64_MAX gives
 * the full definition).  The restriction exists only so that tests can form
 * split-KV partial results; it does not change the definition.
 * sliding_window > 0: query i of a request (absolute position p) sees only
 * positions p - sliding_window < j <= p.  alibi_slopes (one per query head,
 * or NULL) adds -slope_h * (p - j), or -slope_h * sqrt(p - j) when
 * alibi_sqrt is set, to every score of head h.
 *
 *   q        [num_tokens, num_heads, head_dim]
 *   k_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *   v_cache  same shape as k_cache
 *   out      [num_tokens, num_heads, head_dim]  (double)
 *   lse      [num_tokens, num_heads] (double, may be NULL)
 *   rows     optional list of (token * num_heads + head) to compute; NULL = all
 */
int oracle_paged_attention_ex(
    const void *q, const void *k_cache, const void *v_cache, int dtype,
    const int32_t *block_table, const int32_t *seq_lens,
    const int32_t *query_start_loc, int num_seqs, int num_tokens,
    int num_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, double scale,
    long long kv_begin, long long kv_end, long long sliding_window,
    const double *alibi_slopes, int alibi_sqrt, const int64_t *rows,
    long long num_rows, double *out, double *lse) {
  if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
      sliding_window < 0 || (dtype != OR_F32 && dtype != OR_BF16))
    return OR_BAD_ARGS;
  const int group = num_heads / num_kv_heads;
  int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (num_tokens + 1));
  if (!owner) return OR_NO_MEMORY;
  int rc = token_owner(query_start_loc, num_seqs, num_tokens, owner);
  long long max_ctx = 1;
  for (int s = 0; rc == OR_OK && s < num_seqs; ++s) {
    int q_len = query_start_loc[s + 1] - query_start_loc[s];
    if (seq_lens[s] < q_len) rc = OR_BAD_METADATA;
    if (seq_lens[s] > max_ctx) max_ctx = seq_lens[s];
  }
  if (rc != OR_OK) {
    free(owner);
    return rc;
  }
  long long total = rows ? num_rows : (long long)num_tokens * num_heads;
  const size_t kstride = (size_t)num_kv_heads * head_dim;
  int status = OR_OK;

#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_ctx);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
    if (!scores || !qrow) {
#pragma omp atomic write
      status = OR_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (long long r = 0; r < total; ++r) {
      if (!scores || !qrow) continue;
      long long flat = rows ? rows[r] : r;
      int tok = (int)(flat / num_heads);
      int h = (int)(flat % num_heads);
      int s = owner[tok];
      int q_len = query_start_loc[s + 1] - query_start_loc[s];
      long long prefix = (long long)seq_lens[s] - q_len;
      long long i = tok - query_start_loc[s];
      /* Visible positions: 0 .. prefix + i (causal, bottom-right), and with
       * a sliding window only the last sliding_window of them. */
      long long qpos = prefix + i;
      long long lo = kv_begin > 0 ? kv_begin : 0;
      if (sliding_window > 0 && qpos - sliding_window + 1 > lo) lo = qpos - sliding_window + 1;
      long long hi = qpos + 1;
      if (kv_end < hi) hi = kv_end;
      double slope = alibi_slopes ? alibi_slopes[h] : 0.0;
      int kvh = h / group;
      for (int d = 0; d < head_dim; ++d)
        qrow[d] = widen(q, dtype, (size_t)flat * head_dim + d);
      double row_lse;
      int rr = attend_row(qrow, head_dim, head_dim, k_cache, v_cache, dtype,
                          kstride, (size_t)kvh * head_dim, kstride,
                          (size_t)kvh * head_dim, block_table,
                          max_blocks_per_seq, num_blocks, block_size, s, lo, hi,
                          scale, slope, alibi_sqrt, qpos, scores,
                          out + (size_t)flat * head_dim, &row_lse);
      if (lse) lse[flat] = row_lse;
      if (rr != OR_OK) {
#pragma omp atomic write
        status = rr;
      }
    }
    free(scores);
    free(qrow);
  }
  free(owner);
  return status;
}

int oracle_paged_attention_window(
    const void *q, const void *k_cache, const void *v_cache, int dtype,
    const int32_t *block_table, const int32_t *seq_lens,
    const int32_t *query_start_loc, int num_seqs, int num_tokens,
    int num_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, double scale,
    long long kv_begin, long long kv_end, const int64_t *rows,
    long long num_rows, double *out, double *lse) {
  return oracle_paged_attention_ex(
      q, k_cache, v_cache, dtype, block_table, seq_lens, query_start_loc,
      num_seqs, num_tokens, num_heads, num_kv_heads, head_dim, block_size,
      max_blocks_per_seq, num_blocks, scale, kv_begin, kv_end, 0, NULL, 0,
      rows, num_rows, out, lse);
}

int oracle_paged_attention(const void *q, const void *k_cache,
                           const void *v_cache, int dtype,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *query_start_loc, int num_seqs,
                           int num_tokens, int num_heads, int num_kv_heads,
                           int head_dim, int block_size,
                           int max_blocks_per_seq, int num_blocks,
                           double scale, const int64_t *rows,
                           long long num_rows, double *out) {
  return oracle_paged_attention_window(
      q, k_cache, v_cache, dtype, block_table, seq_lens, query_start_loc,
      num_seqs, num_tokens, num_heads, num_kv_heads, head_dim, block_size,
      max_blocks_per_seq, num_blocks, scale, 0, INT64_MAX, rows, num_rows, out,
      NULL);
}

/*
 * Log-sum-exp merge of P partial results of one query row ("vLLM Triton
 * attention backend deep dive", section "Parallel tiled softmax (3D kernel)":
 * instances compute partial results over parts of the KV walk and a second
 * launch combines them; "vLLM AMD ROCm attention backend optimisation",
 * section "Chunked context processing": chunks are combined by an LSE merge).
 *
 * Each partial p is normalised by its own softmax sum and carries
 * lse_p = max_p + log(sum_p).  With M = max_p lse_p:
 *   w_p = exp(lse_p - M) / sum_q exp(lse_q - M),  out = sum_p w_p * O_p.
 * Partials with lse = -inf (empty KV range) get weight 0.  If every partial is
 * empty the output is 0 and *lse_out = -inf.
 */
int oracle_lse_merge(int num_parts, int dim, const double *partial_out,
                     const double *partial_lse, double *out, double *lse_out) {
  if (num_parts < 0 || dim <= 0) return OR_BAD_ARGS;
  double m = -INFINITY;
  for (int p = 0; p < num_parts; ++p)
    if (partial_lse[p] > m) m = partial_lse[p];
  for (int e = 0; e < dim; ++e) out[e] = 0.0;
  if (m == -INFINITY) {
    if (lse_out) *lse_out = -INFINITY;
    return OR_OK;
  }
  double denom = 0.0;
  for (int p = 0; p < num_parts; ++p) denom += exp(partial_lse[p] - m);
  for (int p = 0; p < num_parts; ++p) {
    double w = exp(partial_lse[p] - m) / denom;
    if (w == 0.0) continue;
    for (int e = 0; e < dim; ++e) out[e] += w * partial_out[(size_t)p * dim + e];
  }
  if (lse_out) *lse_out = m + log(denom);
  return OR_OK;
}

/*
 * Absorbed MLA decode ("vLLM AMD ROCm attention backend optimisation",
 * section "AITER MLA backend: optimised for DeepSeek" and its "hybrid
 * processing strategy"): every query head attends directly to the compressed
 * latent rows of one shared cache.
 *   q        [num_seqs, num_heads, kv_lora_rank + rope_dim]  (one token each)
 *   kv_cache [num_blocks, block_size, kv_lora_rank + rope_dim]
 *   out      [num_seqs, num_heads, kv_lora_rank]  (double)
 * score_j = scale * <q_h, c_j> over all latent + rope entries; the value of
 * row j is c_j[0 : kv_lora_rank].  Every position 0..seq_len-1 is visible.
 * rows: optional list of (seq * num_heads + head); NULL = all.
 */
int oracle_mla_decode(const void *q, const void *kv_cache, int dtype,
                      const int32_t *block_table, const int32_t *seq_lens,
                      int num_seqs, int num_heads, int kv_lora_rank,
                      int rope_dim, int block_size, int max_blocks_per_seq,
                      int num_blocks, double scale, const int64_t *rows,
                      long long num_rows, double *out) {
  if (num_seqs < 0 || num_heads <= 0 || kv_lora_rank <= 0 || rope_dim < 0 ||
      block_size <= 0 || (dtype != OR_F32 && dtype != OR_BF16))
    return OR_BAD_ARGS;
  const int dk = kv_lora_rank + rope_dim;
  long long max_ctx = 1;
  for (int s = 0; s < num_seqs; ++s) {
    if (seq_lens[s] < 1) return OR_BAD_METADATA;
    if (seq_lens[s] > max_ctx) max_ctx = seq_lens[s];
  }
  long long total = rows ? num_rows : (long long)num_seqs * num_heads;
  int status = OR_OK;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_ctx);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)dk);
    if (!scores || !qrow) {
#pragma omp atomic write
      status = OR_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (long long r = 0; r < total; ++r) {
      if (!scores || !qrow) continue;
      long long flat = rows ? rows[r] : r;
      int s = (int)(flat / num_heads);
      for (int d = 0; d < dk; ++d)
        qrow[d] = widen(q, dtype, (size_t)flat * dk + d);
      double row_lse;
      int rr = attend_row(qrow, dk, kv_lora_rank, kv_cache, kv_cache, dtype,
                          (size_t)dk, 0, (size_t)dk, 0, block_table,
                          max_blocks_per_seq, num_blocks, block_size, s, 0,
                          seq_lens[s], scale, 0.0, 0, 0, scores,
                          out + (size_t)flat * kv_lora_rank, &row_lse);
      if (rr != OR_OK) {
#pragma omp atomic write
        status = rr;
      }
    }
    free(scores);
    free(qrow);
  }
  return status;
}

/* Dense gather of K rows through the block table, the indexing step alone:
 * dense[s][j][:] = k_cache[block_table[s][j / bs]][j mod bs][:] for
 * j < seq_lens[s], copied as raw element bits (row_elems elements of
 * elem_bytes each).  Positions at or beyond seq_len are left untouched. */
int oracle_gather_rows(const void *k_cache, int elem_bytes, int row_elems,
                       const int32_t *block_table, const int32_t *seq_lens,
                       int num_seqs, int max_blocks_per_seq, int num_blocks,
                       int block_size, long long max_seq_len, void *dense) {
  if (elem_bytes <= 0 || row_elems <= 0 || block_size <= 0) return OR_BAD_ARGS;
  const size_t row_bytes = (size_t)elem_bytes * row_elems;
  for (int s = 0; s < num_seqs; ++s) {
    if (seq_lens[s] > max_seq_len) return OR_BAD_METADATA;
    for (long long j = 0; j < seq_lens[s]; ++j) {
      long long row = cache_row(block_table, max_blocks_per_seq, num_blocks,
                                block_size, s, j);
      if (row < 0) return OR_BAD_METADATA;
      memcpy((char *)dense + ((size_t)s * max_seq_len + j) * row_bytes,
             (const char *)k_cache + (size_t)row * row_bytes, row_bytes);
    }
  }
  return OR_OK;
}

/* Threads an OpenMP parallel region of this library starts (1 without
 * OpenMP): the host cores the timed oracle actually uses. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
