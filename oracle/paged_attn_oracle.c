/*
 * fp64 CPU oracle for paged GQA attention (decode and speculative verify).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this file's library.  It shares no code, header, table or helper with the CUDA
 * path: it is the plain definition of attention written out, slowly, in double precision.
 *
 * What it computes, and where the pages define it:
 *   - Attention of one query over past tokens: score each cached Key against the Query, turn
 *     the scores into weights with a softmax, and sum the Values with those weights
 *     (studybook fde-roadmap ch.10, section 10.3.1).  Scores are scaled by the caller's
 *     `scale` (1/sqrt(d) in every workload).
 *   - GQA: query heads are split into groups and each group shares one Key/Value head
 *     (section 10.1.2).  Reading: the groups are contiguous, query head h uses kv head
 *     h / (Hq / Hkv).
 *   - Paged KV cache: logical block j / bs of a sequence lives in physical block
 *     block_table[b][j / bs], slot j % bs (section 10.4.2 and figure 10.4.2; aegloslab
 *     servingai 5.3.7).  Layout [num_blocks, Hkv, bs, d].
 *   - Speculative verify: the q_len new tokens are the last q_len tokens of the context and
 *     row i sees every token up to and including itself (causal mask; sirzzang "Speculative
 *     Decoding", parallel verification and its causal-mask figure).  With context length L,
 *     row i sees n = L - q_len + i + 1 tokens.  Decode is the case q_len = 1.
 *   - fp8 KV: each stored E4M3 byte is decoded exactly from the OCP 8-bit floating point
 *     definition (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 *     S.1111.111 is NaN) and multiplied by the per-(block, kv head) scale, the symmetric
 *     scale quantisation of section 10.8.2 read backwards.
 *
 * The bf16 inputs are decoded exactly (a bf16 is the top half of an IEEE binary32), so every
 * quantity below is the fp64 value of the stored data.  There is no tiling, no online softmax
 * and no reordering: scores are materialised, the max subtracted, exponentials summed.
 * Readings where the pages are silent: a row that sees no token (n <= 0) yields zeros.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,
  ORACLE_ERR_NOMEM = 4,
  ORACLE_ERR_BLOCK_ID = 5,
};

/* bf16 -> double: the bf16 bits are the upper 16 bits of a binary32. */
double pa_oracle_bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3 -> double: normal (-1)^s * 2^(e-7) * (1 + m/8); subnormal (-1)^s * 2^-6 * m/8. */
double pa_oracle_e4m3_to_double(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

static double kv_value(const void* cache, int kv_fp8, size_t idx) {
  if (kv_fp8) return pa_oracle_e4m3_to_double(((const uint8_t*)cache)[idx]);
  return pa_oracle_bf16_to_double(((const uint16_t*)cache)[idx]);
}

/*
 * out[b, i, h, :] for every sequence b in `seqs` (all sequences when seqs == NULL).
 *   q            [B, q_len, Hq, d]         bf16 bits
 *   k/v cache    [num_blocks, Hkv, bs, d]  bf16 bits, or E4M3 bytes when kv_fp8
 *   k/v scale    [num_blocks, Hkv]         fp32 (kv_fp8 only)
 *   block_table  [B, max_blocks_per_seq]
 *   context_lens [B]
 *   out          [B, q_len, Hq, d]         fp64; rows of sequences not in `seqs` are untouched
 * Returns 0, or ORACLE_ERR_* (a block id outside [0, num_blocks) is an error).
 */
/*
 * Same as pa_oracle_attention, with an optional tree mask (tree attention: the draft tokens form
 * a tree of candidate branches verified in one forward, each node attending to its ancestors;
 * aegloslab servingai 5.3.13).  tree_mask[b * q_len + i] bit t set means new-token row i sees
 * new token t; every token before the q_len new ones stays visible.  tree_mask == NULL is the
 * causal mask (bits 0..i).
 */
int pa_oracle_attention_masked(const uint16_t* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, int kv_fp8,
                               const int32_t* block_table, const int32_t* context_lens,
                               const uint32_t* tree_mask, int num_seqs, int max_blocks_per_seq,
                               int num_blocks, int q_len, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, double scale, const int32_t* seqs,
                               int num_selected, double* out, int num_threads) {
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out) return ORACLE_ERR_ARG;
  if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 ||
      block_size < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return ORACLE_ERR_ARG;
  if (num_q_heads % num_kv_heads) return ORACLE_ERR_ARG;
  if (kv_fp8 && (!k_scale || !v_scale)) return ORACLE_ERR_ARG;
  if (tree_mask && q_len > 32) return ORACLE_ERR_ARG;
  const int group = num_q_heads / num_kv_heads;
  const int nsel = seqs ? num_selected : num_seqs;
  for (int s = 0; s < nsel; ++s) {
    int b = seqs ? seqs[s] : s;
    if (b < 0 || b >= num_seqs) return ORACLE_ERR_ARG;
    int L = context_lens[b];
    if (L < 0 || L > max_blocks_per_seq * block_size) return ORACLE_ERR_ARG;
    for (int j = 0; j < (L + block_size - 1) / block_size; ++j) {
      int pb = block_table[(size_t)b * max_blocks_per_seq + j];
      if (pb < 0 || pb >= num_blocks) return ORACLE_ERR_BLOCK_ID;
    }
  }
  const long total = (long)nsel * q_len * num_q_heads;
  int err = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (long w = 0; w < total; ++w) {
    const int h = (int)(w % num_q_heads);
    const int i = (int)((w / num_q_heads) % q_len);
    const int s = (int)(w / ((long)num_q_heads * q_len));
    const int b = seqs ? seqs[s] : s;
    const int L = context_lens[b];
    const int n = L - q_len + i + 1; /* tokens row i may attend to (causal) */
    const int g = h / group;
    double* o = out + (((size_t)b * q_len + i) * num_q_heads + h) * head_dim;
    const uint16_t* qrow = q + (((size_t)b * q_len + i) * num_q_heads + h) * head_dim;
    for (int c = 0; c < head_dim; ++c) o[c] = 0.0;
    /* visible tokens: the causal prefix, or (tree) every earlier token plus the new tokens whose
       mask bit is set */
    const int first_new = L - q_len;
    const uint32_t mrow = tree_mask ? tree_mask[(size_t)b * q_len + i] : 0u;
    const int nscan = tree_mask ? L : n;
    int nvis = 0;
    for (int j = 0; j < nscan; ++j)
      if (!tree_mask || j < first_new || ((mrow >> (j - first_new)) & 1u)) ++nvis;
    if (nvis <= 0 || nscan <= 0) continue;
    double* sc = (double*)malloc(sizeof(double) * (size_t)nscan);
    if (!sc) {
      err |= 1;
      continue;
    }
    /* scores s_j = scale * q . k_j for the visible j (the others are never summed) */
    for (int j = 0; j < nscan; ++j) {
      if (tree_mask && j >= first_new && !((mrow >> (j - first_new)) & 1u)) {
        sc[j] = -INFINITY;
        continue;
      }
      const int pb = block_table[(size_t)b * max_blocks_per_seq + j / block_size];
      const int t = j % block_size;
      const size_t base = (((size_t)pb * num_kv_heads + g) * block_size + t) * head_dim;
      const double ks = kv_fp8 ? (double)k_scale[(size_t)pb * num_kv_heads + g] : 1.0;
      double dot = 0.0;
      for (int c = 0; c < head_dim; ++c)
        dot += pa_oracle_bf16_to_double(qrow[c]) * (kv_value(k_cache, kv_fp8, base + c) * ks);
      sc[j] = scale * dot;
    }
    /* softmax weights e^{s_j - max} / sum, then the weighted sum of values */
    double mx = -INFINITY;
    for (int j = 0; j < nscan; ++j)
      if (sc[j] > mx) mx = sc[j];
    double denom = 0.0;
    for (int j = 0; j < nscan; ++j) {
      sc[j] = (sc[j] == -INFINITY) ? 0.0 : exp(sc[j] - mx);
      denom += sc[j];
    }
    for (int j = 0; j < nscan; ++j) {
      if (sc[j] == 0.0) continue;
      const int pb = block_table[(size_t)b * max_blocks_per_seq + j / block_size];
      const int t = j % block_size;
      const size_t base = (((size_t)pb * num_kv_heads + g) * block_size + t) * head_dim;
      const double vs = kv_fp8 ? (double)v_scale[(size_t)pb * num_kv_heads + g] : 1.0;
      const double wj = sc[j] / denom;
      for (int c = 0; c < head_dim; ++c) o[c] += wj * (kv_value(v_cache, kv_fp8, base + c) * vs);
    }
    free(sc);
  }
  return err ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Causal form (decode is q_len = 1). */
int pa_oracle_attention(const uint16_t* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, int kv_fp8,
                        const int32_t* block_table, const int32_t* context_lens, int num_seqs,
                        int max_blocks_per_seq, int num_blocks, int q_len, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, double scale,
                        const int32_t* seqs, int num_selected, double* out, int num_threads) {
  return pa_oracle_attention_masked(q, k_cache, v_cache, k_scale, v_scale, kv_fp8, block_table,
                                    context_lens, NULL, num_seqs, max_blocks_per_seq, num_blocks,
                                    q_len, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                    seqs, num_selected, out, num_threads);
}

int pa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
