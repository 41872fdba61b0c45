/*
 * Reference oracle for single-token decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain CPU definition that
 * the CUDA library is checked against.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark load it.  The product path never
 * links, calls or falls back to it, and it shares no code, header, table or
 * constant with the CUDA sources.
 *
 * What it computes (issue "ROCm gfx1200: PagedAttnOnline is 8.1x slower per
 * call ...", section "Where to look": a decode kernel that does online
 * softmax over a KV cache read in NHD layout through strides, after a
 * per-request lookup of the sequence's pages; PR "perf(cuda): head_dim-128
 * arm for the warp-split-KV decode kernel", commit message: 32-token pages,
 * GQA-fused query heads, an optional sliding window):
 *
 *   for every sequence b and every query head i (kv head h = i / g,
 *   g = num_q_heads / num_kv_heads):
 *     L  = context_lens[b]
 *     t0 = window > 0 ? max(0, L - window) : 0
 *     for every token t in [t0, L):
 *        page = block_tables[b][t / block_size], slot = t % block_size
 *        k_t  = k_cache[page][slot][h][:],  v_t = v_cache[page][slot][h][:]
 *        s_t  = scale * sum_d q[b][i][d] * k_t[d]
 *     out[b][i][:] = sum_t softmax(s)_t * v_t
 *
 * Online softmax (what the kernels on those pages use) is an exact
 * reformulation of this; the oracle takes the plain two-pass form instead:
 * pass 1 finds M = max_t s_t, pass 2 forms Z = sum_t exp(s_t - M) and
 * sum_t exp(s_t - M) v_t, and the row is their ratio.  Every stored element is
 * widened exactly to double first (bf16 and binary32 are both subsets of
 * binary64) and all arithmetic is double.
 *
 * Readings taken where the pages are silent:
 *   - a quantised KV cache (FP8 E4M3 codes, a storage extension beyond the
 *     pages) stands for its code values times one scale per kv head, one set
 *     of scales for keys and one for values (oracle_decode_row_kv);
 *   - kv head of query head i is i / g (contiguous query groups);
 *   - cache layout [num_blocks][block_size][num_kv_heads][head_dim], head_dim
 *     contiguous ("NHD");
 *   - block table [num_seqs][max_blocks_per_seq] int32, row-major;
 *   - window W > 0 keeps the keys t with L - W <= t < L; W <= 0 keeps all;
 *   - a sequence with L == 0 yields a zero row;
 *   - multi-token decode: new token j of q_len sits at position L - q_len + j
 *     and attends causally to the tokens up to and including itself
 *     (oracle_decode_multi_row).
 *
 * Error behaviour: returns ORACLE_OK (0) or a negative code, and writes
 * nothing for the offending row, when a context length is negative or longer
 * than the block-table row, or a page id lies outside [0, num_blocks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_CONTEXT (-2)
#define ORACLE_BAD_PAGE (-3)
#define ORACLE_NO_MEMORY (-4)

/* Storage codes for q / k_cache / v_cache elements. */
#define ORACLE_ELEM_BF16 0 /* uint16 bit patterns of bfloat16 */
#define ORACLE_ELEM_F32 1
#define ORACLE_ELEM_F64 2
#define ORACLE_ELEM_E4M3 3 /* uint8 codes of OCP FP8 E4M3 (KV cache storage only) */

/* bfloat16 is the upper half of an IEEE binary32 word: shifting the 16 stored
 * bits into the top of a 32-bit word gives that binary32 value exactly. */
static double widen_bf16(uint16_t bits) {
  uint32_t word = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &word, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 flavour: sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits.  Exponent field 0 holds the subnormals m/8 * 2^-6; the
 * pattern with all exponent and mantissa bits set is NaN; there is no
 * infinity, so exponent field 15 with mantissa 0..6 is an ordinary value
 * (the largest, 1.75 * 2^8 = 448). */
static double widen_e4m3(uint8_t code) {
  const int sign = code >> 7;
  const int ex = (code >> 3) & 0xF;
  const int man = code & 0x7;
  if (ex == 0xF && man == 0x7) return NAN;
  const double mag = (ex == 0) ? ldexp((double)man / 8.0, 1 - 7) : ldexp(1.0 + (double)man / 8.0, ex - 7);
  return sign ? -mag : mag;
}

/* Element e of an array stored with code `elem`, widened to double. */
static double element(const void* base, int elem, size_t e) {
  switch (elem) {
    case ORACLE_ELEM_BF16:
      return widen_bf16(((const uint16_t*)base)[e]);
    case ORACLE_ELEM_F32:
      return (double)((const float*)base)[e];
    case ORACLE_ELEM_E4M3:
      return widen_e4m3(((const uint8_t*)base)[e]);
    default:
      return ((const double*)base)[e];
  }
}

/* Flat index of element d of token slot `slot`, kv head h, in page `page`
 * of a cache laid out [num_blocks][block_size][num_kv_heads][head_dim]. */
static size_t cache_index(int page, int slot, int h, int d, int block_size,
                          int num_kv_heads, int head_dim) {
  return (((size_t)page * block_size + slot) * num_kv_heads + h) * head_dim + d;
}

/* One output row: sequence b, query head i.  out_row has head_dim doubles.
 * q is stored with code q_elem, the caches with kv_elem; a cache element of
 * kv head h stands for its stored value times k_scale[h] (keys) or
 * v_scale[h] (values), the per-head dequantisation scales of a quantised
 * cache (NULL: 1). */
int oracle_decode_row_kv(double* out_row, const void* q, int q_elem,
                         const void* k_cache, const void* v_cache, int kv_elem,
                         const double* k_scale, const double* v_scale,
                         const int32_t* block_tables, const int32_t* context_lens,
                         int num_seqs, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks_per_seq,
                         int num_blocks, double scale, int window, int b, int i) {
  if (!out_row || !q || !k_cache || !v_cache || !block_tables ||
      !context_lens || num_seqs <= 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      num_q_heads % num_kv_heads != 0 || b < 0 || b >= num_seqs || i < 0 ||
      i >= num_q_heads || q_elem < ORACLE_ELEM_BF16 || q_elem > ORACLE_ELEM_F64 ||
      kv_elem < ORACLE_ELEM_BF16 || kv_elem > ORACLE_ELEM_E4M3)
    return ORACLE_BAD_ARG;

  const int group = num_q_heads / num_kv_heads;
  const int h = i / group;
  const double ks = k_scale ? k_scale[h] : 1.0;
  const double vs = v_scale ? v_scale[h] : 1.0;
  const int L = context_lens[b];
  if (L < 0 || (long long)L > (long long)max_blocks_per_seq * block_size)
    return ORACLE_BAD_CONTEXT;
  const int t0 = (window > 0 && L - window > 0) ? L - window : 0;
  const int n = L - t0;

  for (int d = 0; d < head_dim; ++d) out_row[d] = 0.0;
  if (n == 0) return ORACLE_OK;

  /* Request lookup: physical page of every token in the range. */
  int* page_of = (int*)malloc(sizeof(int) * (size_t)n);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!page_of || !s) {
    free(page_of);
    free(s);
    return ORACLE_NO_MEMORY;
  }
  for (int j = 0; j < n; ++j) {
    const int t = t0 + j;
    const int page = block_tables[(size_t)b * max_blocks_per_seq + t / block_size];
    if (page < 0 || page >= num_blocks) {
      free(page_of);
      free(s);
      return ORACLE_BAD_PAGE;
    }
    page_of[j] = page;
  }

  /* Scores s_t = scale * <q_i, k_t>. */
  const size_t q_row = ((size_t)b * num_q_heads + i) * head_dim;
  for (int j = 0; j < n; ++j) {
    const int slot = (t0 + j) % block_size;
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d) {
      const double kd = element(k_cache, kv_elem,
                                cache_index(page_of[j], slot, h, d, block_size,
                                            num_kv_heads, head_dim)) * ks;
      dot += element(q, q_elem, q_row + d) * kd;
    }
    s[j] = scale * dot;
  }

  /* Pass 1: the row maximum. */
  double M = s[0];
  for (int j = 1; j < n; ++j)
    if (s[j] > M) M = s[j];

  /* Pass 2: normaliser and weighted sum of values. */
  double Z = 0.0;
  for (int j = 0; j < n; ++j) {
    const int slot = (t0 + j) % block_size;
    const double w = exp(s[j] - M);
    Z += w;
    for (int d = 0; d < head_dim; ++d)
      out_row[d] += w * element(v_cache, kv_elem,
                                cache_index(page_of[j], slot, h, d, block_size,
                                            num_kv_heads, head_dim)) * vs;
  }
  for (int d = 0; d < head_dim; ++d) out_row[d] /= Z;

  free(page_of);
  free(s);
  return ORACLE_OK;
}

/* The same with one storage code for q and both caches, and no scales. */
int oracle_decode_row(double* out_row, const void* q, const void* k_cache,
                      const void* v_cache, int elem,
                      const int32_t* block_tables, const int32_t* context_lens,
                      int num_seqs, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int max_blocks_per_seq,
                      int num_blocks, double scale, int window, int b, int i) {
  if (elem > ORACLE_ELEM_F64) return ORACLE_BAD_ARG;
  return oracle_decode_row_kv(out_row, q, elem, k_cache, v_cache, elem, NULL, NULL,
                              block_tables, context_lens, num_seqs, num_q_heads,
                              num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                              num_blocks, scale, window, b, i);
}

/* Every row: out is [num_seqs][num_q_heads][head_dim] doubles. */
int oracle_decode(double* out, const void* q, const void* k_cache,
                  const void* v_cache, int elem, const int32_t* block_tables,
                  const int32_t* context_lens, int num_seqs, int num_q_heads,
                  int num_kv_heads, int head_dim, int block_size,
                  int max_blocks_per_seq, int num_blocks, double scale,
                  int window) {
  if (!out || num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0)
    return ORACLE_BAD_ARG;
  for (int b = 0; b < num_seqs; ++b)
    for (int i = 0; i < num_q_heads; ++i) {
      const int rc = oracle_decode_row(
          out + ((size_t)b * num_q_heads + i) * head_dim, q, k_cache, v_cache,
          elem, block_tables, context_lens, num_seqs, num_q_heads,
          num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
          scale, window, b, i);
      if (rc != ORACLE_OK) return rc;
    }
  return ORACLE_OK;
}

/* A chosen list of rows: rows[2*r] = b, rows[2*r+1] = i; out is
 * [num_rows][head_dim].  Used to check sampled outputs of large batches. */
int oracle_decode_rows(double* out, const int32_t* rows, int num_rows,
                       const void* q, const void* k_cache, const void* v_cache,
                       int elem, const int32_t* block_tables,
                       const int32_t* context_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq, int num_blocks,
                       double scale, int window) {
  if (!out || !rows || num_rows < 0 || head_dim <= 0) return ORACLE_BAD_ARG;
  for (int r = 0; r < num_rows; ++r) {
    const int rc = oracle_decode_row(
        out + (size_t)r * head_dim, q, k_cache, v_cache, elem, block_tables,
        context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
        block_size, max_blocks_per_seq, num_blocks, scale, window, rows[2 * r],
        rows[2 * r + 1]);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* Multi-token decode (several new tokens per sequence, e.g. a chunk of a
 * prefill or draft tokens to verify) over the same paged cache.  The PR
 * "perf(rocm): head_dim=128 decode arm", section "Not claimed", lists a
 * d=128 prefill as owed; the reading taken here: every sequence b carries
 * q_len new tokens whose keys and values already sit in its pages as the last
 * q_len of its context_lens[b] tokens; new token j (0 <= j < q_len), at
 * position L - q_len + j, attends causally to the tokens before it and to
 * itself, i.e. it is the single-token decode over a context of
 * L - q_len + 1 + j tokens (the window, if any, counts back from there).
 * q and out are [num_seqs][q_len][num_q_heads][head_dim].  A context shorter
 * than q_len is rejected (ORACLE_BAD_CONTEXT). */
int oracle_decode_multi_row(double* out_row, const void* q, int elem,
                            const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int block_size, int max_blocks_per_seq,
                            int num_blocks, double scale, int window, int b, int j, int i) {
  if (!q || !context_lens || !block_tables || q_len < 1 || j < 0 || j >= q_len ||
      b < 0 || b >= num_seqs || num_q_heads <= 0 || head_dim <= 0 ||
      elem < ORACLE_ELEM_BF16 || elem > ORACLE_ELEM_F64)
    return ORACLE_BAD_ARG;
  const int L = context_lens[b];
  if (L < q_len) return ORACLE_BAD_CONTEXT;
  const int32_t Lj = L - q_len + 1 + j;
  static const size_t elem_size[3] = {2, 4, 8};
  const char* q_tok = (const char*)q +
                      ((size_t)b * q_len + j) * num_q_heads * head_dim * elem_size[elem];
  return oracle_decode_row_kv(out_row, q_tok, elem, k_cache, v_cache, elem, NULL, NULL,
                              block_tables + (size_t)b * max_blocks_per_seq, &Lj, 1,
                              num_q_heads, num_kv_heads, head_dim, block_size,
                              max_blocks_per_seq, num_blocks, scale, window, 0, i);
}

/* Chosen rows of a multi-token decode: rows[3*r .. 3*r+2] = (b, j, i); out is
 * [num_rows][head_dim]. */
int oracle_decode_multi_rows(double* out, const int32_t* rows, int num_rows,
                             const void* q, const void* k_cache, const void* v_cache,
                             int elem, const int32_t* block_tables,
                             const int32_t* context_lens, int num_seqs, int q_len,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq, int num_blocks,
                             double scale, int window) {
  if (!out || !rows || num_rows < 0 || head_dim <= 0) return ORACLE_BAD_ARG;
  for (int r = 0; r < num_rows; ++r) {
    const int rc = oracle_decode_multi_row(
        out + (size_t)r * head_dim, q, elem, k_cache, v_cache, block_tables,
        context_lens, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
        block_size, max_blocks_per_seq, num_blocks, scale, window, rows[3 * r],
        rows[3 * r + 1], rows[3 * r + 2]);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* Chosen rows of a decode whose caches are stored with their own code and
 * per-head scales (quantised KV cache); see oracle_decode_row_kv. */
int oracle_decode_rows_kv(double* out, const int32_t* rows, int num_rows,
                          const void* q, int q_elem, const void* k_cache,
                          const void* v_cache, int kv_elem, const double* k_scale,
                          const double* v_scale, const int32_t* block_tables,
                          const int32_t* context_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int max_blocks_per_seq, int num_blocks,
                          double scale, int window) {
  if (!out || !rows || num_rows < 0 || head_dim <= 0) return ORACLE_BAD_ARG;
  for (int r = 0; r < num_rows; ++r) {
    const int rc = oracle_decode_row_kv(
        out + (size_t)r * head_dim, q, q_elem, k_cache, v_cache, kv_elem, k_scale,
        v_scale, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
        head_dim, block_size, max_blocks_per_seq, num_blocks, scale, window,
        rows[2 * r], rows[2 * r + 1]);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}
