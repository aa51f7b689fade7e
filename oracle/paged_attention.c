/*
 * Oracle for paged decode attention: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header or constant with the CUDA library and never calls it.
 *
 * What it computes (the plain definition, no blocking or reordering):
 *   For sequence i, query head h, kv head g = h / (n_q_heads / n_kv_heads),
 *   length L = seq_lens[i]:
 *     1. gather  K_i[t] = Kpool[table[i][t / bs]][g][t % bs]   (t < L), same
 *        for V - a per-sequence table maps logical positions to physical
 *        fixed-size blocks ("Serving", section 23.4 Paged Attention);
 *     2. out[i][h] = softmax(scale * K_i q[i][h]) V_i in fp64, the max
 *        subtracted before exponentiation.
 *   The cache is exact ("The KV Cache: How Transformers Avoid Recomputing the
 *   Past", inference-serving tag page), so paged attention over the gathered
 *   rows is ordinary attention over the sequence's tokens.
 *   L == 0 gives a zero row (the pages are silent; this is the reading used).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25); /* (1.m) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double to_double(uint16_t x, int dtype) {
  return dtype == 0 ? oracle_fp16_to_double(x) : oracle_bf16_to_double(x);
}

/* One output row.  Returns 0, or -1 if the table names a block outside the
 * pool (nothing is read from it). */
static int decode_row(const uint16_t* q, const uint16_t* k_pool,
                      const uint16_t* v_pool, int dtype, long num_blocks,
                      int bs, int n_kv_heads, int d,
                      const int32_t* block_tables, int max_blocks,
                      const int32_t* seq_lens, int n_q_heads, double scale,
                      int i, int h, double* out_row) {
  int group = n_q_heads / n_kv_heads;
  int g = h / group;
  long L = seq_lens[i];
  for (int k = 0; k < d; ++k) out_row[k] = 0.0;
  if (L <= 0) return 0;

  double* K = (double*)malloc(sizeof(double) * (size_t)L * d);
  double* V = (double*)malloc(sizeof(double) * (size_t)L * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  double* qd = (double*)malloc(sizeof(double) * (size_t)d);
  if (!K || !V || !s || !qd) {
    free(K); free(V); free(s); free(qd);
    return -2;
  }

  /* step 1: gather through the block table */
  for (long t = 0; t < L; ++t) {
    long logical_block = t / bs;
    long offset = t % bs;
    long blk = logical_block < max_blocks
                   ? block_tables[(long)i * max_blocks + logical_block]
                   : -1;
    if (blk < 0 || blk >= num_blocks) {
      free(K); free(V); free(s); free(qd);
      return -1;
    }
    size_t base = (((size_t)blk * n_kv_heads + g) * bs + offset) * d;
    for (int k = 0; k < d; ++k) {
      K[t * d + k] = to_double(k_pool[base + k], dtype);
      V[t * d + k] = to_double(v_pool[base + k], dtype);
    }
  }
  for (int k = 0; k < d; ++k)
    qd[k] = to_double(q[((size_t)i * n_q_heads + h) * d + k], dtype);

  /* step 2: scores, max-subtracted softmax, weighted sum of V */
  double mx = -INFINITY;
  for (long t = 0; t < L; ++t) {
    double dot = 0.0;
    for (int k = 0; k < d; ++k) dot += qd[k] * K[t * d + k];
    s[t] = scale * dot;
    if (s[t] > mx) mx = s[t];
  }
  double z = 0.0;
  for (long t = 0; t < L; ++t) {
    s[t] = exp(s[t] - mx);
    z += s[t];
  }
  for (long t = 0; t < L; ++t) {
    double w = s[t] / z;
    for (int k = 0; k < d; ++k) out_row[k] += w * V[t * d + k];
  }
  free(K); free(V); free(s); free(qd);
  return 0;
}

/* rows == NULL: out is [num_seqs * n_q_heads][d], every row computed.
 * rows != NULL: out is [n_rows][d], row r computed for the flat index
 * rows[r] = i * n_q_heads + h.
 * Returns 0, -1 (block id outside the pool), -2 (allocation failure) or
 * -3 (bad sizes). */
int oracle_paged_decode(const uint16_t* q, const uint16_t* k_pool,
                        const uint16_t* v_pool, int dtype, long num_blocks,
                        int block_size, int n_kv_heads, int d_head,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* seq_lens, int num_seqs, int n_q_heads,
                        double scale, const int32_t* rows, int n_rows,
                        double* out, int n_threads) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0 || block_size <= 0 ||
      d_head <= 0 || num_seqs < 0)
    return -3;
  long total = rows ? n_rows : (long)num_seqs * n_q_heads;
  int status = 0;
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
  for (long r = 0; r < total; ++r) {
    long flat = rows ? rows[r] : r;
    int i = (int)(flat / n_q_heads), h = (int)(flat % n_q_heads);
    int st = decode_row(q, k_pool, v_pool, dtype, num_blocks, block_size,
                        n_kv_heads, d_head, block_tables, max_blocks_per_seq,
                        seq_lens, n_q_heads, scale, i, h,
                        out + (size_t)r * d_head);
    if (st != 0) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/* Threads an OpenMP region would use here (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
