/*
 * TEST INFRASTRUCTURE ONLY -- the fp64 CPU oracle for paged decode attention.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
 * this file's library.  It shares no code, header or table with the CUDA path.
 *
 * What it computes is the plain definition of single-token decode attention over
 * a paged KV cache, as the pages state it:
 *   - "qaqbuyan: vLLM PagedAttention", `paged_attention` pseudocode: every logical
 *     block i of a sequence is found at physical block block_table[i] of
 *     key_blocks/value_blocks laid out [num_blocks, block_size, heads, head_dim];
 *     the gathered K/V are concatenated and fed to softmax(q K^T * scale) V.
 *   - "P06 BlockManager", problem summary: token `pos` lives at
 *     slot = table[pos // bs] * bs + pos % bs, i.e. physical block table[pos // bs],
 *     row pos % bs of that block.
 * Readings taken where the pages are silent:
 *   - exactly context_lens[s] tokens are attended (the page's CUDA sketch would
 *     attend every row of the last block; its signature has no length mask);
 *   - query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups);
 *   - context_lens[s] == 0 gives an all-zero output row.
 * All arithmetic is fp64 on fp16 inputs widened exactly.  The loop order is the
 * definition's: gather, score every token, take the max, exponentiate, normalise,
 * weight V.  No blocking, no online softmax, no split.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_INDEX -5

/* IEEE 754 binary16 -> binary64, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* One (sequence, query head) row of the output. */
static int attend_one(double* out_row, const uint16_t* q, const uint16_t* k_cache,
                      const uint16_t* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, int s, int h, int Hq, int Hkv, int D,
                      int bs, int64_t num_blocks, int max_blocks, double scale) {
  const int group = Hq / Hkv;
  const int g = h / group;
  const int L = context_lens[s];
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  if (L < 0 || (int64_t)L > (int64_t)max_blocks * bs) return ORACLE_BAD_INDEX;
  if (L == 0) return ORACLE_OK;

  const int32_t* table = block_tables + (int64_t)s * max_blocks;
  const uint16_t* qrow = q + ((int64_t)s * Hq + h) * D;
  double* qd = (double*)malloc(sizeof(double) * (size_t)D);
  double* score = (double*)malloc(sizeof(double) * (size_t)L);
  if (!qd || !score) {
    free(qd);
    free(score);
    return ORACLE_BAD_ARG;
  }
  for (int d = 0; d < D; ++d) qd[d] = oracle_half_to_double(qrow[d]);

  /* scores x_t = scale * <q, K[t]>, K[t] gathered through the block table */
  for (int t = 0; t < L; ++t) {
    const int32_t b = table[t / bs];
    if (b < 0 || (int64_t)b >= num_blocks) {
      free(qd);
      free(score);
      return ORACLE_BAD_INDEX;
    }
    const uint16_t* krow = k_cache + (((int64_t)b * bs + t % bs) * Hkv + g) * D;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qd[d] * oracle_half_to_double(krow[d]);
    score[t] = scale * acc;
  }
  /* softmax over the L scores */
  double m = score[0];
  for (int t = 1; t < L; ++t)
    if (score[t] > m) m = score[t];
  double z = 0.0;
  for (int t = 0; t < L; ++t) {
    score[t] = exp(score[t] - m);
    z += score[t];
  }
  for (int t = 0; t < L; ++t) score[t] /= z;
  /* out = sum_t w_t V[t] */
  for (int t = 0; t < L; ++t) {
    const int32_t b = table[t / bs];
    const uint16_t* vrow = v_cache + (((int64_t)b * bs + t % bs) * Hkv + g) * D;
    for (int d = 0; d < D; ++d) out_row[d] += score[t] * oracle_half_to_double(vrow[d]);
  }
  free(qd);
  free(score);
  return ORACLE_OK;
}

static int check_shape(int S, int Hq, int Hkv, int D, int bs, int max_blocks) {
  if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || bs <= 0 || max_blocks < 0) return 0;
  if (Hq % Hkv != 0) return 0;
  return 1;
}

/* out: fp64 [S, Hq, D]; q: fp16 bits [S, Hq, D];
 * k_cache, v_cache: fp16 bits [num_blocks, bs, Hkv, D];
 * block_tables: [S, max_blocks]; context_lens: [S].
 * Returns 0, or the first negative status met (the row is then left zero). */
int oracle_paged_attention_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                                  const uint16_t* v_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, int S, int Hq, int Hkv, int D,
                                  int bs, int64_t num_blocks, int max_blocks, double scale) {
  if (!check_shape(S, Hq, Hkv, D, bs, max_blocks)) return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  const int64_t n = (int64_t)S * Hq;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    const int s = (int)(i / Hq), h = (int)(i % Hq);
    int rc = attend_one(out + i * D, q, k_cache, v_cache, block_tables, context_lens, s, h, Hq,
                        Hkv, D, bs, num_blocks, max_blocks, scale);
    if (rc != ORACLE_OK) {
#pragma omp critical
      if (status == ORACLE_OK) status = rc;
    }
  }
  return status;
}

/* Same definition evaluated only at the listed (seq, head) pairs:
 * out: fp64 [n, D], row i is (seq_idx[i], head_idx[i]). */
int oracle_paged_attention_decode_rows(double* out, const uint16_t* q, const uint16_t* k_cache,
                                       const uint16_t* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int S, int Hq, int Hkv,
                                       int D, int bs, int64_t num_blocks, int max_blocks,
                                       double scale, const int32_t* seq_idx,
                                       const int32_t* head_idx, int n) {
  if (!check_shape(S, Hq, Hkv, D, bs, max_blocks) || n < 0) return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n; ++i) {
    int rc;
    if (seq_idx[i] < 0 || seq_idx[i] >= S || head_idx[i] < 0 || head_idx[i] >= Hq)
      rc = ORACLE_BAD_ARG;
    else
      rc = attend_one(out + (int64_t)i * D, q, k_cache, v_cache, block_tables, context_lens,
                      seq_idx[i], head_idx[i], Hq, Hkv, D, bs, num_blocks, max_blocks, scale);
    if (rc != ORACLE_OK) {
#pragma omp critical
      if (status == ORACLE_OK) status = rc;
    }
  }
  return status;
}

/* Number of OpenMP threads a parallel region here would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads later calls use (n >= 1); for timing the oracle on one core. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
