/*
 * pa_oracle.c -- plain, slow, float64 CPU oracle for single-token decode
 * attention over a paged KV cache, and for paged prefix prefill (a chunk of
 * new tokens attending to a cached context and causally to itself; its own
 * sources are listed above pa_oracle_prefill).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call this code.  It shares nothing with
 * the CUDA library (no headers, no helpers, no tables): it decodes the input
 * element types itself, resolves the block table itself and does every step
 * in double precision, in the order the pages state it.
 *
 * Sources (commit pages of the project "project_6"):
 *   [V2-PT]  commit 4eb83a7e "qwen3_6_scripts", paragraph "Implementation
 *            (paged_attention_v2_pytorch.py)": Phase 1 per-partition
 *            attention (QK^T, softmax, weighted V sum; store tmp_output,
 *            exp_sums, max_logits) and Phase 2 cross-partition log-sum-exp
 *            reduction (global_max, rescale, output).
 *   [V1-HW]  commit 4eb83a7e "qwen3_6_scripts", paragraph "V1
 *            paged_attention (decode <= 8192)": V1 must match plain
 *            ("manual") attention.
 *   [LAYOUT] commit 4eb83a7e "qwen3_6_scripts", paragraph "Hardware testing
 *            confirmed": the V2 cache layout K, V = [blocks, kv_heads,
 *            block_size, head_dim].
 *   [GQA]    same paragraph as [V1-HW]: a head_mapping sends each query
 *            head to one KV head (24 query heads over 4 KV heads).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - query head h reads KV head h / (num_heads / num_kv_heads);
 *   - token t of sequence b sits in physical block
 *     block_tables[b][t / block_size], slot t % block_size;
 *   - the per-partition output is normalised by its own exp-sum, and the
 *     reduction's total_sum is the sum of the rescaled exp-sums;
 *   - partition p of a sequence of length L covers tokens
 *     [p*P, min(L, (p+1)*P)), so there are ceil(L/P) partitions;
 *   - a sequence of length 0 gives an all-zero output row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes of q / k_cache / v_cache */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

/* return codes */
enum { ORC_OK = 0, ORC_BAD_ARG = -1, ORC_BAD_BLOCK = -2, ORC_NO_MEM = -3 };

typedef struct {
  int32_t dtype;              /* ORC_F32 / ORC_BF16 / ORC_F16                */
  int32_t num_seqs;           /* B                                           */
  int32_t num_heads;          /* Hq                                          */
  int32_t num_kv_heads;       /* Hkv, divides Hq                             */
  int32_t head_dim;           /* D                                           */
  int32_t block_size;         /* BS tokens per physical block               */
  int32_t num_blocks;         /* physical blocks in the pool                 */
  int32_t max_blocks_per_seq; /* row length of block_tables                  */
  double scale;               /* logit scale                                 */
} orc_shape;

/* ---- exact widening of the stored element types to double ------------- */

static double orc_bf16(uint16_t bits) {
  /* bfloat16 is the upper half of an IEEE binary32 */
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double orc_f16(uint16_t bits) {
  /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
  int sign = (bits >> 15) & 1;
  int ex = (bits >> 10) & 0x1f;
  int fr = bits & 0x3ff;
  double v;
  if (ex == 0)
    v = ldexp((double)fr, -24); /* zero or subnormal: fr * 2^-24 */
  else if (ex == 31)
    v = fr ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)fr / 1024.0, ex - 15);
  return sign ? -v : v;
}

static double orc_load(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[i];
    case ORC_BF16: return orc_bf16(((const uint16_t*)base)[i]);
    default: return orc_f16(((const uint16_t*)base)[i]);
  }
}

static int orc_check(const orc_shape* s) {
  if (!s) return ORC_BAD_ARG;
  if (s->dtype < ORC_F32 || s->dtype > ORC_F16) return ORC_BAD_ARG;
  if (s->num_seqs < 0 || s->num_heads <= 0 || s->num_kv_heads <= 0) return ORC_BAD_ARG;
  if (s->num_heads % s->num_kv_heads) return ORC_BAD_ARG;
  if (s->head_dim <= 0 || s->block_size <= 0 || s->num_blocks < 0) return ORC_BAD_ARG;
  if (s->max_blocks_per_seq < 0) return ORC_BAD_ARG;
  return ORC_OK;
}

/* Element offset of K/V[blk, kvh, off, 0] in the [blocks, kv_heads,
 * block_size, head_dim] layout [LAYOUT]. */
static int64_t orc_row(const orc_shape* s, int32_t blk, int kvh, int off) {
  return (((int64_t)blk * s->num_kv_heads + kvh) * s->block_size + off) * (int64_t)s->head_dim;
}

/* Physical block holding token t of sequence b, or -1 if the table entry is
 * outside the pool. */
static int32_t orc_block(const orc_shape* s, const int32_t* block_tables, int b, int64_t t) {
  int32_t blk = block_tables[(int64_t)b * s->max_blocks_per_seq + t / s->block_size];
  if (blk < 0 || blk >= s->num_blocks) return -1;
  return blk;
}

/* logit of query head h of sequence b against token t:
 *   l_t = scale * sum_d q[b,h,d] * K[blk, kvh, off, d]                     */
static double orc_logit(const orc_shape* s, const void* q, const void* k_cache,
                        int b, int h, int kvh, int32_t blk, int off) {
  const int64_t qb = ((int64_t)b * s->num_heads + h) * s->head_dim;
  const int64_t kb = orc_row(s, blk, kvh, off);
  double dot = 0.0;
  for (int d = 0; d < s->head_dim; ++d)
    dot += orc_load(q, s->dtype, qb + d) * orc_load(k_cache, s->dtype, kb + d);
  return s->scale * dot;
}

/*
 * One output row by the plain definition of softmax attention for a single
 * query [V1-HW]:
 *   M = max_t l_t,  w_t = exp(l_t - M),
 *   out[d] = sum_t w_t V_t[d] / sum_t w_t.
 * Returns ORC_OK, ORC_BAD_BLOCK or ORC_NO_MEM.
 */
static int orc_direct_row(const orc_shape* s, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_tables, int b, int h,
                          int32_t L, double* out) {
  const int G = s->num_heads / s->num_kv_heads;
  const int kvh = h / G; /* [GQA] */
  const int D = s->head_dim;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0) return ORC_OK;
  double* l = (double*)malloc(sizeof(double) * (size_t)L);
  if (!l) return ORC_NO_MEM;
  double M = -INFINITY;
  for (int64_t t = 0; t < L; ++t) {
    int32_t blk = orc_block(s, block_tables, b, t);
    if (blk < 0) { free(l); return ORC_BAD_BLOCK; }
    l[t] = orc_logit(s, q, k_cache, b, h, kvh, blk, (int)(t % s->block_size));
    if (l[t] > M) M = l[t];
  }
  double den = 0.0;
  for (int64_t t = 0; t < L; ++t) {
    const double w = exp(l[t] - M);
    const int32_t blk = orc_block(s, block_tables, b, t);
    const int64_t vb = orc_row(s, blk, kvh, (int)(t % s->block_size));
    den += w;
    for (int d = 0; d < D; ++d) out[d] += w * orc_load(v_cache, s->dtype, vb + d);
  }
  for (int d = 0; d < D; ++d) out[d] /= den;
  free(l);
  return ORC_OK;
}

/*
 * Direct oracle.  out is float64 [B, Hq, D] when rows == NULL; otherwise
 * only the nrows listed rows (row index b*Hq + h) are computed and row r of
 * the request goes to out[r*D .. r*D + D).
 */
int pa_oracle_decode(const orc_shape* s, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* seq_lens, const int64_t* rows,
                     int64_t nrows, double* out) {
  int rc = orc_check(s);
  if (rc) return rc;
  const int64_t all = (int64_t)s->num_seqs * s->num_heads;
  const int64_t n = rows ? nrows : all;
  for (int64_t r = 0; rows && r < n; ++r)
    if (rows[r] < 0 || rows[r] >= all) return ORC_BAD_ARG;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    const int64_t row = rows ? rows[r] : r;
    const int b = (int)(row / s->num_heads), h = (int)(row % s->num_heads);
    int e = orc_direct_row(s, q, k_cache, v_cache, block_tables, b, h, seq_lens[b],
                           out + r * s->head_dim);
    if (e) {
#pragma omp atomic write
      err = e;
    }
  }
  return err;
}

/*
 * Partitioned oracle: the two phases of [V2-PT], in double.
 *
 * Phase 1, for every (b, h, p < ceil(L/P)) over tokens [p*P, min(L,(p+1)P)):
 *   max_logits[b,h,p] = m_p = max_t l_t
 *   exp_sums[b,h,p]   = s_p = sum_t exp(l_t - m_p)
 *   tmp_out[b,h,p,:]  = o_p = sum_t exp(l_t - m_p) V_t / s_p
 * Phase 2, per (b, h):
 *   global_max = max_p m_p
 *   rescale_p  = exp(m_p - global_max) * s_p
 *   total_sum  = sum_p rescale_p
 *   out        = sum_p (rescale_p / total_sum) * o_p
 *
 * The workspace arrays are [B, Hq, max_partitions] and [B, Hq,
 * max_partitions, D]; entries p >= ceil(L/P) are left untouched.  Any of
 * them may be NULL when the caller only wants out.
 */
int pa_oracle_decode_partitioned(const orc_shape* s, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 const int32_t* seq_lens, int32_t partition_size,
                                 int32_t max_partitions, double* max_logits, double* exp_sums,
                                 double* tmp_out, double* out) {
  int rc = orc_check(s);
  if (rc) return rc;
  if (partition_size <= 0 || max_partitions < 0) return ORC_BAD_ARG;
  const int G = s->num_heads / s->num_kv_heads;
  const int D = s->head_dim;
  const int P = partition_size;
  for (int b = 0; b < s->num_seqs; ++b) {
    const int64_t L = seq_lens[b];
    if (L > 0 && (L + P - 1) / P > max_partitions) return ORC_BAD_ARG;
  }
  const int64_t all = (int64_t)s->num_seqs * s->num_heads;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < all; ++row) {
    const int b = (int)(row / s->num_heads), h = (int)(row % s->num_heads);
    const int kvh = h / G;
    const int64_t L = seq_lens[b];
    double* o = out + row * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (L <= 0) continue;
    const int np = (int)((L + P - 1) / P);
    double* m = (double*)malloc(sizeof(double) * (size_t)np);
    double* sp = (double*)malloc(sizeof(double) * (size_t)np);
    double* op = (double*)malloc(sizeof(double) * (size_t)np * D);
    double* l = (double*)malloc(sizeof(double) * (size_t)(L < P ? L : P));
    if (!m || !sp || !op || !l) {
      free(m); free(sp); free(op); free(l);
#pragma omp atomic write
      err = ORC_NO_MEM;
      continue;
    }
    int bad = 0;
    /* Phase 1 */
    for (int p = 0; p < np && !bad; ++p) {
      const int64_t t0 = (int64_t)p * P;
      const int64_t t1 = (t0 + P < L) ? t0 + P : L;
      double mp = -INFINITY;
      for (int64_t t = t0; t < t1; ++t) {
        int32_t blk = orc_block(s, block_tables, b, t);
        if (blk < 0) { bad = 1; break; }
        l[t - t0] = orc_logit(s, q, k_cache, b, h, kvh, blk, (int)(t % s->block_size));
        if (l[t - t0] > mp) mp = l[t - t0];
      }
      if (bad) break;
      double sum = 0.0;
      double* opp = op + (int64_t)p * D;
      for (int d = 0; d < D; ++d) opp[d] = 0.0;
      for (int64_t t = t0; t < t1; ++t) {
        const double w = exp(l[t - t0] - mp);
        const int64_t vb = orc_row(s, orc_block(s, block_tables, b, t), kvh,
                                   (int)(t % s->block_size));
        sum += w;
        for (int d = 0; d < D; ++d) opp[d] += w * orc_load(v_cache, s->dtype, vb + d);
      }
      for (int d = 0; d < D; ++d) opp[d] /= sum;
      m[p] = mp;
      sp[p] = sum;
      const int64_t ws = row * max_partitions + p;
      if (max_logits) max_logits[ws] = mp;
      if (exp_sums) exp_sums[ws] = sum;
      if (tmp_out)
        for (int d = 0; d < D; ++d) tmp_out[ws * D + d] = opp[d];
    }
    if (bad) {
#pragma omp atomic write
      err = ORC_BAD_BLOCK;
    } else {
      /* Phase 2 */
      double gmax = -INFINITY;
      for (int p = 0; p < np; ++p)
        if (m[p] > gmax) gmax = m[p];
      double total = 0.0;
      for (int p = 0; p < np; ++p) total += exp(m[p] - gmax) * sp[p];
      for (int p = 0; p < np; ++p) {
        const double wgt = exp(m[p] - gmax) * sp[p] / total;
        for (int d = 0; d < D; ++d) o[d] += wgt * op[(int64_t)p * D + d];
      }
    }
    free(m); free(sp); free(op); free(l);
  }
  return err;
}

/* ======================================================================
 * Paged prefix prefill (a chunk of new tokens after a cached context).
 *
 * Sources (same project):
 *   [PREFIX]  commit 1a4e1005 "paged_attn.py", opening paragraph: prefill
 *             is Flash-Attention-style online softmax over key tiles;
 *   [PHASES]  commit 4eb83a7e "qwen3_6_scripts", paragraph on the
 *             pre-allocated buffers of the prefix attention: a tile loop
 *             over the cached context, then one over the current chunk's
 *             tokens, each tile updating a block max (m_blk), the running
 *             max (m_new) and a correction factor (corr);
 *   [GATHER]  same page, paragraph "Complete rewrite of
 *             qwen3_6_scripts/paged_attn.py", item 1: the context keys and
 *             values come from the paged cache through the block table;
 *   [CAUSAL]  same page, paragraph "Prefill (flash_attn_func)": the chunk
 *             attends causally (causal=True).
 *
 * Layout (readings where the pages are silent, listed in the design notes):
 * sequence b owns rows query_start[b] .. query_start[b+1]-1 of q [T, Hq, D],
 * k_new and v_new [T, Hkv, D] (its n_b new tokens, in order), and its first
 * ctx_lens[b] = C_b tokens sit in the paged cache.  New token i (0-based in
 * the chunk) attends to the C_b context tokens and to new tokens 0..i.
 * ====================================================================== */

/* Sequence that owns token row t (query_start is non-decreasing). */
static int orc_seq_of_row(const int32_t* query_start, int num_seqs, int64_t t) {
  int lo = 0, hi = num_seqs; /* largest b with query_start[b] <= t */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (query_start[mid] <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

static int orc_prefill_check(const orc_shape* s, int64_t T, const int32_t* query_start,
                             const int32_t* ctx_lens) {
  int rc = orc_check(s);
  if (rc) return rc;
  if (T < 0 || query_start[0] != 0 || query_start[s->num_seqs] != T) return ORC_BAD_ARG;
  for (int b = 0; b < s->num_seqs; ++b) {
    if (query_start[b + 1] < query_start[b]) return ORC_BAD_ARG;
    if (ctx_lens[b] < 0 || ctx_lens[b] > (int64_t)s->max_blocks_per_seq * s->block_size)
      return ORC_BAD_ARG;
  }
  return ORC_OK;
}

/* Visible key j of new token i of sequence b: context token j < C from the
 * paged cache [GATHER], else new token j - C from k_new / v_new (row
 * query_start[b] + j - C).  Sets *base to the element offset of the key's
 * row in the array it returns through *which (0: cache, 1: new); returns
 * ORC_BAD_BLOCK for a table entry outside the pool. */
static int orc_prefill_key(const orc_shape* s, const int32_t* block_tables, int b, int kvh,
                           int32_t C, int32_t qs, int64_t j, int* which, int64_t* base) {
  if (j < C) {
    const int32_t blk = orc_block(s, block_tables, b, j);
    if (blk < 0) return ORC_BAD_BLOCK;
    *which = 0;
    *base = orc_row(s, blk, kvh, (int)(j % s->block_size));
  } else {
    *which = 1;
    *base = (((int64_t)qs + (j - C)) * s->num_kv_heads + kvh) * (int64_t)s->head_dim;
  }
  return ORC_OK;
}

/* logit of query row (t, h) against key row `base` of `keys`:
 *   l = scale * sum_d q[t,h,d] * K[d]                                       */
static double orc_prefill_logit(const orc_shape* s, const void* q, int64_t t, int h,
                                const void* keys, int64_t base) {
  const int64_t qb = (t * s->num_heads + h) * (int64_t)s->head_dim;
  double dot = 0.0;
  for (int d = 0; d < s->head_dim; ++d)
    dot += orc_load(q, s->dtype, qb + d) * orc_load(keys, s->dtype, base + d);
  return s->scale * dot;
}

/*
 * Direct prefill oracle: for every query row (t, h), plain softmax attention
 * over its visible keys,
 *   M = max_j l_j,  w_j = exp(l_j - M),  out[d] = sum_j w_j V_j[d] / sum_j w_j.
 * out is float64 [T, Hq, D] when rows == NULL; otherwise only the listed
 * rows (index t*Hq + h) are computed, row r of the request going to
 * out[r*D .. r*D + D).
 */
int pa_oracle_prefill(const orc_shape* s, int64_t T, const void* q, const void* k_new,
                      const void* v_new, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* query_start,
                      const int32_t* ctx_lens, const int64_t* rows, int64_t nrows, double* out) {
  int rc = orc_prefill_check(s, T, query_start, ctx_lens);
  if (rc) return rc;
  const int64_t all = T * s->num_heads;
  const int64_t n = rows ? nrows : all;
  for (int64_t r = 0; rows && r < n; ++r)
    if (rows[r] < 0 || rows[r] >= all) return ORC_BAD_ARG;
  const int G = s->num_heads / s->num_kv_heads;
  const int D = s->head_dim;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    const int64_t row = rows ? rows[r] : r;
    const int64_t t = row / s->num_heads;
    const int h = (int)(row % s->num_heads);
    const int kvh = h / G; /* [GQA] */
    const int b = orc_seq_of_row(query_start, s->num_seqs, t);
    const int32_t C = ctx_lens[b], qs = query_start[b];
    const int64_t nvis = (int64_t)C + (t - qs) + 1; /* [CAUSAL]: new tokens 0..i */
    double* o = out + r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    double* l = (double*)malloc(sizeof(double) * (size_t)nvis);
    if (!l) {
#pragma omp atomic write
      err = ORC_NO_MEM;
      continue;
    }
    int e = ORC_OK, which = 0;
    int64_t base = 0;
    double M = -INFINITY;
    for (int64_t j = 0; j < nvis && !e; ++j) {
      e = orc_prefill_key(s, block_tables, b, kvh, C, qs, j, &which, &base);
      if (e) break;
      l[j] = orc_prefill_logit(s, q, t, h, which ? k_new : k_cache, base);
      if (l[j] > M) M = l[j];
    }
    if (!e) {
      double den = 0.0;
      for (int64_t j = 0; j < nvis; ++j) {
        const double w = exp(l[j] - M);
        orc_prefill_key(s, block_tables, b, kvh, C, qs, j, &which, &base);
        const void* vals = which ? v_new : v_cache;
        den += w;
        for (int d = 0; d < D; ++d) o[d] += w * orc_load(vals, s->dtype, base + d);
      }
      for (int d = 0; d < D; ++d) o[d] /= den;
    } else {
#pragma omp atomic write
      err = e;
    }
    free(l);
  }
  return err;
}

/*
 * The pages' tiled prefill [PREFIX] [PHASES], in double: for every query
 * row, the visible keys are taken in tiles of `tile` keys -- first the
 * context [0, C) from the paged cache, then the chunk's new tokens up to
 * the row's own -- and each tile updates the running state
 *   m_blk = max over the tile's logits
 *   m_new = max(m, m_blk)
 *   corr  = exp(m - m_new)            (0 while nothing has been seen)
 *   acc   = acc * corr + sum_j exp(l_j - m_new) V_j
 *   l_sum = l_sum * corr + sum_j exp(l_j - m_new)
 *   m     = m_new
 * and out = acc / l_sum.  Reaches the direct oracle's value up to
 * rounding; out is float64 [T, Hq, D].
 */
int pa_oracle_prefill_tiled(const orc_shape* s, int64_t T, const void* q, const void* k_new,
                            const void* v_new, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* query_start,
                            const int32_t* ctx_lens, int32_t tile, double* out) {
  int rc = orc_prefill_check(s, T, query_start, ctx_lens);
  if (rc) return rc;
  if (tile <= 0) return ORC_BAD_ARG;
  const int G = s->num_heads / s->num_kv_heads;
  const int D = s->head_dim;
  const int64_t all = T * s->num_heads;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < all; ++row) {
    const int64_t t = row / s->num_heads;
    const int h = (int)(row % s->num_heads);
    const int kvh = h / G;
    const int b = orc_seq_of_row(query_start, s->num_seqs, t);
    const int32_t C = ctx_lens[b], qs = query_start[b];
    const int64_t i = t - qs; /* the row's place in its chunk */
    double* acc = out + row * D;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    double* l = (double*)malloc(sizeof(double) * (size_t)tile);
    if (!l) {
#pragma omp atomic write
      err = ORC_NO_MEM;
      continue;
    }
    double m = -INFINITY, lsum = 0.0;
    int e = ORC_OK;
    /* phase 0: context tiles [j0, j1) of [0, C); phase 1: chunk tiles of
     * new tokens [j0, j1) of [0, i + 1) */
    for (int phase = 0; phase < 2 && !e; ++phase) {
      const int64_t end = phase == 0 ? C : i + 1;
      for (int64_t j0 = 0; j0 < end && !e; j0 += tile) {
        const int64_t j1 = (j0 + tile < end) ? j0 + tile : end;
        int which = 0;
        int64_t base = 0;
        double m_blk = -INFINITY;
        for (int64_t j = j0; j < j1; ++j) {
          e = orc_prefill_key(s, block_tables, b, kvh, C, qs, phase == 0 ? j : C + j, &which,
                              &base);
          if (e) break;
          l[j - j0] = orc_prefill_logit(s, q, t, h, which ? k_new : k_cache, base);
          if (l[j - j0] > m_blk) m_blk = l[j - j0];
        }
        if (e) break;
        const double m_new = m > m_blk ? m : m_blk;
        const double corr = m == -INFINITY ? 0.0 : exp(m - m_new);
        for (int d = 0; d < D; ++d) acc[d] *= corr;
        lsum *= corr;
        for (int64_t j = j0; j < j1; ++j) {
          const double p = exp(l[j - j0] - m_new);
          orc_prefill_key(s, block_tables, b, kvh, C, qs, phase == 0 ? j : C + j, &which, &base);
          const void* vals = which ? v_new : v_cache;
          lsum += p;
          for (int d = 0; d < D; ++d) acc[d] += p * orc_load(vals, s->dtype, base + d);
        }
        m = m_new;
      }
    }
    if (e) {
#pragma omp atomic write
      err = e;
    } else {
      for (int d = 0; d < D; ++d) acc[d] /= lsum;
    }
    free(l);
  }
  return err;
}

/* Thread control for the timed CPU baseline. */
int pa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void pa_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
