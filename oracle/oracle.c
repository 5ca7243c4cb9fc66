/*
 * CPU ORACLE for the DeepSeek-Sparse-Attention (DSA) layer -- TEST
 * INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  The product library (libdsa) never links, loads or
 * calls it, and this file shares no code, header, table or helper with it.
 *
 * Every function is the plain definition, written out in the order the
 * method states it, with double-precision accumulation and no blocking,
 * fusion or reordering.  It is deliberately slow.
 *
 * Sources (page title, section):
 *  [SkyRL-1M]  "SkyRL 将 GLM-5.3-Flash 训练上下文扩至 100 万 token"
 *              §模型与瓶颈 (each query reads ~2048 keys; the indexer scores
 *              every query against every 4-token pool) and §1 DSA 真稀疏
 *              (2051 selected keys, no positional encoding, query-chunked
 *              indexer, int32 selected-pool indices).
 *  [Anyscale]  "How Lila Sciences and Anyscale Scaled GLM-5.3-Flash
 *              Training", second lesson, on the indexer (selection scores
 *              each query against the whole sequence; scores computed a few
 *              hundred queries at a time).
 *  [CP-lesson] "128K 的序列,激活放在哪?" (context-parallel lesson),
 *              §改进二 and the evidence table, row ② (blockwise online
 *              softmax gives exactly the one-shot result).
 * The pages give no indexer formula.  The one adopted by this library:
 *   pooled key   Khat_p = fp32 mean of indexer keys 4p..4p+3,
 *   score(i,p)   = sum_h w[i,h] * ReLU(q_idx[i,h,:] . Khat_p), for 4p+3 < i.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes):
 *  - Khat summation order ((k0+k1)+(k2+k3))*0.25 in fp32.
 *  - Ties in the top-k go to the lower pool index; scores are compared after
 *    rounding to fp32; the selected set is written in ascending pool order,
 *    padded with -1.
 *  - Query i attends to the selected pools' keys plus its own partial pool
 *    {4*floor(i/4), ..., i} (1 to 4 tokens, itself included), so that with
 *    every pool selected the layer is dense causal attention.
 *  - Softmax scale is an argument (<= 0 means 1/sqrt(D)); lse is the natural
 *    log of the softmax normaliser of the scaled logits.
 *
 * Layouts (row-major, batch 1): q_idx [S,Hi,Di] bf16, k_idx [S,Di] bf16,
 * w [S,Hi] fp32, q [S,Hq,D] bf16, k,v [S,D] bf16, pool_idx [S,topk] int32,
 * dO [S,Hq,D] bf16.  bf16 arrives as raw uint16 bit patterns.
 *
 * Return codes: 0 ok, -1 bad argument, -2 malformed pool_idx row, -3 out of
 * memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bf16f(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Step 1: key pooling.  [SkyRL-1M §模型与瓶颈] pools are 4 consecutive
 * tokens; Khat_p is their fp32 mean.  Only complete pools (p < S/4) exist;
 * the partial last pool of a sequence with S % 4 != 0 is never scored. */
int oracle_pool_keys(const uint16_t* k_idx, int64_t S, int64_t Di, float* khat) {
  if (S < 0 || Di <= 0) return -1;
  const int64_t P = S / 4;
  for (int64_t p = 0; p < P; ++p) {
    for (int64_t d = 0; d < Di; ++d) {
      float k0 = bf16f(k_idx[(4 * p + 0) * Di + d]);
      float k1 = bf16f(k_idx[(4 * p + 1) * Di + d]);
      float k2 = bf16f(k_idx[(4 * p + 2) * Di + d]);
      float k3 = bf16f(k_idx[(4 * p + 3) * Di + d]);
      float a = k0 + k1;
      float b = k2 + k3;
      float s = a + b;
      khat[p * Di + d] = s * 0.25f;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: indexer scores of one query row i against every eligible pool.
 * [SkyRL-1M §模型与瓶颈] every query is scored against every earlier pool;
 * eligibility 4p+3 < i, i.e. p < floor(i/4).
 * score(i,p) = sum_h w[i,h] * max(0, sum_d q_idx[i,h,d] * Khat_p[d]).
 * Writes out[0 .. floor(i/4)-1] in double. */
static void index_scores_row(const uint16_t* q_idx, const float* khat, const float* w, int64_t Hi, int64_t Di,
                             int64_t i, double* out) {
  const int64_t n = i / 4;
  for (int64_t p = 0; p < n; ++p) {
    double score = 0.0;
    for (int64_t h = 0; h < Hi; ++h) {
      double dot = 0.0;
      for (int64_t d = 0; d < Di; ++d) dot += bf16(q_idx[(i * Hi + h) * Di + d]) * (double)khat[p * Di + d];
      double relu = dot > 0.0 ? dot : 0.0;
      score += (double)w[i * Hi + h] * relu;
    }
    out[p] = score;
  }
}

/* Scores of the listed query rows; row r is written to out + r*row_stride
 * (row_stride >= floor(max row / 4)). */
int oracle_index_scores(const uint16_t* q_idx, const uint16_t* k_idx, const float* w, int64_t S, int64_t Hi,
                        int64_t Di, const int64_t* rows, int64_t nrows, int64_t row_stride, double* out) {
  if (S < 0 || Hi <= 0 || Di <= 0 || nrows < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= S || rows[r] / 4 > row_stride) return -1;
  float* khat = (float*)malloc((size_t)((S / 4) * Di + 1) * sizeof(float));
  if (!khat) return -3;
  oracle_pool_keys(k_idx, S, Di, khat);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) index_scores_row(q_idx, khat, w, Hi, Di, rows[r], out + r * row_stride);
  free(khat);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: per-query top-k by a full sort (the library sort routine is the
 * step).  Order: score (rounded to fp32) descending, pool index ascending on
 * ties.  The first min(k, n) are kept and written in ascending pool order,
 * padded with -1.  *kth receives the fp32 score of the last kept pool (or
 * -inf when n == 0). */
typedef struct {
  float score;
  int32_t pool;
} scored_pool;

static int by_score_desc_pool_asc(const void* a, const void* b) {
  const scored_pool* x = (const scored_pool*)a;
  const scored_pool* y = (const scored_pool*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->pool > y->pool) - (x->pool < y->pool);
}

static int by_int32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

static int topk_row(const double* scores, int64_t n, int64_t k, int32_t* out, float* kth) {
  scored_pool* all = (scored_pool*)malloc((size_t)(n + 1) * sizeof(scored_pool));
  if (!all) return -3;
  for (int64_t p = 0; p < n; ++p) {
    all[p].score = (float)scores[p];
    all[p].pool = (int32_t)p;
  }
  qsort(all, (size_t)n, sizeof(scored_pool), by_score_desc_pool_asc);
  const int64_t kept = n < k ? n : k;
  for (int64_t j = 0; j < kept; ++j) out[j] = all[j].pool;
  qsort(out, (size_t)kept, sizeof(int32_t), by_int32);
  for (int64_t j = kept; j < k; ++j) out[j] = -1;
  *kth = kept > 0 ? all[kept - 1].score : -INFINITY;
  free(all);
  return 0;
}

int oracle_topk(const double* scores, int64_t n, int64_t k, int32_t* out, float* kth) {
  if (n < 0 || k <= 0) return -1;
  return topk_row(scores, n, k, out, kth);
}

/* Indexer + top-k for the listed query rows: pool_idx_out [nrows, topk],
 * kth_out [nrows] (may be NULL). */
int oracle_index_topk(const uint16_t* q_idx, const uint16_t* k_idx, const float* w, int64_t S, int64_t Hi,
                      int64_t Di, int64_t topk, const int64_t* rows, int64_t nrows, int32_t* pool_idx_out,
                      float* kth_out) {
  if (S < 0 || Hi <= 0 || Di <= 0 || topk <= 0 || nrows < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= S) return -1;
  float* khat = (float*)malloc((size_t)((S / 4) * Di + 1) * sizeof(float));
  if (!khat) return -3;
  oracle_pool_keys(k_idx, S, Di, khat);
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double* sc = (double*)malloc((size_t)(i / 4 + 1) * sizeof(double));
    float kth;
    if (!sc) {
      {
#pragma omp atomic write
        status = -3;
      }
      continue;
    }
    index_scores_row(q_idx, khat, w, Hi, Di, i, sc);
    if (topk_row(sc, i / 4, topk, pool_idx_out + r * topk, &kth) != 0) status = -3;
    if (kth_out) kth_out[r] = kth;
    free(sc);
  }
  free(khat);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Key set of query i.  [SkyRL-1M §模型与瓶颈, §1 DSA 真稀疏] each query
 * attends to the keys of its selected pools plus its own partial pool.
 * Keys: 4p..4p+3 for every selected p (ascending), then 4*floor(i/4)..i.
 * Returns the key count, or -2 if the row is malformed (an entry outside
 * [0, floor(i/4)), not strictly ascending, or a pool after a -1). */
static int64_t key_set(const int32_t* row, int64_t topk, int64_t i, int64_t* keys) {
  const int64_t n = i / 4;
  int64_t cnt = 0, prev = -1;
  int seen_pad = 0;
  for (int64_t j = 0; j < topk; ++j) {
    const int64_t p = row[j];
    if (p == -1) {
      seen_pad = 1;
      continue;
    }
    if (seen_pad || p < 0 || p >= n || p <= prev) return -2;
    prev = p;
    for (int64_t t = 0; t < 4; ++t) keys[cnt++] = 4 * p + t;
  }
  for (int64_t j = 4 * n; j <= i; ++j) keys[cnt++] = j;
  return cnt;
}

/* Softmax of one query head over its key set, two-pass (max, then sum), in
 * double.  Writes the logits s[j] (scaled) and returns lse = m + log(l). */
static double head_logits(const uint16_t* q, const uint16_t* k, int64_t Hq, int64_t D, int64_t i, int64_t h,
                          const int64_t* keys, int64_t nk, double scale, double* s) {
  double m = -INFINITY;
  for (int64_t j = 0; j < nk; ++j) {
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += bf16(q[(i * Hq + h) * D + d]) * bf16(k[keys[j] * D + d]);
    s[j] = scale * dot;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < nk; ++j) l += exp(s[j] - m);
  return m + log(l);
}

/* Step 4: sparse attention forward for the listed query rows.
 * o[r,h,:] = sum_j softmax(s)_j v_j ; lse[r,h] = log sum_j exp(s_j). */
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* pool_idx, int64_t S,
                    int64_t Hq, int64_t D, int64_t topk, double scale, const int64_t* rows, int64_t nrows, double* o,
                    double* lse) {
  if (S < 0 || Hq <= 0 || D <= 0 || topk <= 0 || nrows < 0) return -1;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= S) return -1;
  int status = 0;
#pragma omp parallel
  {
    int64_t* keys = (int64_t*)malloc((size_t)(4 * topk + 4) * sizeof(int64_t));
    double* s = (double*)malloc((size_t)(4 * topk + 4) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t i = rows[r];
      if (!keys || !s) {
        {
#pragma omp atomic write
        status = -3;
      }
        continue;
      }
      const int64_t nk = key_set(pool_idx + i * topk, topk, i, keys);
      if (nk < 0) {
        {
#pragma omp atomic write
        status = -2;
      }
        continue;
      }
      for (int64_t h = 0; h < Hq; ++h) {
        const double L = head_logits(q, k, Hq, D, i, h, keys, nk, scale, s);
        lse[r * Hq + h] = L;
        for (int64_t d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int64_t j = 0; j < nk; ++j) acc += exp(s[j] - L) * bf16(v[keys[j] * D + d]);
          o[(r * Hq + h) * D + d] = acc;
        }
      }
    }
    free(keys);
    free(s);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* Step 5/6: backward of the sparse attention for one query row i, in the
 * textbook form (P recomputed from the logits; Dh = sum_d dO*O):
 *   P_hj  = exp(s_hj - lse_h)
 *   dP_hj = dO_h . v_j
 *   dS_hj = P_hj (dP_hj - Dh)
 *   dq_h  = scale * sum_j dS_hj k_j
 *   dk_j += scale * sum_h dS_hj q_h
 *   dv_j += sum_h P_hj dO_h
 * The forward quantities are recomputed here in double from q, k, v. */
typedef struct {
  double* s;   /* [nk]   */
  double* P;   /* [Hq*nk] */
  double* dS;  /* [Hq*nk] */
  double* O;   /* [D]    */
  int64_t* keys;
} row_scratch;

static int row_scratch_init(row_scratch* w, int64_t Hq, int64_t D, int64_t topk) {
  const int64_t kmax = 4 * topk + 4;
  w->s = (double*)malloc((size_t)kmax * sizeof(double));
  w->P = (double*)malloc((size_t)(Hq * kmax) * sizeof(double));
  w->dS = (double*)malloc((size_t)(Hq * kmax) * sizeof(double));
  w->O = (double*)malloc((size_t)D * sizeof(double));
  w->keys = (int64_t*)malloc((size_t)kmax * sizeof(int64_t));
  return (w->s && w->P && w->dS && w->O && w->keys) ? 0 : -3;
}

static void row_scratch_free(row_scratch* w) {
  free(w->s);
  free(w->P);
  free(w->dS);
  free(w->O);
  free(w->keys);
}

/* Fills w->keys, w->P, w->dS for query i; returns the key count or -2. */
static int64_t backward_row(const uint16_t* dO, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const int32_t* pool_idx, int64_t Hq, int64_t D, int64_t topk, double scale, int64_t i,
                            row_scratch* w) {
  const int64_t nk = key_set(pool_idx + i * topk, topk, i, w->keys);
  if (nk < 0) return nk;
  for (int64_t h = 0; h < Hq; ++h) {
    const double L = head_logits(q, k, Hq, D, i, h, w->keys, nk, scale, w->s);
    double* P = w->P + h * nk;
    double* dS = w->dS + h * nk;
    for (int64_t j = 0; j < nk; ++j) P[j] = exp(w->s[j] - L);
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t j = 0; j < nk; ++j) acc += P[j] * bf16(v[w->keys[j] * D + d]);
      w->O[d] = acc;
    }
    double Dh = 0.0;
    for (int64_t d = 0; d < D; ++d) Dh += bf16(dO[(i * Hq + h) * D + d]) * w->O[d];
    for (int64_t j = 0; j < nk; ++j) {
      double dP = 0.0;
      for (int64_t d = 0; d < D; ++d) dP += bf16(dO[(i * Hq + h) * D + d]) * bf16(v[w->keys[j] * D + d]);
      dS[j] = P[j] * (dP - Dh);
    }
  }
  return nk;
}

/* dq [nrows, Hq, D] for the listed query rows. */
int oracle_attn_bwd_dq(const uint16_t* dO, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* pool_idx, int64_t S, int64_t Hq, int64_t D, int64_t topk, double scale,
                       const int64_t* rows, int64_t nrows, double* dq) {
  if (S < 0 || Hq <= 0 || D <= 0 || topk <= 0 || nrows < 0) return -1;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= S) return -1;
  int status = 0;
#pragma omp parallel
  {
    row_scratch w;
    const int ok = row_scratch_init(&w, Hq, D, topk);
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
      if (ok != 0) {
        {
#pragma omp atomic write
        status = -3;
      }
        continue;
      }
      const int64_t i = rows[r];
      const int64_t nk = backward_row(dO, q, k, v, pool_idx, Hq, D, topk, scale, i, &w);
      if (nk < 0) {
        {
#pragma omp atomic write
        status = -2;
      }
        continue;
      }
      for (int64_t h = 0; h < Hq; ++h)
        for (int64_t d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int64_t j = 0; j < nk; ++j) acc += w.dS[h * nk + j] * bf16(k[w.keys[j] * D + d]);
          dq[(r * Hq + h) * D + d] = scale * acc;
        }
    }
    row_scratch_free(&w);
  }
  return status;
}

/* dk, dv [nkeys, D] for the listed key rows: the sum over every query whose
 * key set contains the key.  Each thread accumulates privately; the thread
 * partials are then added in thread order. */
int oracle_attn_bwd_dkdv(const uint16_t* dO, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* pool_idx, int64_t S, int64_t Hq, int64_t D, int64_t topk, double scale,
                         const int64_t* key_rows, int64_t nkeys, double* dk, double* dv) {
  if (S < 0 || Hq <= 0 || D <= 0 || topk <= 0 || nkeys < 0) return -1;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  int64_t* slot = (int64_t*)malloc((size_t)(S + 1) * sizeof(int64_t));
  if (!slot) return -3;
  for (int64_t j = 0; j < S; ++j) slot[j] = -1;
  for (int64_t r = 0; r < nkeys; ++r) {
    if (key_rows[r] < 0 || key_rows[r] >= S || slot[key_rows[r]] >= 0) {
      free(slot);
      return -1;
    }
    slot[key_rows[r]] = r;
  }
  const int nt = oracle_num_threads();
  double* part = (double*)calloc((size_t)nt * (size_t)nkeys * (size_t)D * 2, sizeof(double));
  if (!part) {
    free(slot);
    return -3;
  }
  int status = 0;
#pragma omp parallel num_threads(nt)
  {
#ifdef _OPENMP
    const int tid = omp_get_thread_num();
#else
    const int tid = 0;
#endif
    double* pk = part + (size_t)tid * (size_t)nkeys * (size_t)D * 2;
    double* pv = pk + (size_t)nkeys * (size_t)D;
    row_scratch w;
    const int ok = row_scratch_init(&w, Hq, D, topk);
    int64_t* keys_tmp = (int64_t*)malloc((size_t)(4 * topk + 4) * sizeof(int64_t));
#pragma omp for schedule(static)
    for (int64_t i = 0; i < S; ++i) {
      if (ok != 0 || !keys_tmp) {
        {
#pragma omp atomic write
        status = -3;
      }
        continue;
      }
      /* does query i touch any requested key? */
      const int64_t nk0 = key_set(pool_idx + i * topk, topk, i, keys_tmp);
      if (nk0 < 0) {
        {
#pragma omp atomic write
        status = -2;
      }
        continue;
      }
      int touches = 0;
      for (int64_t j = 0; j < nk0 && !touches; ++j) touches = slot[keys_tmp[j]] >= 0;
      if (!touches) continue;
      const int64_t nk = backward_row(dO, q, k, v, pool_idx, Hq, D, topk, scale, i, &w);
      for (int64_t j = 0; j < nk; ++j) {
        const int64_t r = slot[w.keys[j]];
        if (r < 0) continue;
        for (int64_t d = 0; d < D; ++d) {
          double ak = 0.0, av = 0.0;
          for (int64_t h = 0; h < Hq; ++h) {
            ak += w.dS[h * nk + j] * bf16(q[(i * Hq + h) * D + d]);
            av += w.P[h * nk + j] * bf16(dO[(i * Hq + h) * D + d]);
          }
          pk[r * D + d] += scale * ak;
          pv[r * D + d] += av;
        }
      }
    }
    free(keys_tmp);
    row_scratch_free(&w);
  }
  for (int64_t x = 0; x < nkeys * D; ++x) {
    double sk = 0.0, sv = 0.0;
    for (int t = 0; t < nt; ++t) {
      sk += part[(size_t)t * (size_t)nkeys * (size_t)D * 2 + (size_t)x];
      sv += part[(size_t)t * (size_t)nkeys * (size_t)D * 2 + (size_t)nkeys * (size_t)D + (size_t)x];
    }
    dk[x] = sk;
    dv[x] = sv;
  }
  free(part);
  free(slot);
  return status;
}

/* Backward contributions of the listed query rows: dq [nrows, Hq, D] for
 * those rows, and their dk/dv contributions added into dk, dv [S, D] (which
 * the caller zeroes).  With every row listed this is the whole backward.
 * Concurrent rows add into shared keys with atomic double additions. */
int oracle_attn_bwd_rows(const uint16_t* dO, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* pool_idx, int64_t S, int64_t Hq, int64_t D, int64_t topk, double scale,
                         const int64_t* rows, int64_t nrows, double* dq, double* dk, double* dv) {
  if (S < 0 || Hq <= 0 || D <= 0 || topk <= 0 || nrows < 0) return -1;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= S) return -1;
  int status = 0;
#pragma omp parallel
  {
    row_scratch w;
    const int ok = row_scratch_init(&w, Hq, D, topk);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
      if (ok != 0) {
#pragma omp atomic write
        status = -3;
        continue;
      }
      const int64_t i = rows[r];
      const int64_t nk = backward_row(dO, q, k, v, pool_idx, Hq, D, topk, scale, i, &w);
      if (nk < 0) {
#pragma omp atomic write
        status = -2;
        continue;
      }
      for (int64_t h = 0; h < Hq; ++h)
        for (int64_t d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int64_t j = 0; j < nk; ++j) acc += w.dS[h * nk + j] * bf16(k[w.keys[j] * D + d]);
          dq[(r * Hq + h) * D + d] = scale * acc;
        }
      for (int64_t j = 0; j < nk; ++j) {
        const int64_t key = w.keys[j];
        for (int64_t d = 0; d < D; ++d) {
          double ak = 0.0, av = 0.0;
          for (int64_t h = 0; h < Hq; ++h) {
            ak += w.dS[h * nk + j] * bf16(q[(i * Hq + h) * D + d]);
            av += w.P[h * nk + j] * bf16(dO[(i * Hq + h) * D + d]);
          }
#pragma omp atomic
          dk[key * D + d] += scale * ak;
#pragma omp atomic
          dv[key * D + d] += av;
        }
      }
    }
    row_scratch_free(&w);
  }
  return status;
}
