/*
 * Seeded synthetic inputs for the DSA layer workloads.
 *
 * This file produces INPUT DATA only.  It holds none of the layer's arithmetic
 * (no pooling, scoring, selection or attention); both the CPU oracle tests and
 * the GPU path receive the arrays it writes.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Element n of tensor t under
 * seed s is a pure function of (s, t, n):
 *     key   = mix64(s ^ mix64(t + 1))
 *     r(n)  = mix64(key + (n + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the SplitMix64 output finaliser.  Normals use the Box-Muller
 * transform on two such words (counters 2n and 2n+1).  Every value is then
 * rounded to bfloat16 with round-to-nearest-even where the tensor is bf16.
 *
 * Built with -ffp-contract=off so the float arithmetic is the same on x86-64
 * and aarch64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(seed ^ mix64(tensor_id + 1));
}

static inline uint64_t word(uint64_t key, uint64_t n) {
  return mix64(key + (n + 1) * GAMMA);
}

/* uniform in [0,1) with 53 random bits */
static inline double u01(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* standard normal for element n (Box-Muller, cosine branch) */
static inline double normal_at(uint64_t key, uint64_t n) {
  double u1 = 1.0 - u01(word(key, 2 * n));     /* (0,1] */
  double u2 = u01(word(key, 2 * n + 1));       /* [0,1) */
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf/nan kept */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* N(0, scale^2) values rounded to bf16 */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t n, double scale, uint16_t* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = f32_to_bf16_rne((float)(scale * normal_at(key, (uint64_t)i)));
}

/* U(0,1) fp32 values (24 random bits, exact in fp32) */
void synth_uniform_f32(uint64_t seed, uint64_t tensor_id, uint64_t n, float* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = (float)(word(key, (uint64_t)i) >> 40) * (1.0f / 16777216.0f);
}

static inline int64_t int_at(uint64_t key, uint64_t n, int64_t lo, int64_t hi) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  return lo + (int64_t)(((word(key, n) >> 32) * span) >> 32);
}

/* integers uniform in [lo, hi], stored as bf16 (exact for |x| <= 256) */
void synth_int_bf16(uint64_t seed, uint64_t tensor_id, uint64_t n, int64_t lo, int64_t hi, uint16_t* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = f32_to_bf16_rne((float)int_at(key, (uint64_t)i, lo, hi));
}

/* integers uniform in [lo, hi], stored as fp32 */
void synth_int_f32(uint64_t seed, uint64_t tensor_id, uint64_t n, int64_t lo, int64_t hi, float* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = (float)int_at(key, (uint64_t)i, lo, hi);
}

/*
 * Indexer keys with planted clusters: k_idx [S, Di].
 * n_clusters centroids c_m ~ N(0, I) rescaled to norm `centroid_norm`.
 * A pool (4 consecutive tokens) is planted with probability 1/plant_every; a
 * planted pool picks one centroid and each of its tokens is
 * c_m + noise * N(0, I).  Tokens of other pools are N(0, I).
 */
void synth_cluster_keys_bf16(uint64_t seed, uint64_t tensor_id, int64_t S, int64_t Di, int64_t n_clusters,
                             int64_t plant_every, double centroid_norm, double noise, uint16_t* out) {
  const uint64_t kc = stream_key(seed, tensor_id * 16 + 1);  /* centroids  */
  const uint64_t kp = stream_key(seed, tensor_id * 16 + 2);  /* plant draw */
  const uint64_t kn = stream_key(seed, tensor_id * 16 + 3);  /* token noise */
  double cent[64 * 64];
  if (n_clusters > 64 || Di > 64) return;
  for (int64_t m = 0; m < n_clusters; ++m) {
    double nrm = 0.0;
    for (int64_t d = 0; d < Di; ++d) { cent[m * Di + d] = normal_at(kc, (uint64_t)(m * Di + d)); nrm += cent[m * Di + d] * cent[m * Di + d]; }
    nrm = sqrt(nrm);
    for (int64_t d = 0; d < Di; ++d) cent[m * Di + d] *= centroid_norm / nrm;
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < S; ++t) {
    const int64_t p = t / 4;
    const uint64_t r = word(kp, (uint64_t)p);
    const int planted = (int64_t)((r >> 32) % (uint64_t)plant_every) == 0;
    const int64_t m = (int64_t)((r & 0xFFFFFFFFu) % (uint64_t)n_clusters);
    for (int64_t d = 0; d < Di; ++d) {
      double z = normal_at(kn, (uint64_t)(t * Di + d));
      double x = planted ? cent[m * Di + d] + noise * z : z;
      out[t * Di + d] = f32_to_bf16_rne((float)x);
    }
  }
}

/*
 * Per-pool magnitudes following Zipf's law over ranks: a random permutation
 * gives each pool a rank r >= 1, and its magnitude is 1 + (amax - 1) * r^-s.
 * Writes mag[P] and rank[P] (1-based).  Fisher-Yates driven by the stream.
 */
void synth_zipf_pool_magnitudes(uint64_t seed, uint64_t tensor_id, int64_t P, double s, double amax,
                                float* mag, int64_t* rank) {
  const uint64_t key = stream_key(seed, tensor_id);
  for (int64_t p = 0; p < P; ++p) rank[p] = p + 1;
  for (int64_t p = P - 1; p > 0; --p) {
    int64_t j = (int64_t)(((word(key, (uint64_t)p) >> 32) * (uint64_t)(p + 1)) >> 32);
    int64_t t = rank[p]; rank[p] = rank[j]; rank[j] = t;
  }
  for (int64_t p = 0; p < P; ++p) mag[p] = (float)(1.0 + (amax - 1.0) * pow((double)rank[p], -s));
}

/* multiply rows of x [S, Di] (bf16) by the magnitude of their pool, re-rounding to bf16 */
void synth_scale_pools_bf16(int64_t S, int64_t Di, const float* mag, uint16_t* x) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < S; ++t) {
    for (int64_t d = 0; d < Di; ++d) {
      uint32_t u = (uint32_t)x[t * Di + d] << 16;
      float f;
      memcpy(&f, &u, 4);
      x[t * Di + d] = f32_to_bf16_rne(f * mag[t / 4]);
    }
  }
}

/*
 * A valid pool selection pool_idx [S, topk] (int32) that stands in for an
 * indexer's output when attention is tested on its own.
 * Row i may use pools p < n = floor(i/4).  If n <= topk the row is 0..n-1
 * followed by -1.  Otherwise [0, n) is cut into topk integer strata
 * [floor(j n / topk), floor((j+1) n / topk)) and one pool is drawn from each,
 * so the row is strictly ascending.  `hot` (length n_hot, may be 0) lists
 * popular pools: an eligible hot pool replaces the draw of the stratum it lies
 * in, so popular pools are chosen by nearly every query that may see them.
 */
void synth_pool_selection(uint64_t seed, uint64_t tensor_id, int64_t S, int64_t topk, const int64_t* hot,
                          int64_t n_hot, int32_t* out) {
  const uint64_t key = stream_key(seed, tensor_id);
#pragma omp parallel for schedule(dynamic, 256)
  for (int64_t i = 0; i < S; ++i) {
    const int64_t n = i / 4;
    int32_t* row = out + i * topk;
    if (n <= topk) {
      for (int64_t j = 0; j < topk; ++j) row[j] = j < n ? (int32_t)j : -1;
      continue;
    }
    for (int64_t j = 0; j < topk; ++j) {
      int64_t a = (j * n) / topk, b = ((j + 1) * n) / topk;
      uint64_t r = word(key, (uint64_t)(i * topk + j));
      row[j] = (int32_t)(a + (int64_t)(((r >> 32) * (uint64_t)(b - a)) >> 32));
    }
    for (int64_t h = 0; h < n_hot; ++h) {
      int64_t p = hot[h];
      if (p < 0 || p >= n) continue;
      /* stratum containing p: the largest j with floor(j n / topk) <= p */
      int64_t j = ((p + 1) * topk - 1) / n;
      while (j > 0 && (j * n) / topk > p) --j;
      while (j + 1 < topk && ((j + 1) * n) / topk <= p) ++j;
      row[j] = (int32_t)p;
    }
  }
}
