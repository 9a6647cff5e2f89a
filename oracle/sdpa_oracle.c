/*
 * sdpa_oracle.c — float64 CPU oracle for scaled-dot-product attention
 * (forward).  TEST INFRASTRUCTURE ONLY: it exists to check the CUDA path.
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load it; the library never does, and this file shares no code,
 * header, table or helper with the CUDA sources.
 *
 * Two routines:
 *
 *  oracle_sdpa         the plain definition of the operation, row by row:
 *                      materialise the score row, mask it, take a softmax
 *                      (with the optional sink logit in the denominator) and
 *                      multiply by V.  Pinned by tests/test_oracle_pins.py.
 *
 *  oracle_sdpa_online  the tiled online-softmax recurrence (running max m,
 *                      running sum l, accumulator rescaled by exp(m_old -
 *                      m_new) when the max grows; final O = acc / l and
 *                      LSE = m + log l), as in the forward kernel of the
 *                      rustytorch flash_attention.metal page.  It is only
 *                      used to check, by brute force, that the recurrence
 *                      equals the two-pass definition.  Pinned by the same
 *                      test file.
 *
 * Sources of the definition:
 *  - MLX PR #964, "Metal shaders for memory efficient self attention on large
 *    sequences": o = scaled_dot_product_attention(q, k, v, scale, mask).
 *  - MLX PR #4459, "Add D512 support to Metal vector attention": grouped
 *    query heads (32 query heads over 4 KV heads), sinks as an option of the
 *    same call, scale = d**-0.5 in its reproducer.
 *  - mlx 0.30.7 backend/cuda/scaled_dot_product_attention.cpp,
 *    build_sdpa_graph: bottom-right causal mask, additive bias, sink token
 *    of shape (1, H, 1, 1), log-sum-exp statistics output.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - causal is bottom-right aligned: key j visible to query i iff
 *    j <= i + (Lk - Lq);
 *  - query head h reads key/value head floor(h / (Hq / Hkv));
 *  - a sink is an extra logit, not scaled and not masked, with a zero value
 *    row; it takes part in the max and in the denominator;
 *  - a row with no visible key and no sink gives O = 0 and LSE = -inf;
 *  - LSE is in natural-log units.
 *
 * Everything is double precision.  Build without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element (b, h, i, j) of the additive mask through its element strides. */
static double mask_at(const double* mask, const int64_t* st, int64_t b,
                      int64_t h, int64_t i, int64_t j) {
  return mask[b * st[0] + h * st[1] + i * st[2] + j * st[3]];
}

/* Is key j visible to query i under the bottom-right causal rule? */
static int causal_visible(int64_t i, int64_t j, int64_t Lq, int64_t Lk) {
  return j <= i + (Lk - Lq);
}

/* Score s_j = scale * <q_i, k_j> (+ mask) or -inf when causally hidden. */
static void score_row(int64_t b, int64_t h, int64_t i, int64_t Hq, int64_t Hkv,
                      int64_t Lq, int64_t Lk, int64_t D, double scale,
                      int causal, const double* q, const double* k,
                      const double* mask, const int64_t* mask_stride,
                      double* s) {
  const int64_t G = Hq / Hkv;
  const int64_t g = h / G; /* key/value head of query head h */
  const double* qi = q + ((b * Hq + h) * Lq + i) * D;
  for (int64_t j = 0; j < Lk; ++j) {
    const double* kj = k + ((b * Hkv + g) * Lk + j) * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
    double sj = scale * dot;
    if (mask) sj += mask_at(mask, mask_stride, b, h, i, j);
    if (causal && !causal_visible(i, j, Lq, Lk)) sj = -INFINITY;
    s[j] = sj;
  }
}

/*
 * oracle_sdpa — the plain definition.
 *  q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D], mask (nullable) addressed through
 *  mask_stride[4] over [B,Hq,Lq,Lk], sinks (nullable) [Hq].
 *  rows (nullable): flat row ids r = (b*Hq + h)*Lq + i to evaluate; NULL
 *  means every row in order (nrows is then ignored).
 *  o [nrows, D], lse [nrows] (nullable), probs (nullable) [nrows, Lk]
 *  receives the softmax weight of every key (the sink's weight is
 *  1 - sum of the row).
 *  Returns 0, or -1 on bad sizes.
 */
int oracle_sdpa(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk,
                int64_t D, double scale, int causal, const double* q,
                const double* k, const double* v, const double* mask,
                const int64_t* mask_stride, const double* sinks,
                const int64_t* rows, int64_t nrows, double* o, double* lse,
                double* probs) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1) return -1;
  if (Hq % Hkv != 0) return -1;
  const int64_t total = B * Hq * Lq;
  if (!rows) nrows = total;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc((size_t)Lk * sizeof(double));
    double* p = (double*)malloc((size_t)Lk * sizeof(double));
    if (!s || !p) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t n = 0; n < nrows; ++n) {
      if (!s || !p) continue;
      const int64_t r = rows ? rows[n] : n;
      if (r < 0 || r >= total) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int64_t i = r % Lq;
      const int64_t h = (r / Lq) % Hq;
      const int64_t b = r / (Lq * Hq);
      const int64_t g = h / (Hq / Hkv);
      score_row(b, h, i, Hq, Hkv, Lq, Lk, D, scale, causal, q, k, mask,
                mask_stride, s);
      /* m = max over the visible scores and the sink */
      double m = -INFINITY;
      for (int64_t j = 0; j < Lk; ++j)
        if (s[j] > m) m = s[j];
      if (sinks && sinks[h] > m) m = sinks[h];
      double* oi = o + n * D;
      if (m == -INFINITY) { /* nothing visible, no sink */
        for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
        if (lse) lse[n] = -INFINITY;
        if (probs)
          for (int64_t j = 0; j < Lk; ++j) probs[n * Lk + j] = 0.0;
        continue;
      }
      double den = 0.0;
      for (int64_t j = 0; j < Lk; ++j) {
        p[j] = exp(s[j] - m); /* exp(-inf) = 0 for hidden keys */
        den += p[j];
      }
      if (sinks) den += exp(sinks[h] - m);
      for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
      for (int64_t j = 0; j < Lk; ++j) {
        const double w = p[j] / den;
        if (probs) probs[n * Lk + j] = w;
        if (w == 0.0) continue;
        const double* vj = v + ((b * Hkv + g) * Lk + j) * D;
        for (int64_t d = 0; d < D; ++d) oi[d] += w * vj[d];
      }
      if (lse) lse[n] = m + log(den);
    }
    free(s);
    free(p);
  }
  return bad ? -1 : 0;
}

/*
 * oracle_sdpa_online — the tiled recurrence with key tiles of width `tile`.
 * Same arguments as oracle_sdpa (no probs).  For every key tile:
 *   row_max = max of the tile's visible scores
 *   m_new   = max(m, row_max)
 *   l       = l * exp(m - m_new);  acc *= exp(m - m_new)
 *   for each visible key: e = exp(s - m_new); l += e; acc += e * v
 *   m = m_new
 * then, with a sink, the sink logit is folded in as one more key with a zero
 * value row; finally O = acc / l (0 when l == 0) and LSE = m + log l
 * (-inf when l == 0).
 */
int oracle_sdpa_online(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq,
                       int64_t Lk, int64_t D, double scale, int causal,
                       const double* q, const double* k, const double* v,
                       const double* mask, const int64_t* mask_stride,
                       const double* sinks, const int64_t* rows,
                       int64_t nrows, double* o, double* lse, int64_t tile) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1 || tile < 1)
    return -1;
  if (Hq % Hkv != 0) return -1;
  const int64_t total = B * Hq * Lq;
  if (!rows) nrows = total;
  double* s = (double*)malloc((size_t)Lk * sizeof(double));
  double* acc = (double*)malloc((size_t)D * sizeof(double));
  if (!s || !acc) {
    free(s);
    free(acc);
    return -1;
  }
  int bad = 0;
  for (int64_t n = 0; n < nrows; ++n) {
    const int64_t r = rows ? rows[n] : n;
    if (r < 0 || r >= total) {
      bad = 1;
      continue;
    }
    const int64_t i = r % Lq;
    const int64_t h = (r / Lq) % Hq;
    const int64_t b = r / (Lq * Hq);
    const int64_t g = h / (Hq / Hkv);
    score_row(b, h, i, Hq, Hkv, Lq, Lk, D, scale, causal, q, k, mask,
              mask_stride, s);
    double m = -INFINITY, l = 0.0;
    for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
    for (int64_t j0 = 0; j0 < Lk; j0 += tile) {
      const int64_t j1 = (j0 + tile < Lk) ? j0 + tile : Lk;
      double row_max = -INFINITY;
      for (int64_t j = j0; j < j1; ++j)
        if (s[j] > row_max) row_max = s[j];
      const double m_new = (row_max > m) ? row_max : m;
      if (m_new == -INFINITY) continue; /* nothing visible yet */
      const double corr = exp(m - m_new); /* 0 when m was -inf */
      l *= corr;
      for (int64_t d = 0; d < D; ++d) acc[d] *= corr;
      for (int64_t j = j0; j < j1; ++j) {
        if (s[j] == -INFINITY) continue; /* hidden key */
        const double e = exp(s[j] - m_new);
        l += e;
        const double* vj = v + ((b * Hkv + g) * Lk + j) * D;
        for (int64_t d = 0; d < D; ++d) acc[d] += e * vj[d];
      }
      m = m_new;
    }
    if (sinks) { /* one more key: logit sinks[h], value row 0 */
      const double m_new = (sinks[h] > m) ? sinks[h] : m;
      const double corr = exp(m - m_new);
      l = l * corr + exp(sinks[h] - m_new);
      for (int64_t d = 0; d < D; ++d) acc[d] *= corr;
      m = m_new;
    }
    double* oi = o + n * D;
    for (int64_t d = 0; d < D; ++d) oi[d] = (l > 0.0) ? acc[d] / l : 0.0;
    if (lse) lse[n] = (l > 0.0) ? m + log(l) : -INFINITY;
  }
  free(s);
  free(acc);
  return bad ? -1 : 0;
}

/* Threads the OpenMP runtime will use for oracle_sdpa (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Set the OpenMP thread count for later calls (ignored without OpenMP). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
