/*
 * Plain fp64 CPU oracle for the AttnRes depth-wise aggregation (one read).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct statement
 * of what one AttnRes read computes. Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * helper or constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes, per token row t (the definition, in the pages' order):
 *
 *   DepthBench reading notes, section 2.3 "Full AttnRes" (paper Appendix A):
 *     e_i = w^T RMSNorm_key(v_i)                  (no 1/sqrt(d), temperature 1)
 *     a_i = exp(e_i) / sum_j exp(e_j)
 *     z   = sum_i a_i v_i                         (values are the raw outputs)
 *   LLMRes blog, "Kimi AttnRes": phi(q, k) = exp(q^T RMSNorm(k)), q = w,
 *     k_i = v_i, RMSNorm applied to the key only.
 *
 *   RMSNorm is not written out on the pages. Reading taken here (the plain
 *   one): RMSNorm(x)_k = gamma_k * x_k / sqrt(mean_k(x_k^2) + eps), with eps
 *   inside the root, the mean over the d features and a learned gain gamma.
 *
 * The running max M is subtracted inside exp() only to keep exp() finite; in
 * exact arithmetic it cancels. lse = log(sum_j exp(e_j)) = M + log(sum_j
 * exp(e_j - M)) is returned as well: it is the quantity the two-stage Block
 * AttnRes computation (datacamp explainer, "two-stage computation") merges on.
 *
 * Source storage: fp32, bf16 (raw bit patterns, widened exactly by placing the
 * 16 bits in the high half of an fp32) or fp64. Every value is widened to fp64
 * before any arithmetic. Tokens are independent (the read is per token), so
 * rows are spread over OpenMP threads; nothing else is reordered or fused.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

static double widen(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F64) return ((const double*)base)[idx];
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  /* bf16: the 16 stored bits are the high half of an IEEE fp32 value. */
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* One read for one token. v[i] points at the d fp64 values of source i. */
static void read_token(int n, int d, double* const* v, const double* w,
                       const double* gamma, double eps, double* e, double* out,
                       double* lse) {
  /* Score every source: e_i = w . (gamma * v_i / sqrt(mean(v_i^2) + eps)). */
  for (int i = 0; i < n; ++i) {
    double sq = 0.0;
    for (int k = 0; k < d; ++k) sq += v[i][k] * v[i][k];
    double inv_rms = 1.0 / sqrt(sq / (double)d + eps);
    double dot = 0.0;
    for (int k = 0; k < d; ++k) dot += w[k] * (gamma[k] * v[i][k] * inv_rms);
    e[i] = dot;
  }
  /* Depth softmax. */
  double m = e[0];
  for (int i = 1; i < n; ++i)
    if (e[i] > m) m = e[i];
  double z = 0.0;
  for (int i = 0; i < n; ++i) z += exp(e[i] - m);
  /* Weighted sum of the raw values. */
  for (int k = 0; k < d; ++k) out[k] = 0.0;
  for (int i = 0; i < n; ++i) {
    double a = exp(e[i] - m) / z;
    for (int k = 0; k < d; ++k) out[k] += a * v[i][k];
  }
  if (lse) *lse = m + log(z);
}

/*
 * attnres_oracle_read: one AttnRes read over n_src sources for the token rows
 * listed in rows[0..n_rows).
 *
 *   bases[i], dtypes[i]: source i, a row-major [T, d] array (row t at
 *                        bases[i] + t*d elements) of dtype ORACLE_F32/BF16/F64.
 *   w, gamma:            fp64 [d] pseudo-query and key-RMSNorm gain.
 *   out:                 fp64 [n_rows, d]; lse: fp64 [n_rows] or NULL.
 *
 * Returns 0 on success, 1 on invalid arguments (nothing written), 2 if scratch
 * memory could not be obtained.
 */
int attnres_oracle_read(int n_src, const void* const* bases, const int* dtypes,
                        int64_t T, int d, const double* w, const double* gamma,
                        double eps, const int64_t* rows, int64_t n_rows,
                        double* out, double* lse) {
  if (n_src < 1 || d < 1 || T < 0 || n_rows < 0 || !bases || !dtypes || !w ||
      !gamma || (n_rows > 0 && (!rows || !out)))
    return 1;
  for (int i = 0; i < n_src; ++i)
    if (!bases[i] || dtypes[i] < ORACLE_F32 || dtypes[i] > ORACLE_F64) return 1;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return 1;

  int failed = 0;
#pragma omp parallel
  {
    double* buf = (double*)malloc(sizeof(double) * ((size_t)n_src * (size_t)d + (size_t)n_src));
    double** v = (double**)malloc(sizeof(double*) * (size_t)n_src);
    if (!buf || !v) {
#pragma omp atomic write
      failed = 1;
    }
    double* e = buf ? buf + (size_t)n_src * (size_t)d : NULL;
    if (buf && v)
      for (int i = 0; i < n_src; ++i) v[i] = buf + (size_t)i * (size_t)d;
    /* Every thread reaches the work-sharing loop, even one whose scratch
     * allocation failed (it then skips its rows and the call reports 2). */
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!buf || !v) continue;
      int64_t t = rows[r];
      for (int i = 0; i < n_src; ++i)
        for (int k = 0; k < d; ++k) v[i][k] = widen(bases[i], dtypes[i], t * (int64_t)d + k);
      read_token(n_src, d, v, w, gamma, eps, e, out + r * (int64_t)d, lse ? lse + r : NULL);
    }
    free(v);
    free(buf);
  }
  return failed ? 2 : 0;
}

/* Number of OpenMP threads a call uses (1 without OpenMP). */
int attnres_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads later calls use (n >= 1); scheduling only, the arithmetic per token
   does not depend on it. */
void attnres_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
