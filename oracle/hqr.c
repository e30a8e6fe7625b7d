/*
 * Householder QR+ of a square float64 matrix, Q factor only -- the same
 * unblocked algorithm as hqr_plus() in rot_oracle.py, written in plain C so
 * that the oracle can handle 2048..12288-sized bases in seconds.
 *
 * TEST INFRASTRUCTURE ONLY (part of the CPU oracle).  Shares nothing with the
 * CUDA path.
 *
 * Definition (page "分布式训练中的流水线并行与梯度陈旧性优化", section 2.2:
 * orthonormalise the power-iteration product with a QR; the full-basis,
 * positive-diagonal and numerical-rank readings are the oracle's): tau =
 * rank_rtol * max_j ||a_j||; for k = 0, 1, ...: x = (H_{k-1}..H_0 A)[k:, k];
 * stop when ||x|| <= tau; else beta_k = -sgn(x_0) ||x|| (sgn(0) = +1),
 * w = x - beta_k e_0, H_k = I - 2 w w^T / (w^T w).  Q = H_0 .. H_{r-1} I,
 * accumulated backwards; column k < r of Q is multiplied by sgn(beta_k).
 *
 * Storage: column-major p x p (column j contiguous).  A is overwritten.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static double dot(const double* a, const double* b, long n) {
  double s = 0.0;
  for (long i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* Returns r (the number of reflectors), or -1 if memory ran out.
 * A: p x p column-major input (overwritten).  Q: p x p column-major output.
 * beta: p entries, R's diagonal before the sign fix (first r are set). */
long hqr_plus_f64(long p, double* A, double rank_rtol, double* Q, double* beta) {
  double* ww = (double*)malloc(sizeof(double) * (size_t)(p > 0 ? p : 1));
  if (!ww) return -1;
  double maxn = 0.0;
  for (long j = 0; j < p; ++j) {
    const double n = sqrt(dot(A + j * p, A + j * p, p));
    if (n > maxn) maxn = n;
  }
  const double tau = rank_rtol * maxn;

  long r = 0;
  for (long k = 0; k < p; ++k) {
    double* x = A + k * p + k; /* column k, rows k.. */
    const long len = p - k;
    const double nx = sqrt(dot(x, x, len));
    if (nx <= tau) break;
    const double b = x[0] >= 0.0 ? -nx : nx;
    x[0] -= b; /* x now holds w */
    const double wwk = dot(x, x, len);
    /* H_k applied to the trailing columns */
#pragma omp parallel for schedule(static)
    for (long j = k + 1; j < p; ++j) {
      double* c = A + j * p + k;
      const double f = 2.0 * dot(x, c, len) / wwk;
      for (long i = 0; i < len; ++i) c[i] -= f * x[i];
    }
    beta[k] = b;
    ww[k] = wwk;
    r = k + 1;
  }

  /* Q = H_0 (H_1 (... (H_{r-1} I))): when H_k is applied, columns 0..k-1 are
   * still unit vectors with zero rows k.., so only columns k.. change */
  memset(Q, 0, sizeof(double) * (size_t)p * (size_t)p);
  for (long j = 0; j < p; ++j) Q[j * p + j] = 1.0;
  for (long k = r - 1; k >= 0; --k) {
    const double* w = A + k * p + k;
    const long len = p - k;
#pragma omp parallel for schedule(static)
    for (long j = k; j < p; ++j) {
      double* c = Q + j * p + k;
      const double f = 2.0 * dot(w, c, len) / ww[k];
      for (long i = 0; i < len; ++i) c[i] -= f * w[i];
    }
  }
  for (long k = 0; k < r; ++k)
    if (beta[k] < 0.0)
      for (long i = 0; i < p; ++i) Q[k * p + i] = -Q[k * p + i];
  free(ww);
  return r;
}
