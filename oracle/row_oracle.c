/*
 * row_oracle.c -- plain, slow, fp64 CPU oracle for LayerNorm and RMSNorm,
 * forward and backward, over the last dimension of a row-major [M, N] array.
 * TEST INFRASTRUCTURE ONLY: it is called by the tests and the benchmark's
 * reference leg, never by the product path.  It shares no code, header or
 * constant with the CUDA library, nor with the GroupNorm oracle.
 *
 * The operations are the ones the ROCm/pytorch PR #3564 page ("Optimize AMD
 * normalization backward kernel by using tiled and two pass") benchmarks and
 * tests: layer_norm and rms_norm backward, the gradients of the per-feature
 * weight (gamma) and bias (beta) included ("Layer Norm Backward Benchmark"
 * table; test list: gamma/beta backward, output masks, M = 1 and N = 1 edge
 * cases).  The page does not print the formulas; this file uses the plain
 * definitions, per row m with mean and variance over its N features:
 *
 *   LayerNorm:  mean = sum_n x / N,  var = sum_n (x - mean)^2 / N (biased),
 *               rstd = 1 / sqrt(var + eps),  xhat = (x - mean) * rstd,
 *               y = xhat * gamma[n] + beta[n]
 *   RMSNorm:    rstd = 1 / sqrt(sum_n x^2 / N + eps),  xhat = x * rstd,
 *               y = xhat * gamma[n]
 *
 * and their exact gradients (g = gamma[n] * dy):
 *   LayerNorm:  dx = rstd * (g - mean_n(g) - xhat * mean_n(g * xhat))
 *   RMSNorm:    dx = rstd * (g - xhat * mean_n(g * xhat))
 *   dgamma[n] = sum_m dy * xhat,   dbeta[n] = sum_m dy (LayerNorm only)
 *
 * The backward recomputes mean and rstd from x in fp64.  Every sum is a plain
 * sequential fp64 sum; the variance takes a second pass over the deviations.
 *
 * RNO_MUTANT (compile-time, default 0) plants one deliberate mistake; only the
 * mutation test sets it, to check that the pins catch each one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef RNO_MUTANT
#define RNO_MUTANT 0
#endif

#define RNO_OK 0
#define RNO_EINVAL 1

int rno_mutant_id(void) { return RNO_MUTANT; }

/* Mean and rstd of one row (rms != 0: RMSNorm, mean reported as 0). */
static void row_stats(const double* x, int64_t N, double eps, int rms, double* mean,
                      double* rstd) {
  double mu = 0.0;
  if (!rms) {
    for (int64_t n = 0; n < N; ++n) mu += x[n];
    mu /= (double)N;
  }
  double v = 0.0;
  for (int64_t n = 0; n < N; ++n) {
    const double d = x[n] - mu;
    v += d * d;
  }
#if RNO_MUTANT == 1
  /* mutant: unbiased variance */
  v /= (double)(N > 1 ? N - 1 : 1);
#else
  v /= (double)N;
#endif
#if RNO_MUTANT == 2
  /* mutant: eps outside the square root */
  *rstd = 1.0 / (sqrt(v) + eps);
#else
  *rstd = 1.0 / sqrt(v + eps);
#endif
  *mean = mu;
}

/* Forward of rows [0, M).  gamma / beta may be NULL (1 / 0); mean may be NULL. */
static int fwd(const double* x, int64_t M, int64_t N, const double* gamma, const double* beta,
               double eps, int rms, double* y, double* mean, double* rstd) {
  if (M < 0 || N <= 0 || !(eps >= 0.0)) return RNO_EINVAL;
  for (int64_t m = 0; m < M; ++m) {
    const double* xr = x + m * N;
    double mu, r;
    row_stats(xr, N, eps, rms, &mu, &r);
    if (mean) mean[m] = mu;
    rstd[m] = r;
    for (int64_t n = 0; n < N; ++n) {
      const double xh = (xr[n] - mu) * r;
#if RNO_MUTANT == 3
      /* mutant: the affine weight indexed by row */
      const double gm = gamma ? gamma[m % N] : 1.0;
#else
      const double gm = gamma ? gamma[n] : 1.0;
#endif
      const double bt = (!rms && beta) ? beta[n] : 0.0;
      y[m * N + n] = xh * gm + bt;
    }
  }
  return RNO_OK;
}

/* Backward of rows [0, M); dgamma / dbeta receive the sums over these rows
 * (zeroed first).  dbeta is ignored for RMSNorm and may be NULL. */
static int bwd(const double* dy, const double* x, int64_t M, int64_t N, const double* gamma,
               double eps, int rms, double* dx, double* dgamma, double* dbeta) {
  if (M < 0 || N <= 0 || !(eps >= 0.0)) return RNO_EINVAL;
  for (int64_t n = 0; n < N; ++n) {
    dgamma[n] = 0.0;
    if (dbeta) dbeta[n] = 0.0;
  }
  for (int64_t m = 0; m < M; ++m) {
    const double* xr = x + m * N;
    const double* dr = dy + m * N;
    double mu, r;
    row_stats(xr, N, eps, rms, &mu, &r);
    double sg = 0.0, sgx = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double gm = gamma ? gamma[n] : 1.0;
      const double xh = (xr[n] - mu) * r;
      sg += gm * dr[n];
      sgx += gm * dr[n] * xh;
    }
    sg /= (double)N;
    sgx /= (double)N;
    for (int64_t n = 0; n < N; ++n) {
      const double gm = gamma ? gamma[n] : 1.0;
      const double xh = (xr[n] - mu) * r;
      const double g = gm * dr[n];
#if RNO_MUTANT == 4
      /* mutant: the mean-gradient term dropped for LayerNorm */
      (void)sg;
      dx[m * N + n] = r * (g - xh * sgx);
#elif RNO_MUTANT == 5
      /* mutant: the xhat term with the wrong sign */
      dx[m * N + n] = r * (g - (rms ? 0.0 : sg) + xh * sgx);
#elif RNO_MUTANT == 6
      /* mutant: RMSNorm keeps the mean-gradient term */
      dx[m * N + n] = r * (g - sg - xh * sgx);
#else
      dx[m * N + n] = r * (g - (rms ? 0.0 : sg) - xh * sgx);
#endif
#if RNO_MUTANT == 7
      /* mutant: dgamma of raw x */
      dgamma[n] += dr[n] * xr[n];
#else
      dgamma[n] += dr[n] * xh;
#endif
#if RNO_MUTANT == 8
      /* mutant: dbeta weighted by gamma */
      if (dbeta && !rms) dbeta[n] += g;
#else
      if (dbeta && !rms) dbeta[n] += dr[n];
#endif
    }
  }
  return RNO_OK;
}

int rno_ln_forward(const double* x, int64_t M, int64_t N, const double* gamma,
                   const double* beta, double eps, double* y, double* mean, double* rstd) {
  return fwd(x, M, N, gamma, beta, eps, 0, y, mean, rstd);
}

int rno_rms_forward(const double* x, int64_t M, int64_t N, const double* gamma, double eps,
                    double* y, double* rstd) {
  return fwd(x, M, N, gamma, NULL, eps, 1, y, NULL, rstd);
}

int rno_ln_backward(const double* dy, const double* x, int64_t M, int64_t N,
                    const double* gamma, double eps, double* dx, double* dgamma, double* dbeta) {
  return bwd(dy, x, M, N, gamma, eps, 0, dx, dgamma, dbeta);
}

int rno_rms_backward(const double* dy, const double* x, int64_t M, int64_t N,
                     const double* gamma, double eps, double* dx, double* dgamma) {
  return bwd(dy, x, M, N, gamma, eps, 1, dx, dgamma, NULL);
}
