/*
 * gn_oracle.c -- plain, slow, fp64 CPU oracle for GroupNorm forward and
 * backward.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by the
 * smoke check and by the CPU-baseline leg of the benchmark, never by the
 * product path.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (GroupNorm over an activation [N, C, *spatial] flattened to
 * [N, C, HW]; channels are split into G equal groups of Cg = C/G consecutive
 * channels):
 *
 *   Forward -- "Kimi-K2.6 l1_p35" POPCORNBENCH transcript, opening problem
 *   analysis (GroupNorm definition): for every sample n and group g the mean
 *   and the *biased* variance (divisor Cg*HW) are taken over the Cg channels of
 *   the group and all HW positions; x is normalised by sqrt(var + eps) and a
 *   per-channel affine weight/bias (shape [C]) is applied.
 *
 *   Backward -- "baracuda-kernels src/norm/group_norm_backward.rs", module
 *   comment (three-stage scheme): per (n, g) two sums are formed, then dx per
 *   element, then per-channel dgamma/dbeta.  The closed form used here is the
 *   exact gradient of the forward definition (eps inside the square root):
 *       g_i   = gamma_c * dy_i
 *       dx_i  = rstd * ( g_i - mean_S(g) - xhat_i * mean_S(g * xhat) )
 *       dbeta_c  = sum_{n,hw} dy
 *       dgamma_c = sum_{n,hw} dy * xhat
 *   where S is the (n, g) group and mean_S averages over its Cg*HW elements.
 *
 * Element addressing ("Fix GroupNorm NHWC one-pass backward execution",
 * NVIDIA/apex PR #2018, reproducer in the review thread, uses channels_last):
 *   layout 0 (NCHW):                offset = (n*C + c)*HW + hw
 *   layout 1 (NHWC, channels_last): offset = (n*HW + hw)*C + c
 *
 * Every statistic is computed in the plainest way: the mean by one pass, the
 * variance by a second pass over squared deviations, sequential fp64 sums.
 *
 * GNO_MUTANT (compile-time, default 0) plants one deliberate mistake; it is
 * only ever set by the mutation test, which checks that every planted mistake
 * is caught by at least one of the oracle's pins.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef GNO_MUTANT
#define GNO_MUTANT 0
#endif

#define GNO_OK 0
#define GNO_EINVAL 1

static int64_t off_of(int layout, int64_t n, int64_t c, int64_t hw, int64_t C,
                      int64_t HW) {
#if GNO_MUTANT == 7
  /* mutant: the channels_last index is formed like NCHW */
  (void)layout;
  return (n * C + c) * HW + hw;
#else
  if (layout == 0) return (n * C + c) * HW + hw;
  return (n * HW + hw) * C + c;
#endif
}

static int check_args(int64_t N, int64_t C, int64_t HW, int64_t G, int layout) {
  if (N < 0 || C < 0 || HW < 0 || G <= 0) return GNO_EINVAL;
  if (C % G != 0) return GNO_EINVAL;
  if (layout != 0 && layout != 1) return GNO_EINVAL;
  return GNO_OK;
}

/* Per-channel affine parameter lookup; a NULL gamma means weight 1, a NULL
 * beta means bias 0 (GroupNorm without affine). */
static double gamma_of(const double* gamma, int64_t c, int64_t Cg) {
  (void)Cg;
  if (!gamma) return 1.0;
#if GNO_MUTANT == 8
  /* mutant: weight indexed by group instead of channel */
  return gamma[c / Cg];
#else
  return gamma[c];
#endif
}

static double beta_of(const double* beta, int64_t c) {
  return beta ? beta[c] : 0.0;
}

/* Mean, biased variance and 1/sqrt(var + eps) of one (n, g) group. */
static void group_moments(const double* x, int64_t n, int64_t g, int64_t C,
                          int64_t HW, int64_t G, int layout, double eps,
                          double* mu_out, double* var_out, double* rstd_out) {
  const int64_t Cg = C / G;
  const int64_t M = Cg * HW;
  double s = 0.0;
#if GNO_MUTANT == 9
  /* mutant: statistics taken over the group's first channel only */
  const int64_t c_end = g * Cg + 1;
  const int64_t Mx = HW;
  (void)M;
#else
  const int64_t c_end = (g + 1) * Cg;
  const int64_t Mx = M;
#endif
  for (int64_t c = g * Cg; c < c_end; ++c)
    for (int64_t hw = 0; hw < HW; ++hw) s += x[off_of(layout, n, c, hw, C, HW)];
  const double mu = s / (double)Mx;
  double ss = 0.0;
  for (int64_t c = g * Cg; c < c_end; ++c)
    for (int64_t hw = 0; hw < HW; ++hw) {
      const double d = x[off_of(layout, n, c, hw, C, HW)] - mu;
      ss += d * d;
    }
#if GNO_MUTANT == 1
  /* mutant: unbiased variance */
  const double var = ss / (double)(Mx > 1 ? Mx - 1 : 1);
#else
  const double var = ss / (double)Mx;
#endif
#if GNO_MUTANT == 2
  /* mutant: eps added outside the square root */
  const double rstd = 1.0 / (sqrt(var) + eps);
#else
  const double rstd = 1.0 / sqrt(var + eps);
#endif
  *mu_out = mu;
  *var_out = var;
  *rstd_out = rstd;
}

/* Group statistics for every (n, g): mean[n*G+g], var[n*G+g] (biased) and
 * rstd[n*G+g] = 1/sqrt(var + eps).  Any output pointer may be NULL.  Groups
 * with no elements (HW == 0) are left untouched. */
int gno_stats(const double* x, int64_t N, int64_t C, int64_t HW, int64_t G,
              int layout, double eps, double* mean, double* var, double* rstd) {
  int rc = check_args(N, C, HW, G, layout);
  if (rc) return rc;
  if (N == 0 || C == 0 || HW == 0) return GNO_OK;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      double mu, v, r;
      group_moments(x, n, g, C, HW, G, layout, eps, &mu, &v, &r);
      if (mean) mean[n * G + g] = mu;
      if (var) var[n * G + g] = v;
      if (rstd) rstd[n * G + g] = r;
    }
  return GNO_OK;
}

/* Forward: y = (x - mean) * rstd * gamma[c] + beta[c] for every element, plus
 * the per-group mean and rstd (either may be NULL). */
int gno_forward(const double* x, int64_t N, int64_t C, int64_t HW, int64_t G,
                int layout, const double* gamma, const double* beta, double eps,
                double* y, double* mean, double* rstd) {
  int rc = check_args(N, C, HW, G, layout);
  if (rc) return rc;
  if (N == 0 || C == 0 || HW == 0) return GNO_OK;
  const int64_t Cg = C / G;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      double mu, v, r;
      group_moments(x, n, g, C, HW, G, layout, eps, &mu, &v, &r);
      if (mean) mean[n * G + g] = mu;
      if (rstd) rstd[n * G + g] = r;
      for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c)
        for (int64_t hw = 0; hw < HW; ++hw) {
          const int64_t o = off_of(layout, n, c, hw, C, HW);
          const double xhat = (x[o] - mu) * r;
          y[o] = xhat * gamma_of(gamma, c, Cg) + beta_of(beta, c);
        }
    }
  return GNO_OK;
}

/* The two per-group means of the backward pass, mean_S(g) and
 * mean_S(g*xhat), for one group whose moments are (mu, rstd). */
static void group_grad_means(const double* dy, const double* x, int64_t n,
                             int64_t g, int64_t C, int64_t HW, int64_t G,
                             int layout, const double* gamma, double mu,
                             double rstd, double* mg_out, double* mgx_out) {
  const int64_t Cg = C / G;
  const int64_t M = Cg * HW;
  double sg = 0.0, sgx = 0.0;
  for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c)
    for (int64_t hw = 0; hw < HW; ++hw) {
      const int64_t o = off_of(layout, n, c, hw, C, HW);
      const double gi = gamma_of(gamma, c, Cg) * dy[o];
      const double xhat = (x[o] - mu) * rstd;
      sg += gi;
      sgx += gi * xhat;
    }
  *mg_out = sg / (double)M;
  *mgx_out = sgx / (double)M;
}

static double dx_of(double gi, double xhat, double rstd, double mg, double mgx) {
#if GNO_MUTANT == 3
  /* mutant: the mean(g) term is dropped */
  (void)mg;
  return rstd * (gi - xhat * mgx);
#elif GNO_MUTANT == 4
  /* mutant: the xhat * mean(g*xhat) term is dropped */
  (void)mgx;
  (void)xhat;
  return rstd * (gi - mg);
#elif GNO_MUTANT == 5
  /* mutant: wrong sign on the xhat term */
  return rstd * (gi - mg + xhat * mgx);
#else
  return rstd * (gi - mg - xhat * mgx);
#endif
}

/* dgamma/dbeta accumulation for one element. */
static void accum_param_grads(double dyi, double xi, double mu, double rstd,
                              double* dgamma_c, double* dbeta_c) {
#if GNO_MUTANT == 6
  /* mutant: dgamma uses the raw input instead of the normalised one */
  (void)mu;
  (void)rstd;
  *dgamma_c += dyi * xi;
#else
  *dgamma_c += dyi * ((xi - mu) * rstd);
#endif
  *dbeta_c += dyi;
}

/* Backward.  Recomputes its own fp64 moments from x (it never reads the
 * forward's saved statistics), then writes dx for every element (dx may be
 * NULL) and the per-channel dgamma/dbeta (either may be NULL). */
int gno_backward(const double* dy, const double* x, int64_t N, int64_t C,
                 int64_t HW, int64_t G, int layout, const double* gamma,
                 double eps, double* dx, double* dgamma, double* dbeta) {
  int rc = check_args(N, C, HW, G, layout);
  if (rc) return rc;
  if (dgamma)
    for (int64_t c = 0; c < C; ++c) dgamma[c] = 0.0;
  if (dbeta)
    for (int64_t c = 0; c < C; ++c) dbeta[c] = 0.0;
  if (N == 0 || C == 0 || HW == 0) return GNO_OK;
  const int64_t Cg = C / G;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      double mu, v, r, mg, mgx;
      group_moments(x, n, g, C, HW, G, layout, eps, &mu, &v, &r);
      group_grad_means(dy, x, n, g, C, HW, G, layout, gamma, mu, r, &mg, &mgx);
      for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c) {
        double dgc = 0.0, dbc = 0.0;
        for (int64_t hw = 0; hw < HW; ++hw) {
          const int64_t o = off_of(layout, n, c, hw, C, HW);
          const double xhat = (x[o] - mu) * r;
          if (dx) dx[o] = dx_of(gamma_of(gamma, c, Cg) * dy[o], xhat, r, mg, mgx);
          accum_param_grads(dy[o], x[o], mu, r, &dgc, &dbc);
        }
#if GNO_MUTANT == 10
        /* mutant: parameter gradients keep only the first sample */
        if (n > 0) dgc = dbc = 0.0;
#endif
        if (dgamma) dgamma[c] += dgc;
        if (dbeta) dbeta[c] += dbc;
      }
    }
  return GNO_OK;
}

static void n_c_of(int64_t o, int64_t C, int64_t HW, int layout, int64_t* n,
                   int64_t* c) {
  *n = o / (C * HW);
  *c = (layout == 0) ? (o / HW) % C : o % C;
}

/* Sampled forward: the exact y at nidx flat offsets idx[k] (offsets in the
 * given layout).  Group moments are computed over the whole input first. */
int gno_forward_at(const double* x, int64_t N, int64_t C, int64_t HW, int64_t G,
                   int layout, const double* gamma, const double* beta,
                   double eps, const int64_t* idx, int64_t nidx, double* y_at,
                   double* mean, double* rstd) {
  int rc = check_args(N, C, HW, G, layout);
  if (rc) return rc;
  if (N == 0 || C == 0 || HW == 0) return nidx == 0 ? GNO_OK : GNO_EINVAL;
  const int64_t Cg = C / G;
  double* mu = (double*)malloc(sizeof(double) * (size_t)(N * G));
  double* rs = (double*)malloc(sizeof(double) * (size_t)(N * G));
  if (!mu || !rs) {
    free(mu);
    free(rs);
    return GNO_EINVAL;
  }
  gno_stats(x, N, C, HW, G, layout, eps, mu, NULL, rs);
  rc = GNO_OK;
  for (int64_t k = 0; k < nidx; ++k) {
    const int64_t o = idx[k];
    if (o < 0 || o >= N * C * HW) {
      rc = GNO_EINVAL;
      break;
    }
    int64_t n, c;
    n_c_of(o, C, HW, layout, &n, &c);
    const int64_t ng = n * G + c / Cg;
    y_at[k] = (x[o] - mu[ng]) * rs[ng] * gamma_of(gamma, c, Cg) + beta_of(beta, c);
  }
  if (mean)
    for (int64_t i = 0; i < N * G; ++i) mean[i] = mu[i];
  if (rstd)
    for (int64_t i = 0; i < N * G; ++i) rstd[i] = rs[i];
  free(mu);
  free(rs);
  return rc;
}

/* Sampled backward: exact dx at nidx flat offsets, plus the full dgamma and
 * dbeta (either may be NULL). */
int gno_backward_at(const double* dy, const double* x, int64_t N, int64_t C,
                    int64_t HW, int64_t G, int layout, const double* gamma,
                    double eps, const int64_t* idx, int64_t nidx, double* dx_at,
                    double* dgamma, double* dbeta) {
  int rc = check_args(N, C, HW, G, layout);
  if (rc) return rc;
  if (dgamma)
    for (int64_t c = 0; c < C; ++c) dgamma[c] = 0.0;
  if (dbeta)
    for (int64_t c = 0; c < C; ++c) dbeta[c] = 0.0;
  if (N == 0 || C == 0 || HW == 0) return nidx == 0 ? GNO_OK : GNO_EINVAL;
  const int64_t Cg = C / G;
  const int64_t NG = N * G;
  double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * NG));
  if (!buf) return GNO_EINVAL;
  double *mu = buf, *rs = buf + NG, *mg = buf + 2 * NG, *mgx = buf + 3 * NG;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      double v;
      const int64_t ng = n * G + g;
      group_moments(x, n, g, C, HW, G, layout, eps, &mu[ng], &v, &rs[ng]);
      group_grad_means(dy, x, n, g, C, HW, G, layout, gamma, mu[ng], rs[ng],
                       &mg[ng], &mgx[ng]);
      for (int64_t c = g * Cg; c < (g + 1) * Cg; ++c) {
        double dgc = 0.0, dbc = 0.0;
        for (int64_t hw = 0; hw < HW; ++hw) {
          const int64_t o = off_of(layout, n, c, hw, C, HW);
          accum_param_grads(dy[o], x[o], mu[ng], rs[ng], &dgc, &dbc);
        }
#if GNO_MUTANT == 10
        if (n > 0) dgc = dbc = 0.0;
#endif
        if (dgamma) dgamma[c] += dgc;
        if (dbeta) dbeta[c] += dbc;
      }
    }
  rc = GNO_OK;
  for (int64_t k = 0; k < nidx; ++k) {
    const int64_t o = idx[k];
    if (o < 0 || o >= N * C * HW) {
      rc = GNO_EINVAL;
      break;
    }
    int64_t n, c;
    n_c_of(o, C, HW, layout, &n, &c);
    const int64_t ng = n * G + c / Cg;
    const double xhat = (x[o] - mu[ng]) * rs[ng];
    dx_at[k] = dx_of(gamma_of(gamma, c, Cg) * dy[o], xhat, rs[ng], mg[ng], mgx[ng]);
  }
  free(buf);
  return rc;
}

/* Which mistake (if any) this compiled copy plants; 0 for the real oracle. */
int gno_mutant_id(void) { return GNO_MUTANT; }
