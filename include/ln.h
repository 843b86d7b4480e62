/*
 * ln.h -- C ABI of the row-normalization kernels: LayerNorm and RMSNorm over
 * the last dimension of a row-major [M, N] array, forward and backward, with
 * the per-feature weight (gamma) and bias (beta) gradients.
 *
 * The operations are those of "Optimize AMD normalization backward kernel by
 * using tiled and two pass" (ROCm/pytorch PR #3564): layer_norm and rms_norm
 * backward with their gamma/beta gradients, on the shapes of its "Layer Norm
 * Backward Benchmark" table, with output masks (dgamma only, dbeta only) and
 * the M = 1 / N = 1 and non-contiguous-input cases of its test list.  Per
 * row m, over its N features (biased variance, eps inside the square root):
 *
 *   LayerNorm:  mean = sum x / N,  rstd = 1 / sqrt(sum (x - mean)^2 / N + eps),
 *               xhat = (x - mean) * rstd,  y = xhat * gamma[n] + beta[n]
 *   RMSNorm:    rstd = 1 / sqrt(sum x^2 / N + eps),  xhat = x * rstd,
 *               y = xhat * gamma[n]
 *   backward, g = gamma[n] * dy:
 *     LayerNorm dx = rstd * (g - mean(g) - xhat * mean(g * xhat))
 *     RMSNorm   dx = rstd * (g - xhat * mean(g * xhat))
 *     dgamma[n] = sum over rows of dy * xhat,  dbeta[n] = sum over rows of dy
 *
 * Types, ownership and errors are as in gn.h: x, y, dy, dx are `dtype`
 * (GN_DTYPE_F32 / F16 / BF16); gamma, beta, mean, rstd, dgamma, dbeta are
 * fp32; every reduction is fp32; y and dx are rounded once to nearest even.
 * All pointers are device pointers owned by the caller; the library allocates
 * nothing and enqueues its kernels on `stream` (a cudaStream_t, NULL = legacy
 * default stream).  Arguments are validated on the host before anything is
 * enqueued.  Results are bit-identical from run to run on the same device
 * (every sum has a fixed order).  Rows must be 16-byte aligned for the vector
 * path (N * element size a multiple of 16 and 16-byte aligned bases); any
 * other shape or alignment takes the scalar path.
 */
#ifndef LN_H_
#define LN_H_

#include "gn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace that ln_bwd / rms_bwd need for [M, N] of `dtype` on the
 * current device: one fp32 (dgamma, dbeta) partial per feature for each CTA
 * of the backward kernel.  The workspace is scratch: no zero-fill is needed
 * and its contents are dead between calls.  0 for invalid or empty problems.
 * Host-only. */
GN_API size_t ln_workspace_size(int64_t M, int64_t N, int dtype);

/* LayerNorm forward.  Reads x [M, N], gamma [N] and beta [N] (either may be
 * NULL: weight 1 / bias 0).  Writes y [M, N] (may be x itself), mean [M] and
 * rstd [M].  M = 0: GN_OK, nothing launched.  N <= 0, M < 0, eps < 0 or a
 * NULL x / y / mean / rstd: GN_ERR_INVALID. */
GN_API int ln_fwd(const void* x, int64_t M, int64_t N, int dtype, const float* gamma,
                  const float* beta, float eps, void* y, float* mean, float* rstd, void* stream);

/* LayerNorm backward.  Reads dy, x [M, N], the forward's mean and rstd [M]
 * and gamma [N] (NULL: weight 1).  Writes dx [M, N] (may be dy itself),
 * dgamma [N] and dbeta [N]; each of dgamma and dbeta may be NULL (that
 * gradient is not written: the output masks).  With M = 0, dgamma and dbeta
 * (when given) are set to 0.  The workspace must hold ln_workspace_size()
 * bytes (GN_ERR_WORKSPACE otherwise, unless both gradients are NULL). */
GN_API int ln_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
                  const float* gamma, int64_t M, int64_t N, int dtype, void* dx, float* dgamma,
                  float* dbeta, void* workspace, size_t workspace_bytes, void* stream);

/* RMSNorm forward: y [M, N] and rstd [M] from x and gamma (NULL: weight 1). */
GN_API int rms_fwd(const void* x, int64_t M, int64_t N, int dtype, const float* gamma, float eps,
                   void* y, float* rstd, void* stream);

/* RMSNorm backward: dx [M, N] and dgamma [N] (NULL: not written) from dy, x,
 * the forward's rstd and gamma.  Workspace as for ln_bwd. */
GN_API int rms_bwd(const void* dy, const void* x, const float* rstd, const float* gamma,
                   int64_t M, int64_t N, int dtype, void* dx, float* dgamma, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Strided rows (the non-contiguous inputs of the page's test list): the same
 * operations on rows `ld*` elements apart (ld >= N) for x, dy and the output
 * y or dx; the functions above are these with every ld = N.  In place needs
 * equal strides.  The vector path needs every ld * element size to be a
 * multiple of 16 bytes as well. */
GN_API int ln_fwd_ex(const void* x, int64_t ldx, int64_t M, int64_t N, int dtype,
                     const float* gamma, const float* beta, float eps, void* y, int64_t ldy,
                     float* mean, float* rstd, void* stream);
GN_API int ln_bwd_ex(const void* dy, int64_t lddy, const void* x, int64_t ldx, const float* mean,
                     const float* rstd, const float* gamma, int64_t M, int64_t N, int dtype,
                     void* dx, int64_t lddx, float* dgamma, float* dbeta, void* workspace,
                     size_t workspace_bytes, void* stream);
GN_API int rms_fwd_ex(const void* x, int64_t ldx, int64_t M, int64_t N, int dtype,
                      const float* gamma, float eps, void* y, int64_t ldy, float* rstd,
                      void* stream);
GN_API int rms_bwd_ex(const void* dy, int64_t lddy, const void* x, int64_t ldx,
                      const float* rstd, const float* gamma, int64_t M, int64_t N, int dtype,
                      void* dx, int64_t lddx, float* dgamma, void* workspace,
                      size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LN_H_ */
