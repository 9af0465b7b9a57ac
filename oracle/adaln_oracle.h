/*
 * oracle/adaln_oracle.h -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, fp64 CPU statement of the fused AdaLN LayerNorm-Modulate
 * operator (AdaptiveLoad, "Technical summary" section 2.B "Fused
 * LayerNorm-Modulate CUDA kernels": normalisation and modulation fused into
 * one operator; backward with a sequence-dimension reduction of the
 * modulation gradients).  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load it.  It shares no code with the CUDA path.
 *
 * Definitions written out (fp64 throughout; b = seg_id[t]):
 *   mu_t    = (1/D) sum_d x[t,d]
 *   var_t   = (1/D) sum_d (x[t,d] - mu_t)^2           (biased, centred)
 *   rstd_t  = 1 / sqrt(var_t + eps)
 *   xhat    = (x - mu_t) * rstd_t
 *   y       = xhat * (1 + scale[b,d]) + shift[b,d]
 *   g       = dy * (1 + scale[b,d])
 *   dx      = rstd_t * (g - mean_d(g) - xhat * mean_d(g * xhat))
 *   dscale[b,d] = sum_{t : seg_id[t] = b} dy[t,d] * xhat[t,d]
 *   dshift[b,d] = sum_{t : seg_id[t] = b} dy[t,d]
 */
#ifndef ADALN_ORACLE_H
#define ADALN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the inputs.  bf16 is given as its 16 raw bits and widened
 * exactly; f64 exists so that finite-difference pins can perturb inputs. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* Return codes. */
enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_SEG = 2 };

int oracle_hw_threads(void);

/* Per-row statistics of x [T, D]: mean and rstd (fp64) for every row. */
int oracle_row_stats(const void* x, int64_t T, int32_t D, int dtype, double eps,
                     double* mean, double* rstd, int nthreads);

/* Forward.  rows[0..nrows) lists the rows to evaluate (NULL = all T rows, in
 * order).  y is [nrows, D], mean/rstd are [nrows] (either may be NULL). */
int oracle_adaln_fwd(const void* x, const void* shift, const void* scale,
                     const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
                     int dtype, double eps, const int64_t* rows, int64_t nrows,
                     double* y, double* mean, double* rstd, int nthreads);

/* Backward.  Statistics come from the oracle's own fp64 pass over x, unless
 * mean_in and rstd_in (fp32 [T]) are both given, in which case those saved
 * statistics are used (this isolates backward error from forward error).
 * dx is [nrows, D] for the listed rows (NULL rows = all; dx NULL = skip).
 * dshift/dscale are [nseg, D] and always reduce over ALL T rows (NULL = skip). */
int oracle_adaln_bwd(const void* dy, const void* x, const void* scale,
                     const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
                     int dtype, double eps, const float* mean_in,
                     const float* rstd_in, const int64_t* rows, int64_t nrows,
                     double* dx, double* dshift, double* dscale, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
