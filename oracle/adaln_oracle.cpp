// oracle/adaln_oracle.cpp -- TEST INFRASTRUCTURE, not part of the product.
//
// Plain fp64 CPU statement of the fused AdaLN LayerNorm-Modulate operator
// (AdaptiveLoad, "Technical summary" section 2.B).  Each quantity is computed
// by its own loop, in the order the definition states it, with no fusion.
// Multithreading only splits independent work: rows for the row-wise
// quantities, columns for the sequence reductions (each column is still summed
// over rows in increasing row order, so results do not depend on nthreads).
//
// Parity pins (tests/test_oracle_pins.py): closed forms (D = 2, constant
// rows), per-row invariants, fp64 central finite differences, torch's CPU
// fp64 layer_norm + autograd per segment, and exact integer column sums.

#include "adaln_oracle.h"

#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Widen one input element to fp64.  bf16 is the top half of an IEEE float,
// so widening is exact.
double elem(const void* p, int dtype, int64_t i) {
  if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
  if (dtype == ORACLE_F64) return ((const double*)p)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return (double)f;
}

bool dtype_ok(int dtype) {
  return dtype == ORACLE_F32 || dtype == ORACLE_BF16 || dtype == ORACLE_F64;
}

int clamp_threads(int nthreads, int64_t work) {
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > work) nthreads = (int)(work > 0 ? work : 1);
  return nthreads;
}

// Run body(lo, hi) over [0, n) split into nthreads contiguous ranges.
template <class F>
void parallel_ranges(int64_t n, int nthreads, F body) {
  nthreads = clamp_threads(nthreads, n);
  if (nthreads == 1) { body((int64_t)0, n); return; }
  std::vector<std::thread> pool;
  for (int k = 0; k < nthreads; ++k) {
    int64_t lo = n * k / nthreads, hi = n * (k + 1) / nthreads;
    pool.emplace_back([=] { body(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

// mu_t = (1/D) sum_d x[t,d]
double row_mean(const void* x, int dtype, int64_t t, int32_t D) {
  double s = 0.0;
  for (int32_t d = 0; d < D; ++d) s += elem(x, dtype, t * D + d);
  return s / D;
}

// var_t = (1/D) sum_d (x[t,d] - mu_t)^2   (biased, centred second pass)
double row_var(const void* x, int dtype, int64_t t, int32_t D, double mu) {
  double s = 0.0;
  for (int32_t d = 0; d < D; ++d) {
    double c = elem(x, dtype, t * D + d) - mu;
    s += c * c;
  }
  return s / D;
}

// rstd_t = 1 / sqrt(var_t + eps)
double rstd_of(double var, double eps) { return 1.0 / std::sqrt(var + eps); }

bool segs_ok(const int32_t* seg_id, int64_t T, int32_t nseg) {
  for (int64_t t = 0; t < T; ++t)
    if (seg_id[t] < 0 || seg_id[t] >= nseg) return false;
  return true;
}

}  // namespace

extern "C" int oracle_hw_threads(void) {
  unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

extern "C" int oracle_row_stats(const void* x, int64_t T, int32_t D, int dtype,
                                double eps, double* mean, double* rstd,
                                int nthreads) {
  if (T < 0 || D <= 0 || !dtype_ok(dtype) || (T > 0 && !x)) return ORACLE_ERR_ARG;
  parallel_ranges(T, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t t = lo; t < hi; ++t) {
      double mu = row_mean(x, dtype, t, D);
      double var = row_var(x, dtype, t, D, mu);
      if (mean) mean[t] = mu;
      if (rstd) rstd[t] = rstd_of(var, eps);
    }
  });
  return ORACLE_OK;
}

// Forward: y = xhat * (1 + scale[b]) + shift[b], row by row.
extern "C" int oracle_adaln_fwd(const void* x, const void* shift,
                                const void* scale, const int32_t* seg_id,
                                int64_t T, int32_t D, int32_t nseg, int dtype,
                                double eps, const int64_t* rows, int64_t nrows,
                                double* y, double* mean, double* rstd,
                                int nthreads) {
  if (T < 0 || D <= 0 || nseg <= 0 || !dtype_ok(dtype)) return ORACLE_ERR_ARG;
  if (T > 0 && (!x || !shift || !scale || !seg_id)) return ORACLE_ERR_ARG;
  if (!segs_ok(seg_id, T, nseg)) return ORACLE_ERR_SEG;
  if (!rows) nrows = T;
  for (int64_t i = 0; i < (rows ? nrows : 0); ++i)
    if (rows[i] < 0 || rows[i] >= T) return ORACLE_ERR_ARG;

  parallel_ranges(nrows, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) {
      const int64_t t = rows ? rows[i] : i;
      const int64_t b = seg_id[t];
      const double mu = row_mean(x, dtype, t, D);
      const double var = row_var(x, dtype, t, D, mu);
      const double rs = rstd_of(var, eps);
      if (mean) mean[i] = mu;
      if (rstd) rstd[i] = rs;
      if (!y) continue;
      for (int32_t d = 0; d < D; ++d) {
        const double xhat = (elem(x, dtype, t * D + d) - mu) * rs;
        const double sc = elem(scale, dtype, b * D + d);
        const double sh = elem(shift, dtype, b * D + d);
        y[i * D + d] = xhat * (1.0 + sc) + sh;
      }
    }
  });
  return ORACLE_OK;
}

// Backward of L = sum y * dy through the forward above.
extern "C" int oracle_adaln_bwd(const void* dy, const void* x, const void* scale,
                                const int32_t* seg_id, int64_t T, int32_t D,
                                int32_t nseg, int dtype, double eps,
                                const float* mean_in, const float* rstd_in,
                                const int64_t* rows, int64_t nrows, double* dx,
                                double* dshift, double* dscale, int nthreads) {
  if (T < 0 || D <= 0 || nseg <= 0 || !dtype_ok(dtype)) return ORACLE_ERR_ARG;
  if (T > 0 && (!x || !dy || !scale || !seg_id)) return ORACLE_ERR_ARG;
  if (!segs_ok(seg_id, T, nseg)) return ORACLE_ERR_SEG;
  if (!rows) nrows = T;
  for (int64_t i = 0; i < (rows ? nrows : 0); ++i)
    if (rows[i] < 0 || rows[i] >= T) return ORACLE_ERR_ARG;

  // Row statistics: the saved fp32 ones when given, else the oracle's own.
  std::vector<double> mu(T), rs(T);
  if (mean_in && rstd_in) {
    for (int64_t t = 0; t < T; ++t) {
      mu[t] = (double)mean_in[t];
      rs[t] = (double)rstd_in[t];
    }
  } else {
    oracle_row_stats(x, T, D, dtype, eps, mu.data(), rs.data(), nthreads);
  }

  // dx for the listed rows.
  if (dx) {
    parallel_ranges(nrows, nthreads, [&](int64_t lo, int64_t hi) {
      std::vector<double> g(D), xhat(D);
      for (int64_t i = lo; i < hi; ++i) {
        const int64_t t = rows ? rows[i] : i;
        const int64_t b = seg_id[t];
        for (int32_t d = 0; d < D; ++d) {
          xhat[d] = (elem(x, dtype, t * D + d) - mu[t]) * rs[t];
          g[d] = elem(dy, dtype, t * D + d) * (1.0 + elem(scale, dtype, b * D + d));
        }
        double mean_g = 0.0;
        for (int32_t d = 0; d < D; ++d) mean_g += g[d];
        mean_g /= D;
        double mean_gx = 0.0;
        for (int32_t d = 0; d < D; ++d) mean_gx += g[d] * xhat[d];
        mean_gx /= D;
        for (int32_t d = 0; d < D; ++d)
          dx[i * D + d] = rs[t] * (g[d] - mean_g - xhat[d] * mean_gx);
      }
    });
  }

  // Sequence reductions: every column is summed over rows in row order.
  if (dshift || dscale) {
    if (dshift) std::memset(dshift, 0, sizeof(double) * (size_t)nseg * D);
    if (dscale) std::memset(dscale, 0, sizeof(double) * (size_t)nseg * D);
    parallel_ranges(D, nthreads, [&](int64_t d0, int64_t d1) {
      for (int64_t t = 0; t < T; ++t) {
        const int64_t b = seg_id[t];
        for (int64_t d = d0; d < d1; ++d) {
          const double dyv = elem(dy, dtype, t * D + d);
          if (dshift) dshift[b * D + d] += dyv;
          if (dscale) {
            const double xhat = (elem(x, dtype, t * D + d) - mu[t]) * rs[t];
            dscale[b * D + d] += dyv * xhat;
          }
        }
      }
    });
  }
  return ORACLE_OK;
}
