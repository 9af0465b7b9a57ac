// Host-side interface between the C ABI (api.cu) and the kernel launchers
// (fwd.cu, bwd.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/adaln.h"

#ifdef __CUDACC__
#define ADALN_HD __host__ __device__
#else
#define ADALN_HD
#endif

namespace adaln {

// Rows handled per reduction round (compile-time in the kernels).
constexpr int kRowsPerRound = 2;
// Largest number of consumer warps in a CTA (any VPT).
constexpr int kMaxConsumerWarps = 16;

// Vectors per thread for a row of `nvec` 16-byte vectors, and the largest
// consumer-warp count used with it.  The cap keeps (warps + producer) low
// enough that each SM sub-partition can give every thread the registers the
// VPT variant needs: 17 warps -> 96 regs, 13 -> 128, 9 -> 168.
ADALN_HD constexpr int max_consumer_warps(int vpt) {
  return vpt == 1 ? 16 : (vpt == 2 ? 12 : 8);
}
ADALN_HD constexpr int max_threads(int vpt) {
  return (max_consumer_warps(vpt) + 1) * 32;
}
ADALN_HD inline int choose_vpt(int nvec) {
  return nvec <= 32 * max_consumer_warps(1) ? 1
         : (nvec <= 64 * max_consumer_warps(2) ? 2 : 4);
}

struct Shape {
  int vpt;        // 16-byte vectors per thread per row (1, 2 or 4)
  int nc;         // consumer warps
  int threads;    // (nc + 1) * 32: consumers plus one producer warp
  int stages;     // depth of the shared-memory ring
  int smem;       // dynamic shared memory bytes
  int grid;       // persistent CTAs
  int nvec;       // 16-byte vectors per row
  int row_bytes;  // bytes of one row of x
};

struct FwdArgs {
  const void* x;
  const void* shift;
  const void* scale;
  const int32_t* seg;
  void* y;
  float* mean;
  float* rstd;
  int64_t T;
  int32_t D;
  int32_t nseg;
  float eps;
  unsigned* status;
};

struct BwdArgs {
  const void* dy;
  const void* x;
  const float* mean;
  const float* rstd;
  const void* scale;
  const int32_t* seg;
  void* dx;
  float* dshift;
  float* dscale;
  float* partials;  // [G + nseg - 1][2][D] fp32: (dscale, dshift) partials
  int64_t T;
  int32_t D;
  int32_t nseg;
  unsigned* status;
};

// Launch shapes (depend on the current device).  Return cudaSuccess or the
// error of the device query.
cudaError_t fwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s);
cudaError_t bwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s);

// Number of fp32 partial slots of the backward: G + nseg - 1.
inline int64_t bwd_slots(const Shape& s, int32_t nseg) {
  return (int64_t)s.grid + nseg - 1;
}

cudaError_t launch_fwd(const FwdArgs& a, adaln_dtype_t dt, const Shape& s,
                       cudaStream_t st);
cudaError_t launch_bwd_rows(const BwdArgs& a, adaln_dtype_t dt,
                            const Shape& s, cudaStream_t st);
cudaError_t launch_bwd_finalize(const BwdArgs& a, const Shape& s,
                                cudaStream_t st);

// Shared-memory header of the staging kernels (barriers, flags, reduction
// scratch), before the 128-byte aligned ring.
ADALN_HD inline int ring_header_bytes(int stages) {
  int b = 16 * stages            // full[] and empty[] mbarriers
          + 16                   // abort flag (+ pad)
          + 2 * kMaxConsumerWarps * kRowsPerRound * 2 * 4  // reduction values
          + 2 * kMaxConsumerWarps * 4;                     // ok flags
  return (b + 127) & ~127;
}

}  // namespace adaln
