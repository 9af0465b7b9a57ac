// Self-test of the bounded pipeline wait: one thread waits on an mbarrier
// that nothing ever arrives at, through the same bounded wait the staging
// kernels use, with a short limit.  The wait must give up, record
// ADALN_DEV_TIMEOUT in the device status word and return, leaving the
// context usable.  Nothing here traps or faults.
#include "common.cuh"
#include "internal.h"

namespace adaln {

__global__ void adaln_wait_timeout_probe_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  mbar_init_fence();
  if (!mbar_wait_bounded(b, 0, nullptr, limit_ns)) atomicOr(status, ADALN_DEV_TIMEOUT);
}

cudaError_t launch_wait_timeout_probe(unsigned* status, uint64_t limit_ns, cudaStream_t st) {
  adaln_wait_timeout_probe_kernel<<<1, 1, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace adaln
