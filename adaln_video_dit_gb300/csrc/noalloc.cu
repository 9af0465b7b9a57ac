// adaln_bwd_noalloc: the backward for callers that cannot allocate device
// memory.
//
// Some callers have no way to call cudaMalloc: code embedded in a host
// framework that owns all device memory through its own allocator and allows
// no side allocations, or code on a latency-critical path where
// cudaMalloc/cudaFree would synchronise the device.  They still own their
// inputs and outputs, but cannot provide the backward's scratch
// (per-(CTA, segment) column partials).  This entry point takes that scratch
// from a fixed file-scope device array instead, so it allocates nothing.
//
// The array takes ADALN_NOALLOC_SCRATCH_BYTES of device memory on every GPU
// where this file's module is loaded, until the process exits.  Under CUDA's
// default lazy module loading that happens at the first adaln_bwd_noalloc
// call on the device (its address lookup loads the module); with eager
// loading (CUDA_MODULE_LOADING=EAGER) it happens when the library is first
// used on the device.  All calls on a device share the array and it keeps the
// last call's contents; the backward writes every partial slot it later
// reads, so nothing needs clearing between calls.  Calls that overlap on the
// GPU (on different streams, or from different threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/adaln.h"

namespace {

constexpr size_t kScratchBytes = ADALN_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return ADALN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return ADALN_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ADALN_OK;
}

}  // namespace

extern "C" int adaln_bwd_noalloc(const void* dy, const void* x, const float* mean,
                                 const float* rstd, const void* scale,
                                 const int32_t* seg_id, int64_t T, int32_t D,
                                 int32_t nseg, adaln_dtype_t dtype, void* dx,
                                 float* dshift, float* dscale, void* stream) {
  size_t need = 0;
  int rc = adaln_bwd_workspace_size(T, D, nseg, dtype, &need);
  if (rc != ADALN_OK) return rc;
  if (need > kScratchBytes) return ADALN_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != ADALN_OK) return rc;
  return adaln_bwd(dy, x, mean, rstd, scale, seg_id, T, D, nseg, dtype, dx, dshift,
                   dscale, scratch, kScratchBytes, stream);
}
