// C ABI of libadaln: argument checks (all before any CUDA call), launch-shape
// cache, the per-device status word, and the kernel timing trace.
#include <cmath>
#include <mutex>
#include <vector>

#include "internal.h"

namespace adaln {
// Device status word: kernels OR ADALN_DEV_* bits into it.
__device__ unsigned int g_status_word;
}  // namespace adaln

using namespace adaln;

namespace {

constexpr int kMaxDevices = 64;

int esize_of(adaln_dtype_t dt) { return dt == ADALN_BF16 ? 2 : 4; }

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int check_dims(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dt) {
  if (dt != ADALN_F32 && dt != ADALN_BF16) return ADALN_ERR_DTYPE;
  const int32_t dmax = dt == ADALN_BF16 ? ADALN_MAX_D_BF16 : ADALN_MAX_D_F32;
  if (T < 0 || T > (int64_t)INT32_MAX) return ADALN_ERR_DIM;
  if (D < 1 || D > dmax || (D * esize_of(dt)) % 16 != 0) return ADALN_ERR_DIM;
  if (nseg < 1 || nseg > ADALN_MAX_NSEG) return ADALN_ERR_DIM;
  return ADALN_OK;
}

// ----- launch-shape cache, keyed by (device, kernel, variant, dtype, D) ------
struct ShapeKey {
  int dev, which, variant, dt, D;
  bool operator==(const ShapeKey& o) const {
    return dev == o.dev && which == o.which && variant == o.variant && dt == o.dt && D == o.D;
  }
};
std::mutex g_shape_mu;
std::vector<std::pair<ShapeKey, Shape>> g_shapes;

// seg_rows: rows per segment of the whole batch (the forward's variant
// choice; a call on a chunk of a batch passes the batch's).
cudaError_t get_shape(int which, int64_t T, int32_t D, int64_t seg_rows, adaln_dtype_t dt,
                      Shape* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int nvec = D * (dt == ADALN_BF16 ? 2 : 4) / 16;
  const int variant = which == ADALN_KERNEL_FWD ? choose_fwd_variant(nvec, seg_rows)
                                                : choose_bwd_variant(nvec);
  const ShapeKey key{dev, which, variant, (int)dt, D};
  Shape full{};
  bool found = false;
  {
    std::lock_guard<std::mutex> lk(g_shape_mu);
    for (auto& kv : g_shapes)
      if (kv.first == key) { full = kv.second; found = true; break; }
  }
  if (!found) {
    // Computed with an unbounded T: grid = SMs x resident CTAs per SM.
    const int64_t big = (int64_t)1 << 40;
    e = which == ADALN_KERNEL_FWD ? fwd_shape(big, D, dt, variant, &full)
                                  : bwd_shape(big, D, dt, &full);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_shape_mu);
    g_shapes.push_back({key, full});
  }
  *out = full;
  out->grid = (int)(T < full.grid ? (T < 1 ? 1 : T) : full.grid);
  if (which == ADALN_KERNEL_BWD_ROWS && T < virtual_ctas(full)) {
    // Every team of the backward owns a row range of its own: at most T of
    // them (fewer CTAs, or one team per CTA when T < teams).
    if (T >= full.teams) {
      out->grid = (int)(T / full.teams);
    } else {
      out->teams = 1;
      out->threads = (full.nc + 1) * 32;
      out->smem = full.team_bytes;
    }
  }
  return cudaSuccess;
}

// ----- status word -----------------------------------------------------------
std::mutex g_status_mu;
unsigned* g_status_ptr[kMaxDevices] = {};

// Status word bound by the calling host thread (adaln_status_bind), or none.
thread_local unsigned* t_bound_status = nullptr;

cudaError_t status_ptr(unsigned** out) {
  if (t_bound_status != nullptr) {
    *out = t_bound_status;
    return cudaSuccess;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// ----- launch slots ----------------------------------------------------------
struct SlotPool {
  cudaEvent_t ev[kLaunchSlots] = {};
  bool recorded[kLaunchSlots] = {};
  bool pending[kLaunchSlots] = {};  // handed out, event not yet recorded
  int cursor = 0;
};
std::mutex g_slot_mu;
SlotPool g_slot_pools[kNumSlotPools][kMaxDevices];

// ----- timing trace -----------------------------------------------------------
struct TraceRec {
  int kernel;
  cudaEvent_t start, end;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
int g_trace_used = 0;
std::vector<TraceRec> g_trace;
int64_t g_trace_count[ADALN_NUM_KERNELS] = {};
double g_trace_ms[ADALN_NUM_KERNELS] = {};

template <class F>
cudaError_t traced(int kernel, cudaStream_t st, F launch) {
  TraceRec* rec = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (g_trace_on && g_trace_used < (int)g_trace.size()) {
      rec = &g_trace[g_trace_used++];
      rec->kernel = kernel;
    }
  }
  if (rec) {
    cudaError_t e = cudaEventRecord(rec->start, st);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) return e;
  if (rec) return cudaEventRecord(rec->end, st);
  return cudaSuccess;
}

int cuda_fail(cudaError_t e) {
  (void)cudaGetLastError();  // clear a sticky launch error of this thread
  (void)e;
  return ADALN_ERR_CUDA;
}

}  // namespace

namespace adaln {

int launch_slot_acquire(int pool, cudaStream_t st) {
  if (pool < 0 || pool >= kNumSlotPools) return -1;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return -1;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  std::lock_guard<std::mutex> lk(g_slot_mu);
  SlotPool& p = g_slot_pools[pool][dev];
  for (int i = 0; i < kLaunchSlots; ++i) {
    const int slot = (p.cursor + i) % kLaunchSlots;
    if (p.pending[slot]) continue;
    if (p.recorded[slot]) {
      const cudaError_t q = cudaEventQuery(p.ev[slot]);
      if (q == cudaErrorNotReady) continue;
      if (q != cudaSuccess) return -1;
    } else if (p.ev[slot] == nullptr &&
               cudaEventCreateWithFlags(&p.ev[slot], cudaEventDisableTiming) != cudaSuccess) {
      return -1;
    }
    p.pending[slot] = true;
    p.cursor = (slot + 1) % kLaunchSlots;
    return slot;
  }
  return -1;
}

cudaError_t launch_slot_release(int pool, int slot, cudaStream_t st, bool launched) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_slot_mu);
  SlotPool& p = g_slot_pools[pool][dev];
  p.pending[slot] = false;
  if (!launched) return cudaSuccess;
  e = cudaEventRecord(p.ev[slot], st);
  if (e == cudaSuccess)
    p.recorded[slot] = true;
  else
    p.pending[slot] = true;  // completion unknown: never hand it out again
  return e;
}

int run_fwd(const void* x, const void* shift, const void* scale, const int32_t* seg_id,
            int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype, float eps, void* y,
            float* mean, float* rstd, cudaStream_t st, int64_t seg_rows) {
  if (T == 0) return ADALN_OK;
  Shape s;
  cudaError_t e = get_shape(ADALN_KERNEL_FWD, T, D, seg_rows, dtype, &s);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned* status = nullptr;
  e = status_ptr(&status);
  if (e != cudaSuccess) return cuda_fail(e);
  FwdArgs a{x, shift, scale, seg_id, y, mean, rstd, T, D, nseg, eps, 1.0f / (float)D, status,
            nullptr, 0};
  e = traced(ADALN_KERNEL_FWD, st, [&] { return launch_fwd(a, dtype, s, st); });
  return e == cudaSuccess ? ADALN_OK : cuda_fail(e);
}

int run_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
            const void* scale, const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
            adaln_dtype_t dtype, void* dx, float* dshift, float* dscale, void* workspace,
            size_t workspace_bytes, cudaStream_t st, int accumulate) {
  Shape s;
  cudaError_t e = get_shape(ADALN_KERNEL_BWD_ROWS, T, D, 0, dtype, &s);
  if (e != cudaSuccess) return cuda_fail(e);
  const size_t need = bwd_workspace_bytes(s, D, nseg);
  if (workspace_bytes < need) return ADALN_ERR_WORKSPACE;
  unsigned* status = nullptr;
  e = status_ptr(&status);
  if (e != cudaSuccess) return cuda_fail(e);

  float* partials = static_cast<float*>(workspace);
  int32_t* seg_start = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) +
                                                  bwd_partials_bytes(s, D, nseg));
  BwdArgs a{dy, x, mean, rstd, scale, seg_id, dx, dshift, dscale,
            partials, seg_start, T, D, nseg, 1.0f / (float)D, status, accumulate};
  if (T > 0) {
    e = traced(ADALN_KERNEL_BWD_ROWS, st, [&] { return launch_bwd_rows(a, dtype, s, st); });
    if (e != cudaSuccess) return cuda_fail(e);
  } else if (accumulate) {
    return ADALN_OK;  // nothing to add
  }
  e = traced(ADALN_KERNEL_BWD_FINALIZE, st, [&] { return launch_bwd_finalize(a, s, st); });
  return e == cudaSuccess ? ADALN_OK : cuda_fail(e);
}

size_t bwd_workspace_need(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype, int* rc) {
  Shape s;
  cudaError_t e = get_shape(ADALN_KERNEL_BWD_ROWS, T, D, 0, dtype, &s);
  if (e != cudaSuccess) {
    *rc = cuda_fail(e);
    return 0;
  }
  *rc = ADALN_OK;
  return (bwd_workspace_bytes(s, D, nseg) + 255) & ~(size_t)255;
}

int check_dims_public(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dt) {
  return check_dims(T, D, nseg, dt);
}

}  // namespace adaln

extern "C" {

int adaln_fwd(const void* x, const void* shift, const void* scale,
              const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
              adaln_dtype_t dtype, float eps, void* y, float* mean, float* rstd,
              void* stream) {
  int rc = check_dims(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (T == 0) return ADALN_OK;
  if (!x || !shift || !scale || !seg_id || !y || !mean || !rstd) return ADALN_ERR_NULL;
  if (!aligned(x, 16) || !aligned(shift, 16) || !aligned(scale, 16) || !aligned(y, 16) ||
      !aligned(seg_id, 4) || !aligned(mean, 4) || !aligned(rstd, 4))
    return ADALN_ERR_ALIGN;
  if (!std::isfinite(eps) || eps < 0.0f) return ADALN_ERR_ARG;
  return adaln::run_fwd(x, shift, scale, seg_id, T, D, nseg, dtype, eps, y, mean, rstd,
                        static_cast<cudaStream_t>(stream), T / nseg);
}

int adaln_bwd_workspace_size(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype,
                             size_t* bytes) {
  int rc = check_dims(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (!bytes) return ADALN_ERR_NULL;
  Shape s;
  cudaError_t e = get_shape(ADALN_KERNEL_BWD_ROWS, T, D, 0, dtype, &s);
  if (e != cudaSuccess) return cuda_fail(e);
  const size_t need = bwd_workspace_bytes(s, D, nseg);
  *bytes = (need + 255) & ~(size_t)255;
  return ADALN_OK;
}

int adaln_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
              const void* scale, const int32_t* seg_id, int64_t T, int32_t D,
              int32_t nseg, adaln_dtype_t dtype, void* dx, float* dshift,
              float* dscale, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_dims(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (!dshift || !dscale || !workspace) return ADALN_ERR_NULL;
  if (T > 0 && (!dy || !x || !mean || !rstd || !scale || !seg_id || !dx)) return ADALN_ERR_NULL;
  if (!aligned(dshift, 16) || !aligned(dscale, 16) || !aligned(workspace, 16))
    return ADALN_ERR_ALIGN;
  if (T > 0 && (!aligned(dy, 16) || !aligned(x, 16) || !aligned(scale, 16) ||
                !aligned(dx, 16) || !aligned(mean, 4) || !aligned(rstd, 4) ||
                !aligned(seg_id, 4)))
    return ADALN_ERR_ALIGN;

  return adaln::run_bwd(dy, x, mean, rstd, scale, seg_id, T, D, nseg, dtype, dx, dshift, dscale,
                        workspace, workspace_bytes, static_cast<cudaStream_t>(stream), 0);
}

int adaln_get_status(uint32_t* host_bits, void* stream) {
  unsigned* p = nullptr;
  cudaError_t e = status_ptr(&p);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned bits = 0;
  e = cudaMemcpyAsync(&bits, p, sizeof bits, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof bits, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (host_bits) *host_bits = bits;
  if (bits & (ADALN_DEV_SEG_RANGE | ADALN_DEV_SEG_ORDER)) return ADALN_ERR_SEG;
  if (bits & ADALN_DEV_TIMEOUT) return ADALN_ERR_TIMEOUT;
  return ADALN_OK;
}

int adaln_status_bind(uint32_t* device_word) {
  if (device_word != nullptr && !aligned(device_word, 4)) return ADALN_ERR_ALIGN;
  t_bound_status = reinterpret_cast<unsigned*>(device_word);
  return ADALN_OK;
}

const char* adaln_strerror(int code) {
  switch (code) {
    case ADALN_OK: return "ok";
    case ADALN_ERR_NULL: return "a required pointer is NULL";
    case ADALN_ERR_DIM: return "T, D or nseg outside the supported range";
    case ADALN_ERR_ALIGN: return "a pointer is not aligned as required";
    case ADALN_ERR_DTYPE: return "unknown dtype";
    case ADALN_ERR_SEG: return "seg_id out of range or decreasing (device status)";
    case ADALN_ERR_WORKSPACE: return "workspace missing or too small";
    case ADALN_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case ADALN_ERR_ARG: return "invalid argument (eps or trace capacity)";
    case ADALN_ERR_TIMEOUT: return "an internal pipeline wait gave up (device status)";
    default: return "unknown status code";
  }
}

int adaln_trace_begin(int capacity) {
  if (capacity < 1 || capacity > (1 << 20)) return ADALN_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& r : g_trace) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.end);
  }
  g_trace.clear();
  g_trace.resize(capacity);
  for (auto& r : g_trace) {
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.end) != cudaSuccess) {
      g_trace.clear();
      return cuda_fail(cudaErrorUnknown);
    }
  }
  g_trace_used = 0;
  for (int k = 0; k < ADALN_NUM_KERNELS; ++k) {
    g_trace_count[k] = 0;
    g_trace_ms[k] = 0.0;
  }
  g_trace_on = true;
  return ADALN_OK;
}

int adaln_trace_end(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  int rc = ADALN_OK;
  for (int i = 0; i < g_trace_used; ++i) {
    TraceRec& r = g_trace[i];
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.end) != cudaSuccess) {
      rc = cuda_fail(cudaErrorUnknown);
      continue;
    }
    g_trace_count[r.kernel] += 1;
    g_trace_ms[r.kernel] += ms;
  }
  for (auto& r : g_trace) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.end);
  }
  g_trace.clear();
  g_trace_used = 0;
  return rc;
}

int adaln_trace_get(int kernel_id, int64_t* launches, double* total_ms) {
  if (kernel_id < 0 || kernel_id >= ADALN_NUM_KERNELS) return ADALN_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (launches) *launches = g_trace_count[kernel_id];
  if (total_ms) *total_ms = g_trace_ms[kernel_id];
  return ADALN_OK;
}

int adaln_selftest_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 100000) return ADALN_ERR_ARG;
  unsigned* status = nullptr;
  cudaError_t e = status_ptr(&status);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_wait_timeout_probe(status, (uint64_t)limit_us * 1000ull,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADALN_OK : cuda_fail(e);
}

int adaln_launch_shape(int which, int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype,
                       int32_t* grid, int32_t* threads, int32_t* stages, int32_t* smem_bytes) {
  int rc = check_dims(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (which != ADALN_KERNEL_FWD && which != ADALN_KERNEL_BWD_ROWS) return ADALN_ERR_ARG;
  Shape s;
  cudaError_t e = get_shape(which, T, D, T / nseg, dtype, &s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (grid) *grid = s.grid;
  if (threads) *threads = s.threads;
  if (stages) *stages = s.stages;
  if (smem_bytes) *smem_bytes = s.smem;
  return ADALN_OK;
}

}  // extern "C"
