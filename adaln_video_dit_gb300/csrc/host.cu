// One forward + backward step on host-resident tensors, pipelined in row
// chunks: while chunk i is computed, chunk i + 1 is copied in and chunk i - 1
// is copied out, on three internal streams of the device (copies in, compute,
// copies out) and a ring of kSlots staging slots in the caller's device
// scratch.  The forward and the backward row pass work per row, so each chunk
// is an ordinary call on its rows; the backward's per-segment sums are added
// chunk by chunk, in chunk order, into one device copy of dshift/dscale
// (deterministic for a given chunk size and device).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace adaln {
namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;

struct HostCtx {
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, mod = nullptr, end = nullptr;
  cudaEvent_t in[kSlots] = {}, done[kSlots] = {}, out[kSlots] = {};
};

std::mutex g_host_mu;  // one pipelined call enqueues at a time
HostCtx g_host[kMaxDevices];

cudaError_t host_ctx(HostCtx** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  HostCtx& c = g_host[dev];
  if (!c.ready) {
    const unsigned ef = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.comp, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.mod, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.end, ef);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&c.in[i], ef);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.done[i], ef);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.out[i], ef);
    }
    if (e != cudaSuccess) return e;
    c.ready = true;
  }
  *out = &c;
  return cudaSuccess;
}

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

// Offsets of the device scratch: modulation and gradient sums, the backward
// workspace of one chunk, then kSlots staging slots of one chunk each.
struct Layout {
  size_t shift, scale, dshift, dscale, ws, ws_bytes, slot0, slot_bytes;
  size_t x, dy, y, dx, mean, rstd, seg;  // within a slot
  size_t total;
};

Layout layout(int64_t C, int32_t D, int32_t nseg, adaln_dtype_t dt, size_t ws_bytes) {
  const size_t es = dt == ADALN_BF16 ? 2 : 4;
  const size_t mod = up256((size_t)nseg * D * es), grad = up256((size_t)nseg * D * 4);
  const size_t rowsz = up256((size_t)C * D * es), vec = up256((size_t)C * 4);
  Layout L;
  L.shift = 0;
  L.scale = mod;
  L.dshift = 2 * mod;
  L.dscale = 2 * mod + grad;
  L.ws = 2 * mod + 2 * grad;
  L.ws_bytes = up256(ws_bytes);
  L.slot0 = L.ws + L.ws_bytes;
  L.x = 0;
  L.dy = rowsz;
  L.y = 2 * rowsz;
  L.dx = 3 * rowsz;
  L.mean = 4 * rowsz;
  L.rstd = 4 * rowsz + vec;
  L.seg = 4 * rowsz + 2 * vec;
  L.slot_bytes = 4 * rowsz + 3 * vec;
  L.total = L.slot0 + kSlots * L.slot_bytes;
  return L;
}

int64_t default_chunk(int32_t D, adaln_dtype_t dt) {
  const int64_t row = (int64_t)D * (dt == ADALN_BF16 ? 2 : 4);
  const int64_t c = ((int64_t)32 << 20) / row;  // about 32 MB per tensor and chunk
  return c < 1 ? 1 : c;
}

int fail(cudaError_t) {
  (void)cudaGetLastError();
  return ADALN_ERR_CUDA;
}

}  // namespace
}  // namespace adaln

using namespace adaln;

extern "C" int adaln_fwd_bwd_host_scratch_size(int64_t T, int32_t D, int32_t nseg,
                                               adaln_dtype_t dtype, int64_t chunk_rows,
                                               size_t* bytes) {
  int rc = check_dims_public(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (!bytes) return ADALN_ERR_NULL;
  if (chunk_rows < 0) return ADALN_ERR_ARG;
  const int64_t C = chunk_rows ? chunk_rows : default_chunk(D, dtype);
  const size_t ws = bwd_workspace_need(C, D, nseg, dtype, &rc);
  if (rc != ADALN_OK) return rc;
  *bytes = layout(C, D, nseg, dtype, ws).total;
  return ADALN_OK;
}

extern "C" int adaln_fwd_bwd_host(const void* x, const void* dy, const void* shift,
                                  const void* scale, const int32_t* seg_id, int64_t T,
                                  int32_t D, int32_t nseg, adaln_dtype_t dtype, float eps,
                                  void* y, float* mean, float* rstd, void* dx, float* dshift,
                                  float* dscale, int64_t chunk_rows, void* scratch,
                                  size_t scratch_bytes, void* stream) {
  int rc = check_dims_public(T, D, nseg, dtype);
  if (rc != ADALN_OK) return rc;
  if (!shift || !scale || !dshift || !dscale || !scratch) return ADALN_ERR_NULL;
  if (T > 0 && (!x || !dy || !seg_id || !y || !mean || !rstd || !dx)) return ADALN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255) != 0) return ADALN_ERR_ALIGN;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return ADALN_ERR_ARG;
  if (chunk_rows < 0) return ADALN_ERR_ARG;
  const int64_t C = chunk_rows ? chunk_rows : default_chunk(D, dtype);
  const size_t ws_need = bwd_workspace_need(C, D, nseg, dtype, &rc);
  if (rc != ADALN_OK) return rc;
  const Layout L = layout(C, D, nseg, dtype, ws_need);
  if (scratch_bytes < L.total) return ADALN_ERR_WORKSPACE;

  std::lock_guard<std::mutex> lk(g_host_mu);
  HostCtx* cx = nullptr;
  cudaError_t e = host_ctx(&cx);
  if (e != cudaSuccess) return fail(e);
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(scratch);
  const size_t es = dtype == ADALN_BF16 ? 2 : 4;
  const size_t mod_bytes = (size_t)nseg * D * es, grad_bytes = (size_t)nseg * D * 4;
  float* d_dshift = reinterpret_cast<float*>(base + L.dshift);
  float* d_dscale = reinterpret_cast<float*>(base + L.dscale);

#define ADALN_CK(call)          \
  do {                          \
    e = (call);                 \
    if (e != cudaSuccess) return fail(e); \
  } while (0)

  // Everything starts after the work already queued on the caller's stream,
  // and after the previous call on this device has finished (its last copy
  // out records `end`; waiting on an event never recorded returns at once),
  // so calls from different caller streams never share the internal slots.
  ADALN_CK(cudaEventRecord(cx->start, user));
  ADALN_CK(cudaStreamWaitEvent(cx->h2d, cx->end, 0));
  ADALN_CK(cudaStreamWaitEvent(cx->h2d, cx->start, 0));
  ADALN_CK(cudaStreamWaitEvent(cx->comp, cx->start, 0));
  ADALN_CK(cudaStreamWaitEvent(cx->d2h, cx->start, 0));
  ADALN_CK(cudaMemcpyAsync(base + L.shift, shift, mod_bytes, cudaMemcpyHostToDevice, cx->h2d));
  ADALN_CK(cudaMemcpyAsync(base + L.scale, scale, mod_bytes, cudaMemcpyHostToDevice, cx->h2d));
  ADALN_CK(cudaEventRecord(cx->mod, cx->h2d));
  ADALN_CK(cudaStreamWaitEvent(cx->comp, cx->mod, 0));

  const int64_t nchunks = (T + C - 1) / C;
  if (nchunks == 0) {
    ADALN_CK(cudaMemsetAsync(d_dshift, 0, grad_bytes, cx->comp));
    ADALN_CK(cudaMemsetAsync(d_dscale, 0, grad_bytes, cx->comp));
  }
  const size_t row = (size_t)D * es;
  for (int64_t i = 0; i < nchunks; ++i) {
    const int sl = (int)(i % kSlots);
    const int64_t r0 = i * C;
    const int64_t rows = T - r0 < C ? T - r0 : C;
    unsigned char* S = base + L.slot0 + (size_t)sl * L.slot_bytes;
    // Copies in (after the slot's previous chunk has been copied out).
    if (i >= kSlots) ADALN_CK(cudaStreamWaitEvent(cx->h2d, cx->out[sl], 0));
    ADALN_CK(cudaMemcpyAsync(S + L.x, static_cast<const unsigned char*>(x) + r0 * row,
                             rows * row, cudaMemcpyHostToDevice, cx->h2d));
    ADALN_CK(cudaMemcpyAsync(S + L.dy, static_cast<const unsigned char*>(dy) + r0 * row,
                             rows * row, cudaMemcpyHostToDevice, cx->h2d));
    ADALN_CK(cudaMemcpyAsync(S + L.seg, seg_id + r0, rows * 4, cudaMemcpyHostToDevice, cx->h2d));
    ADALN_CK(cudaEventRecord(cx->in[sl], cx->h2d));
    // Compute: forward, then the backward of the chunk, its sums added in order.
    ADALN_CK(cudaStreamWaitEvent(cx->comp, cx->in[sl], 0));
    rc = run_fwd(S + L.x, base + L.shift, base + L.scale, reinterpret_cast<int32_t*>(S + L.seg),
                 rows, D, nseg, dtype, eps, S + L.y, reinterpret_cast<float*>(S + L.mean),
                 reinterpret_cast<float*>(S + L.rstd), cx->comp);
    if (rc != ADALN_OK) return rc;
    rc = run_bwd(S + L.dy, S + L.x, reinterpret_cast<float*>(S + L.mean),
                 reinterpret_cast<float*>(S + L.rstd), base + L.scale,
                 reinterpret_cast<int32_t*>(S + L.seg), rows, D, nseg, dtype, S + L.dx,
                 d_dshift, d_dscale, base + L.ws, L.ws_bytes, cx->comp, i > 0 ? 1 : 0);
    if (rc != ADALN_OK) return rc;
    ADALN_CK(cudaEventRecord(cx->done[sl], cx->comp));
    // Copies out.
    ADALN_CK(cudaStreamWaitEvent(cx->d2h, cx->done[sl], 0));
    ADALN_CK(cudaMemcpyAsync(static_cast<unsigned char*>(y) + r0 * row, S + L.y, rows * row,
                             cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaMemcpyAsync(static_cast<unsigned char*>(dx) + r0 * row, S + L.dx, rows * row,
                             cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaMemcpyAsync(mean + r0, S + L.mean, rows * 4, cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaMemcpyAsync(rstd + r0, S + L.rstd, rows * 4, cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaEventRecord(cx->out[sl], cx->d2h));
  }
  // The gradient sums, once every chunk is in.
  ADALN_CK(cudaEventRecord(cx->done[0], cx->comp));
  ADALN_CK(cudaStreamWaitEvent(cx->d2h, cx->done[0], 0));
  ADALN_CK(cudaMemcpyAsync(dshift, d_dshift, grad_bytes, cudaMemcpyDeviceToHost, cx->d2h));
  ADALN_CK(cudaMemcpyAsync(dscale, d_dscale, grad_bytes, cudaMemcpyDeviceToHost, cx->d2h));
  ADALN_CK(cudaEventRecord(cx->end, cx->d2h));
  ADALN_CK(cudaStreamWaitEvent(user, cx->end, 0));
#undef ADALN_CK
  return ADALN_OK;
}
