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
#include <vector>

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

// Offsets of the device scratch: modulation rows, gradient sums, seg_id,
// mean and rstd of all T rows (small: 12 bytes a row, so each crosses the
// host link in one copy rather than one per chunk), the backward workspace of
// one chunk, then kSlots staging slots of one chunk of x, dy, y, dx each.
struct Layout {
  size_t shift, scale, dshift, dscale, seg, mean, rstd, ws, ws_bytes, slot0, slot_bytes;
  size_t x, dy, y, dx;  // within a slot
  size_t total;
};

Layout layout(int64_t T, int64_t C, int32_t D, int32_t nseg, adaln_dtype_t dt,
              size_t ws_bytes) {
  const size_t es = dt == ADALN_BF16 ? 2 : 4;
  const size_t mod = up256((size_t)nseg * D * es), grad = up256((size_t)nseg * D * 4);
  const size_t vec = up256((size_t)T * 4), rowsz = up256((size_t)C * D * es);
  Layout L;
  L.shift = 0;
  L.scale = mod;
  L.dshift = 2 * mod;
  L.dscale = L.dshift + grad;
  L.seg = L.dscale + grad;
  L.mean = L.seg + vec;
  L.rstd = L.mean + vec;
  L.ws = L.rstd + vec;
  L.ws_bytes = up256(ws_bytes);
  L.slot0 = L.ws + L.ws_bytes;
  L.x = 0;
  L.dy = rowsz;
  L.y = 2 * rowsz;
  L.dx = 3 * rowsz;
  L.slot_bytes = 4 * rowsz;
  L.total = L.slot0 + kSlots * L.slot_bytes;
  return L;
}

int64_t default_chunk(int32_t D, adaln_dtype_t dt) {
  const int64_t row = (int64_t)D * (dt == ADALN_BF16 ? 2 : 4);
  const int64_t c = ((int64_t)32 << 20) / row;  // about 32 MB per tensor and chunk
  return c < 1 ? 1 : c;
}

// Row ranges of the chunks.  The first copy in and the last copy out run
// alone on the host link, so when there are enough rows the pipeline starts
// and ends with chunks of C/8, C/4 and C/2 rows; the rows between are split
// into near-equal chunks of at most C rows (no short ragged chunk).
struct Chunk {
  int64_t r0, rows;
};

std::vector<Chunk> chunk_plan(int64_t T, int64_t C) {
  std::vector<Chunk> v;
  auto split = [&v](int64_t r0, int64_t n, int64_t C) {
    const int64_t k = (n + C - 1) / C;
    for (int64_t i = 0; i < k; ++i) {
      const int64_t a = r0 + n * i / k, b = r0 + n * (i + 1) / k;
      v.push_back({a, b - a});
    }
  };
  const int64_t ramp[3] = {C / 8, C / 4, C / 2};
  const int64_t ramp_rows = 2 * (ramp[0] + ramp[1] + ramp[2]);
  if (ramp[0] < 1 || T < ramp_rows + C) {
    split(0, T, C);
    return v;
  }
  int64_t r = 0;
  for (int i = 0; i < 3; ++i) {
    v.push_back({r, ramp[i]});
    r += ramp[i];
  }
  const int64_t mid = T - ramp_rows;
  split(r, mid, C);
  r += mid;
  for (int i = 2; i >= 0; --i) {
    v.push_back({r, ramp[i]});
    r += ramp[i];
  }
  return v;
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
  *bytes = layout(T, C, D, nseg, dtype, ws).total;
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
  const Layout L = layout(T, C, D, nseg, dtype, ws_need);
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
  int32_t* d_seg = reinterpret_cast<int32_t*>(base + L.seg);
  float* d_mean = reinterpret_cast<float*>(base + L.mean);
  float* d_rstd = reinterpret_cast<float*>(base + L.rstd);

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
  if (T > 0)
    ADALN_CK(cudaMemcpyAsync(d_seg, seg_id, (size_t)T * 4, cudaMemcpyHostToDevice, cx->h2d));
  ADALN_CK(cudaEventRecord(cx->mod, cx->h2d));
  ADALN_CK(cudaStreamWaitEvent(cx->comp, cx->mod, 0));

  std::vector<Chunk> plan;
  try {
    plan = chunk_plan(T, C);
  } catch (...) {
    return ADALN_ERR_CUDA;
  }
  const int64_t nchunks = (int64_t)plan.size();
  if (nchunks == 0) {
    ADALN_CK(cudaMemsetAsync(d_dshift, 0, grad_bytes, cx->comp));
    ADALN_CK(cudaMemsetAsync(d_dscale, 0, grad_bytes, cx->comp));
  }
  const size_t row = (size_t)D * es;
  for (int64_t i = 0; i < nchunks; ++i) {
    const int sl = (int)(i % kSlots);
    const int64_t r0 = plan[i].r0, rows = plan[i].rows;
    unsigned char* S = base + L.slot0 + (size_t)sl * L.slot_bytes;
    // Copies in (after the slot's previous chunk has been copied out).
    if (i >= kSlots) ADALN_CK(cudaStreamWaitEvent(cx->h2d, cx->out[sl], 0));
    ADALN_CK(cudaMemcpyAsync(S + L.x, static_cast<const unsigned char*>(x) + r0 * row,
                             rows * row, cudaMemcpyHostToDevice, cx->h2d));
    ADALN_CK(cudaMemcpyAsync(S + L.dy, static_cast<const unsigned char*>(dy) + r0 * row,
                             rows * row, cudaMemcpyHostToDevice, cx->h2d));
    ADALN_CK(cudaEventRecord(cx->in[sl], cx->h2d));
    // Compute: forward, then the backward of the chunk, its sums added in order.
    ADALN_CK(cudaStreamWaitEvent(cx->comp, cx->in[sl], 0));
    rc = run_fwd(S + L.x, base + L.shift, base + L.scale, d_seg + r0, rows, D, nseg, dtype, eps,
                 S + L.y, d_mean + r0, d_rstd + r0, cx->comp, T / nseg);
    if (rc != ADALN_OK) return rc;
    rc = run_bwd(S + L.dy, S + L.x, d_mean + r0, d_rstd + r0, base + L.scale, d_seg + r0, rows,
                 D, nseg, dtype, S + L.dx, d_dshift, d_dscale, base + L.ws, L.ws_bytes,
                 cx->comp, i > 0 ? 1 : 0);
    if (rc != ADALN_OK) return rc;
    ADALN_CK(cudaEventRecord(cx->done[sl], cx->comp));
    // Copies out.
    ADALN_CK(cudaStreamWaitEvent(cx->d2h, cx->done[sl], 0));
    ADALN_CK(cudaMemcpyAsync(static_cast<unsigned char*>(y) + r0 * row, S + L.y, rows * row,
                             cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaMemcpyAsync(static_cast<unsigned char*>(dx) + r0 * row, S + L.dx, rows * row,
                             cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaEventRecord(cx->out[sl], cx->d2h));
  }
  // The statistics and the gradient sums, once every chunk is computed.
  ADALN_CK(cudaEventRecord(cx->done[0], cx->comp));
  ADALN_CK(cudaStreamWaitEvent(cx->d2h, cx->done[0], 0));
  if (T > 0) {
    ADALN_CK(cudaMemcpyAsync(mean, d_mean, (size_t)T * 4, cudaMemcpyDeviceToHost, cx->d2h));
    ADALN_CK(cudaMemcpyAsync(rstd, d_rstd, (size_t)T * 4, cudaMemcpyDeviceToHost, cx->d2h));
  }
  ADALN_CK(cudaMemcpyAsync(dshift, d_dshift, grad_bytes, cudaMemcpyDeviceToHost, cx->d2h));
  ADALN_CK(cudaMemcpyAsync(dscale, d_dscale, grad_bytes, cudaMemcpyDeviceToHost, cx->d2h));
  ADALN_CK(cudaEventRecord(cx->end, cx->d2h));
  ADALN_CK(cudaStreamWaitEvent(user, cx->end, 0));
#undef ADALN_CK
  return ADALN_OK;
}
