// Fused AdaLN forward: y = (x - mean) * rstd * (1 + scale[b]) + shift[b].
//
// AdaptiveLoad, Technical summary section 2.B, forward pass: statistics are
// reduced on chip in two stages (warp shuffles, then across warps) and the
// modulation is applied in the same launch, so x is read from HBM once and y
// written once.  Here each persistent CTA streams its contiguous row range
// through a shared-memory ring (bulk async copies issued by one producer
// lane); consumer threads hold their column slice of R rows in registers,
// compute the row mean, then the centred sum of squares (two-pass, exact
// definition of the biased variance), and write y with 16-byte streaming
// stores.
#include "ring.cuh"

namespace adaln {

template <class E, int VPT, int R>
__global__ void __launch_bounds__(max_threads(VPT), 1)
    adaln_fwd_kernel(FwdArgs a, int nc, int stages, int nvec) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int EPV = E::EPV;
  const Ring rg = ring_layout(smem, stages);
  ring_init(rg, nc);

  const int64_t G = gridDim.x;
  const int64_t r0 = part_begin(blockIdx.x, a.T, G);
  const int64_t nrows = part_begin(blockIdx.x + 1, a.T, G) - r0;
  const int row_bytes = nvec * 16;
  const int warp = threadIdx.x >> 5;

  if (warp == nc) {  // producer warp
    if ((threadIdx.x & 31) == 0) {
      const unsigned char* src[1] = {
          static_cast<const unsigned char*>(a.x) + (size_t)r0 * row_bytes};
      ring_produce<R, 1>(rg, src, nrows, row_bytes, a.status);
    }
    return;
  }

  const int j = threadIdx.x;
  const int NT = nc * 32;
  const int64_t nchunks = (nrows + R - 1) / R;
  const uint32_t ring0 = smem_addr(rg.ring);
  const uint32_t stage_bytes = (uint32_t)R * row_bytes;

  // Modulation of the current segment for this thread's columns.
  float s1[VPT][EPV], sh[VPT][EPV];
  int cur_b = -1;
  int prev_b = 0;
  if (r0 > 0) {
    int p = a.seg[r0 - 1];
    prev_b = p < 0 ? 0 : (p >= a.nseg ? a.nseg - 1 : p);
  }
  int phase = 0;

  for (int64_t k = 0; k < nchunks; ++k) {
    const int s = (int)(k % stages);
    const uint32_t par = (uint32_t)((k / stages) & 1);
    const int rows = (int)min((int64_t)R, nrows - k * R);
    const int64_t t0 = r0 + k * R;
    int sg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sg[r] = r < rows ? __ldg(a.seg + t0 + r) : 0;

    const bool ok = mbar_wait_bounded(rg.full(s), par, rg.abort);
    uint4 xv[R][VPT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int v = j + q * NT;
        xv[r][q] = make_uint4(0, 0, 0, 0);
        if (ok && r < rows && v < nvec)
          xv[r][q] = ld_shared_v4(ring0 + s * stage_bytes + (uint32_t)(r * nvec + v) * 16);
      }
    __syncwarp();
    if (ok && (threadIdx.x & 31) == 0) mbar_arrive(rg.empty(s));

    // Pass 1: row sums -> mean.
    float acc[R][1];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float t = 0.0f;
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        float f[EPV];
        E::unpack(xv[r][q], f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) t += f[e];
      }
      acc[r][0] = t;
    }
    if (!team_sum<R, 1>(acc, ok, rg, nc, phase)) {
      if (j == 0) {
        atomicOr(a.status, ADALN_DEV_TIMEOUT);
        *rg.abort = 1;
      }
      break;
    }
    phase ^= 1;
    float mu[R];
#pragma unroll
    for (int r = 0; r < R; ++r) mu[r] = acc[r][0] / (float)a.D;

    // Pass 2: centred sum of squares -> rstd.
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float t = 0.0f;
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        if (j + q * NT < nvec) {
          float f[EPV];
          E::unpack(xv[r][q], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float c = f[e] - mu[r];
            t = fmaf(c, c, t);
          }
        }
      }
      acc[r][0] = t;
    }
    team_sum<R, 1>(acc, true, rg, nc, phase);
    phase ^= 1;

    // Modulate and store.
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r >= rows) break;
      const int64_t t = t0 + r;
      const float rs = 1.0f / sqrtf(acc[r][0] / (float)a.D + a.eps);
      const int b = checked_seg(sg[r], prev_b, a.nseg, a.status);
      prev_b = b;
      if (b != cur_b) {
        cur_b = b;
#pragma unroll
        for (int q = 0; q < VPT; ++q) {
          const int v = j + q * NT;
          if (v < nvec) {
            const size_t off = ((size_t)b * nvec + v) * 16;
            float fs[EPV], fh[EPV];
            E::unpack(ld_global_v4(static_cast<const unsigned char*>(a.scale) + off), fs);
            E::unpack(ld_global_v4(static_cast<const unsigned char*>(a.shift) + off), fh);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              s1[q][e] = 1.0f + fs[e];
              sh[q][e] = fh[e];
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        const int v = j + q * NT;
        if (v < nvec) {
          float f[EPV];
          E::unpack(xv[r][q], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) f[e] = fmaf((f[e] - mu[r]) * rs, s1[q][e], sh[q][e]);
          st_global_cs_v4(static_cast<unsigned char*>(a.y) + ((size_t)t * nvec + v) * 16,
                          E::pack(f));
        }
      }
      if (j == 0) {
        a.mean[t] = mu[r];
        a.rstd[t] = rs;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {

template <class E, int VPT>
void* fwd_kernel_ptr() {
  return reinterpret_cast<void*>(&adaln_fwd_kernel<E, VPT, kRowsPerRound>);
}

template <class E>
void* pick_fwd_e(int vpt) {
  return vpt == 1 ? fwd_kernel_ptr<E, 1>()
                  : (vpt == 2 ? fwd_kernel_ptr<E, 2>() : fwd_kernel_ptr<E, 4>());
}

void* pick_fwd(adaln_dtype_t dt, int vpt) {
  return dt == ADALN_BF16 ? pick_fwd_e<BF16>(vpt) : pick_fwd_e<F32>(vpt);
}

}  // namespace

// Common shape rule of the staging kernels: vectors per thread (1, 2 or 4),
// consumer warps, ring depth sized for roughly `ring_target` bytes in flight
// per SM, and persistent CTAs = SMs x resident CTAs per SM (at most T).
cudaError_t staging_shape(void* kernel, int64_t T, int32_t D, adaln_dtype_t dt,
                          int ntensors, int rows_per_round, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  s->row_bytes = D * esize;
  s->nvec = s->row_bytes / 16;
  s->vpt = choose_vpt(s->nvec);
  s->nc = (s->nvec + 32 * s->vpt - 1) / (32 * s->vpt);
  s->threads = (s->nc + 1) * 32;

  int dev = 0, sms = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;

  // Target CTAs per SM by warps (about 16 resident warps), then ring depth.
  const int ctas_target = s->nc + 1 >= 16 ? 1 : 16 / (s->nc + 1);
  const int ring_target = 160 * 1024 / ctas_target;
  const int stage_bytes = rows_per_round * s->row_bytes * ntensors;
  int stages = ring_target / stage_bytes;
  stages = stages < 2 ? 2 : (stages > 16 ? 16 : stages);
  while (stages > 2 && ring_header_bytes(stages) + stages * stage_bytes > optin) --stages;
  s->stages = stages;
  s->smem = ring_header_bytes(stages) + stages * stage_bytes;
  if (s->smem > optin) return cudaErrorInvalidValue;

  // Allow the device maximum: other D values reuse this template instance
  // with larger rings.
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, s->threads, s->smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t g = (int64_t)sms * per_sm;
  if (g > T) g = T;
  s->grid = (int)(g < 1 ? 1 : g);
  return cudaSuccess;
}

cudaError_t fwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  const int nvec = D * esize / 16;
  return staging_shape(pick_fwd(dt, choose_vpt(nvec)), T, D, dt, 1, kRowsPerRound, s);
}

cudaError_t launch_fwd(const FwdArgs& a, adaln_dtype_t dt, const Shape& s,
                       cudaStream_t st) {
  void* k = pick_fwd(dt, s.vpt);
  int nc = s.nc, stages = s.stages, nvec = s.nvec;
  FwdArgs args = a;
  void* params[] = {&args, &nc, &stages, &nvec};
  return cudaLaunchKernel(k, dim3(s.grid), dim3(s.threads), params, s.smem, st);
}

}  // namespace adaln
