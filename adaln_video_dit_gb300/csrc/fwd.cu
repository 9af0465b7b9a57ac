// Fused AdaLN forward: y = (x - mean) * rstd * (1 + scale[b]) + shift[b].
//
// AdaptiveLoad, Technical summary section 2.B, forward pass: statistics are
// reduced on chip in two stages (warp shuffles, then across warps) and the
// modulation is applied in the same launch, so x is read from HBM once and y
// written once.  Here each persistent CTA streams its contiguous row range
// through a shared-memory ring (bulk async copies issued by one producer
// lane); for each round of R rows the consumer threads read their column
// slice from the stage three times (row sums -> mean; centred sum of squares
// -> rstd, the two-pass definition of the biased variance; modulate) and
// write y with 16-byte streaming stores, keeping only the segment's
// (1 + scale) and shift in registers.  Element arithmetic uses packed fp32x2
// instructions.
#include <cstdlib>

#include "ring.cuh"

namespace adaln {

// EXACT: the row fills the variant's largest consumer-warp count exactly
// (nvec = max warps x 32 x VPT: D = 1536, 3072, 5120, 8192 in bf16), so
// the warp count and row length are compile-time constants (offsets fold
// into immediates, no per-vector guards).
template <class E, int VARIANT, int R, bool EXACT>
__global__ void __launch_bounds__(variant_max_threads(VARIANT), variant_min_blocks(VARIANT))
    adaln_fwd_kernel(FwdArgs a, int nc_rt, int stages, int nvec_rt) {
  constexpr int VPT = variant_vpt(VARIANT);
  constexpr int NC_X = variant_max_warps(VARIANT);
  const int nc = EXACT ? NC_X : nc_rt;
  const int nvec = EXACT ? NC_X * 32 * VPT : nvec_rt;
  constexpr int H = E::EPV / 2;  // float2 pairs per vector
  extern __shared__ __align__(128) unsigned char smem[];
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
  bool valid[VPT];
#pragma unroll
  for (int q = 0; q < VPT; ++q) valid[q] = EXACT || j + q * NT < nvec;

  // (1 + scale) and shift of the current segment for this thread's columns.
  float2 s1[VPT][H], sh[VPT][H];
  int cur_b = -1;
  int prev_b = 0;
  if (r0 > 0) {
    int p = a.seg[r0 - 1];
    prev_b = p < 0 ? 0 : (p >= a.nseg ? a.nseg - 1 : p);
  }
  int phase = 0;

  // Segment ids are loaded one chunk ahead, so their latency hides behind
  // the current chunk's work.
  int n_sg[R];
#pragma unroll
  for (int r = 0; r < R; ++r) n_sg[r] = r < nrows ? __ldg(a.seg + r0 + r) : 0;

  // Every thread's vectors are all in the row when nvec is a multiple of the
  // consumer thread count times VPT (true for D = 1536, 3072, 5120 bf16).
  const bool all_valid = EXACT || nvec == NT * VPT;

  for (int64_t k = 0; k < nchunks; ++k) {
    const int s = (int)(k % stages);
    const uint32_t par = (uint32_t)((k / stages) & 1);
    const int rows = (int)min((int64_t)R, nrows - k * R);
    const int64_t t0 = r0 + k * R;
    int sg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      sg[r] = n_sg[r];
      const int64_t u = (k + 1) * R + r;
      n_sg[r] = u < nrows ? __ldg(a.seg + r0 + u) : 0;
    }

    // x stays in the stage until the outputs are written: each pass reads
    // its rows from shared memory (registers hold only column state).
    const bool ok = mbar_wait_bounded(rg.full(s), par, rg.abort);
    const uint32_t st0 = ring0 + s * stage_bytes;

    // One round over the chunk's rows.  FULL (all R rows present, every
    // vector of this thread in the row, pipeline ok) drops the per-row and
    // per-vector guards, so the rows' work interleaves freely.
    auto round = [&](auto full_tag) -> bool {
      constexpr bool FULL = decltype(full_tag)::value;
      // Pass 1: row sums -> mean.
      float acc[R][1];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float2 t[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if (FULL || (ok && r < rows)) {
#pragma unroll
          for (int q = 0; q < VPT; ++q) {
            if (FULL || valid[q]) {
              float2 f[H];
              E::unpack2(ld_shared_v4(st0 + (uint32_t)(r * nvec + j + q * NT) * 16), f);
#pragma unroll
              for (int e = 0; e < H; ++e) t[e & 1] = add2(t[e & 1], f[e]);
            }
          }
        }
        t[0] = add2(t[0], t[1]);
        acc[r][0] = t[0].x + t[0].y;
      }
      if (!team_sum<R, 1>(acc, ok, rg, nc, phase)) return false;
      phase ^= 1;
      float mu[R];
#pragma unroll
      for (int r = 0; r < R; ++r) mu[r] = acc[r][0] * a.inv_d;

      // Pass 2: centred sum of squares -> rstd.
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 nm = splat2(-mu[r]);
        float2 t[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if (FULL || r < rows) {
#pragma unroll
          for (int q = 0; q < VPT; ++q) {
            if (FULL || valid[q]) {
              float2 f[H];
              E::unpack2(ld_shared_v4(st0 + (uint32_t)(r * nvec + j + q * NT) * 16), f);
#pragma unroll
              for (int e = 0; e < H; ++e) {
                const float2 c = add2(f[e], nm);
                t[e & 1] = fma2(c, c, t[e & 1]);
              }
            }
          }
        }
        t[0] = add2(t[0], t[1]);
        acc[r][0] = t[0].x + t[0].y;
      }
      team_sum<R, 1>(acc, true, rg, nc, phase);
      phase ^= 1;

      // Segment bookkeeping for the chunk's rows, then the modulated outputs.
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (FULL || r < rows) {
          const int b = checked_seg(sg[r], prev_b, a.nseg, a.status);
          prev_b = b;
          sg[r] = b;
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (FULL || r < rows) {
          const int64_t t = t0 + r;
          const float rs = rsqrtf(fmaf(acc[r][0], a.inv_d, a.eps));
          const int b = sg[r];
          if (b != cur_b) {
            cur_b = b;
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
              if (valid[q]) {
                const size_t off = ((size_t)b * nvec + j + q * NT) * 16;
                E::unpack2(ld_global_v4(static_cast<const unsigned char*>(a.scale) + off), s1[q]);
                E::unpack2(ld_global_v4(static_cast<const unsigned char*>(a.shift) + off), sh[q]);
#pragma unroll
                for (int e = 0; e < H; ++e) s1[q][e] = add2(s1[q][e], splat2(1.0f));
              }
            }
          }
          const float2 nm = splat2(-mu[r]), rs2 = splat2(rs);
#pragma unroll
          for (int q = 0; q < VPT; ++q) {
            if (FULL || valid[q]) {
              const int v = j + q * NT;
              float2 f[H];
              E::unpack2(ld_shared_v4(st0 + (uint32_t)(r * nvec + v) * 16), f);
#pragma unroll
              for (int e = 0; e < H; ++e) f[e] = fma2(mul2(add2(f[e], nm), rs2), s1[q][e], sh[q][e]);
              st_global_cs_v4(static_cast<unsigned char*>(a.y) + ((size_t)t * nvec + v) * 16,
                              E::pack2(f));
            }
          }
          if (j == 0) {
            a.mean[t] = mu[r];
            a.rstd[t] = rs;
          }
        }
      }
      return true;
    };
    const bool full = ok && rows == R && all_valid;
    if (!(full ? round(Tag<true>()) : round(Tag<false>()))) {
      if (j == 0) {
        atomicOr(a.status, ADALN_DEV_TIMEOUT);
        *rg.abort = 1;
      }
      break;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(rg.empty(s));
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {

template <class E, int V>
void* fwd_kernel_for_v(bool exact) {
  return exact ? reinterpret_cast<void*>(&adaln_fwd_kernel<E, V, fwd_rows(V), true>)
               : reinterpret_cast<void*>(&adaln_fwd_kernel<E, V, fwd_rows(V), false>);
}

template <class E>
void* fwd_kernel_for(int variant, bool exact) {
  switch (variant) {
    case 0: return fwd_kernel_for_v<E, 0>(exact);
    case 1: return fwd_kernel_for_v<E, 1>(exact);
    case 2: return fwd_kernel_for_v<E, 2>(exact);
    default: return fwd_kernel_for_v<E, 3>(exact);
  }
}

void* pick_fwd(adaln_dtype_t dt, int variant, bool exact) {
  return dt == ADALN_BF16 ? fwd_kernel_for<BF16>(variant, exact) : fwd_kernel_for<F32>(variant, exact);
}

}  // namespace

// Common shape rule of the staging kernels: the compiled variant for the row
// length, consumer warps to cover the row, ring depth sized for about 160 KB
// of staged rows per SM, and persistent CTAs = SMs x resident CTAs per SM
// (at most T).
cudaError_t staging_shape(void* kernel, int64_t T, int32_t D, adaln_dtype_t dt,
                          int ntensors, int rows_per_round, int variant, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  s->row_bytes = D * esize;
  s->nvec = s->row_bytes / 16;
  s->variant = variant;
  s->exact = variant_exact(variant, s->nvec);
  s->vpt = variant_vpt(s->variant);
  s->nc = (s->nvec + 32 * s->vpt - 1) / (32 * s->vpt);
  s->threads = (s->nc + 1) * 32;

  int dev = 0, sms = 0, optin = 0, smem_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;

  // Ring depth: about 160 KB of staged rows per SM (ADALN_RING_KB overrides,
  // for launch-shape sweeps), split over the CTAs the variant is sized for,
  // and no more than fits beside them.
  const int ctas = variant_min_blocks(s->variant);
  const int stage_bytes = rows_per_round * s->row_bytes * ntensors;
  const int per_cta = smem_sm / ctas - 2048;  // room for the per-CTA reserve
  int ring_kb = 160;
  if (const char* env = getenv("ADALN_RING_KB")) {
    const int v = atoi(env);
    if (v >= 16 && v <= 256) ring_kb = v;
  }
  int budget = ring_kb * 1024 / ctas;
  if (budget > per_cta) budget = per_cta;
  int stages = budget / stage_bytes;
  stages = stages < 2 ? 2 : (stages > 16 ? 16 : stages);
  while (stages > 2 && ring_header_bytes(stages) + stages * stage_bytes > per_cta) --stages;
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
  // ADALN_CTAS_PER_SM lowers the resident CTAs per SM (launch-shape sweeps).
  if (const char* env = getenv("ADALN_CTAS_PER_SM")) {
    const int v = atoi(env);
    if (v >= 1 && v < per_sm) per_sm = v;
  }
  int64_t g = (int64_t)sms * per_sm;
  if (g > T) g = T;
  s->grid = (int)(g < 1 ? 1 : g);
  return cudaSuccess;
}

cudaError_t fwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  const int nvec = D * esize / 16;
  const int v = choose_variant(nvec);
  return staging_shape(pick_fwd(dt, v, variant_exact(v, nvec)), T, D, dt, 1, fwd_rows(v), v, s);
}

cudaError_t launch_fwd(const FwdArgs& a, adaln_dtype_t dt, const Shape& s,
                       cudaStream_t st) {
  void* k = pick_fwd(dt, s.variant, s.exact);
  int nc = s.nc, stages = s.stages, nvec = s.nvec;
  FwdArgs args = a;
  void* params[] = {&args, &nc, &stages, &nvec};
  return cudaLaunchKernel(k, dim3(s.grid), dim3(s.threads), params, s.smem, st);
}

}  // namespace adaln
