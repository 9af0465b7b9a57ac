// Fused AdaLN backward.
//
// AdaptiveLoad, Technical summary section 2.B, backward pass ("D-tile
// coalesced reduction"): the modulation gradients are reduced along the
// sequence by threads that each own a feature column d and accumulate down
// the rows, so every warp access is contiguous along d.  Here that column
// reduction is fused into the row pass: each persistent CTA streams its
// contiguous row range of x and dy through a shared-memory ring (read from
// HBM exactly once), computes dx per row, and accumulates dy * xhat and dy in
// registers of the thread that owns each column.  At a segment change and at
// the end of its range a CTA writes one fp32 partial per (CTA, segment) to
// the workspace; a second launch sums the partials of each segment in CTA
// order.  No floating-point atomics, no inter-CTA waits.
//
//   dx[t,d]      = rstd_t (g - mean_d g - xhat mean_d(g xhat)),  g = dy (1 + scale_b)
//   dscale[b,d]  = sum over rows of segment b of dy xhat
//   dshift[b,d]  = sum over rows of segment b of dy
//
// Partial slots: the (CTA c, segment b) pairs met along the rows form a
// monotone path in which every step increases c, b or both, so slot c + b is
// unique per pair and G + nseg - 1 slots suffice.
#include "ring.cuh"

namespace adaln {

template <class E, int VPT>
__device__ __forceinline__ void load_one_plus_scale(const void* scale, int b, int j,
                                                    int NT, int nvec,
                                                    float (&s1)[VPT][E::EPV]) {
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    const int v = j + q * NT;
    if (v < nvec) {
      float f[E::EPV];
      E::unpack(ld_global_v4(static_cast<const unsigned char*>(scale) +
                             ((size_t)b * nvec + v) * 16), f);
#pragma unroll
      for (int e = 0; e < E::EPV; ++e) s1[q][e] = 1.0f + f[e];
    }
  }
}

template <class E, int VPT>
__device__ __forceinline__ void flush_partials(float* partials, int64_t slot, int D,
                                               int j, int NT, int nvec,
                                               float (&acc_s)[VPT][E::EPV],
                                               float (&acc_b)[VPT][E::EPV]) {
  float* ps = partials + (size_t)slot * 2 * D;
  float* pb = ps + D;
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    const int v = j + q * NT;
    if (v < nvec) {
#pragma unroll
      for (int e = 0; e < E::EPV; e += 4) {
        *reinterpret_cast<float4*>(ps + (size_t)v * E::EPV + e) =
            make_float4(acc_s[q][e], acc_s[q][e + 1], acc_s[q][e + 2], acc_s[q][e + 3]);
        *reinterpret_cast<float4*>(pb + (size_t)v * E::EPV + e) =
            make_float4(acc_b[q][e], acc_b[q][e + 1], acc_b[q][e + 2], acc_b[q][e + 3]);
      }
    }
  }
}

template <class E, int VPT, int R>
__global__ void __launch_bounds__(max_threads(VPT), 1)
    adaln_bwd_rows_kernel(BwdArgs a, int nc, int stages, int nvec) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int EPV = E::EPV;
  const Ring rg = ring_layout(smem, stages);
  ring_init(rg, nc);

  const int64_t G = gridDim.x;
  const int64_t r0 = part_begin(blockIdx.x, a.T, G);
  const int64_t nrows = part_begin(blockIdx.x + 1, a.T, G) - r0;
  const int row_bytes = nvec * 16;
  const int warp = threadIdx.x >> 5;

  if (warp == nc) {  // producer warp: x and dy rows into each stage
    if ((threadIdx.x & 31) == 0) {
      const unsigned char* src[2] = {
          static_cast<const unsigned char*>(a.x) + (size_t)r0 * row_bytes,
          static_cast<const unsigned char*>(a.dy) + (size_t)r0 * row_bytes};
      ring_produce<R, 2>(rg, src, nrows, row_bytes, a.status);
    }
    return;
  }

  const int j = threadIdx.x;
  const int NT = nc * 32;
  const int64_t nchunks = (nrows + R - 1) / R;
  const uint32_t ring0 = smem_addr(rg.ring);
  const uint32_t stage_bytes = (uint32_t)R * row_bytes * 2;

  float acc_s[VPT][EPV], acc_b[VPT][EPV], s1[VPT][EPV];
#pragma unroll
  for (int q = 0; q < VPT; ++q)
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc_s[q][e] = acc_b[q][e] = s1[q][e] = 0.0f;
  int acc_seg = -1;  // segment whose sums are in acc_s / acc_b
  int s1_seg = -1;   // segment whose (1 + scale) is in s1
  int prev_b = 0;
  if (r0 > 0) {
    int p = a.seg[r0 - 1];
    prev_b = p < 0 ? 0 : (p >= a.nseg ? a.nseg - 1 : p);
  }
  int phase = 0;
  bool aborted = false;

  for (int64_t k = 0; k < nchunks; ++k) {
    const int s = (int)(k % stages);
    const uint32_t par = (uint32_t)((k / stages) & 1);
    const int rows = (int)min((int64_t)R, nrows - k * R);
    const int64_t t0 = r0 + k * R;
    int sg[R];
    float mu[R], rs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool in = r < rows;
      sg[r] = in ? __ldg(a.seg + t0 + r) : 0;
      mu[r] = in ? __ldg(a.mean + t0 + r) : 0.0f;
      rs[r] = in ? __ldg(a.rstd + t0 + r) : 0.0f;
    }

    // The stage stays in use until phase 2 has read it: x and dy are read
    // from shared memory in both phases instead of being held in registers.
    const bool ok = mbar_wait_bounded(rg.full(s), par, rg.abort);
    const uint32_t st0 = ring0 + s * stage_bytes;

    // Phase 1 (rows in order): segment bookkeeping, column sums, row partials.
    float part[R][2];
    int bs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      part[r][0] = part[r][1] = 0.0f;
      bs[r] = 0;
      if (r < rows && ok) {
        const int b = checked_seg(sg[r], prev_b, a.nseg, a.status);
        prev_b = b;
        bs[r] = b;
        if (b != acc_seg) {
          if (acc_seg >= 0)
            flush_partials<E, VPT>(a.partials, blockIdx.x + acc_seg, a.D, j, NT, nvec, acc_s, acc_b);
#pragma unroll
          for (int q = 0; q < VPT; ++q)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc_s[q][e] = acc_b[q][e] = 0.0f;
          acc_seg = b;
        }
        if (b != s1_seg) {
          load_one_plus_scale<E, VPT>(a.scale, b, j, NT, nvec, s1);
          s1_seg = b;
        }
#pragma unroll
        for (int q = 0; q < VPT; ++q) {
          if (j + q * NT < nvec) {
            const int v = j + q * NT;
            float fx[EPV], fd[EPV];
            E::unpack(ld_shared_v4(st0 + (uint32_t)(r * nvec + v) * 16), fx);
            E::unpack(ld_shared_v4(st0 + (uint32_t)((R + r) * nvec + v) * 16), fd);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const float xh = (fx[e] - mu[r]) * rs[r];
              const float g = fd[e] * s1[q][e];
              part[r][0] += g;
              part[r][1] = fmaf(g, xh, part[r][1]);
              acc_s[q][e] = fmaf(fd[e], xh, acc_s[q][e]);
              acc_b[q][e] += fd[e];
            }
          }
        }
      }
    }
    if (!team_sum<R, 2>(part, ok, rg, nc, phase)) {
      if (j == 0) {
        atomicOr(a.status, ADALN_DEV_TIMEOUT);
        *rg.abort = 1;
      }
      aborted = true;
      break;
    }
    phase ^= 1;

    // Phase 2 (rows in reverse, so a mid-chunk segment change reloads the
    // scale vector at most once more): dx.
#pragma unroll
    for (int r = R - 1; r >= 0; --r) {
      if (r < rows) {
        const int64_t t = t0 + r;
        if (bs[r] != s1_seg) {
          load_one_plus_scale<E, VPT>(a.scale, bs[r], j, NT, nvec, s1);
          s1_seg = bs[r];
        }
        const float mg = part[r][0] / (float)a.D;
        const float mgx = part[r][1] / (float)a.D;
#pragma unroll
        for (int q = 0; q < VPT; ++q) {
          const int v = j + q * NT;
          if (v < nvec) {
            float fx[EPV], fd[EPV];
            E::unpack(ld_shared_v4(st0 + (uint32_t)(r * nvec + v) * 16), fx);
            E::unpack(ld_shared_v4(st0 + (uint32_t)((R + r) * nvec + v) * 16), fd);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const float xh = (fx[e] - mu[r]) * rs[r];
              const float g = fd[e] * s1[q][e];
              fx[e] = rs[r] * (g - mg - xh * mgx);
            }
            st_global_cs_v4(static_cast<unsigned char*>(a.dx) + ((size_t)t * nvec + v) * 16,
                            E::pack(fx));
          }
        }
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(rg.empty(s));
  }
  if (!aborted && acc_seg >= 0)
    flush_partials<E, VPT>(a.partials, blockIdx.x + acc_seg, a.D, j, NT, nvec, acc_s, acc_b);
}

// Sum the partials of each segment in CTA order.  Block (b, column block):
// 32 float4 columns x J warps; warp w sums a contiguous run of the segment's
// CTAs, then warp 0 adds the J results in warp order.
__global__ void __launch_bounds__(32 * 16)
    adaln_bwd_finalize_kernel(BwdArgs a, int G, int J) {
  __shared__ float4 sh_s[16][32], sh_b[16][32];
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int ncol4 = a.D / 4;
  const int col4 = blockIdx.y * 32 + lane;

  // Rows of segment b: [lower_bound(b), lower_bound(b + 1)).
  int64_t sb = 0, eb = 0;
  {
    int64_t lo = 0, hi = a.T;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(a.seg + mid) < b) lo = mid + 1; else hi = mid;
    }
    sb = lo;
    hi = a.T;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(a.seg + mid) < b + 1) lo = mid + 1; else hi = mid;
    }
    eb = lo;
  }
  float4 ps = make_float4(0.f, 0.f, 0.f, 0.f), pb = ps;
  if (eb > sb && col4 < ncol4) {
    const int64_t c0 = part_owner(sb, a.T, G), c1 = part_owner(eb - 1, a.T, G);
    const int64_t n = c1 - c0 + 1;
    const int64_t lo = c0 + (n * w) / J, hi = c0 + (n * (w + 1)) / J;
    const size_t D2 = 2 * (size_t)a.D;
    for (int64_t c = lo; c < hi; ++c) {
      const float4* p = reinterpret_cast<const float4*>(a.partials + (size_t)(c + b) * D2);
      const float4 u = p[col4], v = p[ncol4 + col4];
      ps.x += u.x; ps.y += u.y; ps.z += u.z; ps.w += u.w;
      pb.x += v.x; pb.y += v.y; pb.z += v.z; pb.w += v.w;
    }
  }
  sh_s[w][lane] = ps;
  sh_b[w][lane] = pb;
  __syncthreads();
  if (w == 0 && col4 < ncol4) {
    float4 ts = sh_s[0][lane], tb = sh_b[0][lane];
    for (int i = 1; i < J; ++i) {
      const float4 u = sh_s[i][lane], v = sh_b[i][lane];
      ts.x += u.x; ts.y += u.y; ts.z += u.z; ts.w += u.w;
      tb.x += v.x; tb.y += v.y; tb.z += v.z; tb.w += v.w;
    }
    reinterpret_cast<float4*>(a.dscale + (size_t)b * a.D)[col4] = ts;
    reinterpret_cast<float4*>(a.dshift + (size_t)b * a.D)[col4] = tb;
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
cudaError_t staging_shape(void* kernel, int64_t T, int32_t D, adaln_dtype_t dt,
                          int ntensors, int rows_per_round, Shape* s);

namespace {

// Rows per reduction round of the backward: 2, except 1 for the widest rows
// (VPT = 4), whose column accumulators already fill the register budget.
constexpr int bwd_rows_per_round(int vpt) { return vpt == 4 ? 1 : kRowsPerRound; }

template <class E, int VPT>
void* rows_kernel_ptr() {
  return reinterpret_cast<void*>(&adaln_bwd_rows_kernel<E, VPT, bwd_rows_per_round(VPT)>);
}

template <class E>
void* pick_rows_e(int vpt) {
  return vpt == 1 ? rows_kernel_ptr<E, 1>()
                  : (vpt == 2 ? rows_kernel_ptr<E, 2>() : rows_kernel_ptr<E, 4>());
}

void* pick_rows(adaln_dtype_t dt, int vpt) {
  return dt == ADALN_BF16 ? pick_rows_e<BF16>(vpt) : pick_rows_e<F32>(vpt);
}

}  // namespace

cudaError_t bwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  const int nvec = D * esize / 16;
  const int vpt = choose_vpt(nvec);
  return staging_shape(pick_rows(dt, vpt), T, D, dt, 2, bwd_rows_per_round(vpt), s);
}

cudaError_t launch_bwd_rows(const BwdArgs& a, adaln_dtype_t dt, const Shape& s,
                            cudaStream_t st) {
  void* k = pick_rows(dt, s.vpt);
  int nc = s.nc, stages = s.stages, nvec = s.nvec;
  BwdArgs args = a;
  void* params[] = {&args, &nc, &stages, &nvec};
  return cudaLaunchKernel(k, dim3(s.grid), dim3(s.threads), params, s.smem, st);
}

cudaError_t launch_bwd_finalize(const BwdArgs& a, const Shape& s, cudaStream_t st) {
  // Warps per block: about 8 partials per warp for a segment spanning all
  // CTAs, fewer when many segments share the CTAs.
  const int64_t per_seg = ((int64_t)s.grid + a.nseg - 1) / a.nseg;
  int J = (int)((per_seg + 7) / 8);
  J = J < 1 ? 1 : (J > 16 ? 16 : J);
  int G = s.grid;
  BwdArgs args = a;
  void* params[] = {&args, &G, &J};
  const dim3 grid((unsigned)a.nseg, (unsigned)((a.D / 4 + 31) / 32));
  return cudaLaunchKernel(reinterpret_cast<void*>(&adaln_bwd_finalize_kernel), grid,
                          dim3(32 * J), params, 0, st);
}

}  // namespace adaln
