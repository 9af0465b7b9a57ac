// Fused AdaLN backward.
//
// AdaptiveLoad, Technical summary section 2.B, backward pass ("D-tile
// coalesced reduction"): the modulation gradients are reduced along the
// sequence by threads that each own a feature column d and accumulate down
// the rows, so every warp access is contiguous along d.  Here that column
// reduction is fused into the row pass: each persistent team (consumer warps
// + a producer warp; a CTA per SM holds one to three) streams the contiguous
// row range of its virtual CTA through a shared-memory ring (x and dy read
// from HBM exactly once), computes dx per row (phase 1: the two row sums and
// the column sums; phase 2: dx, both reading the rows from the stage), and
// accumulates dy * xhat and dy in registers of the thread that owns each
// column.  At a segment change and at the end of its range a team writes one
// fp32 partial per (virtual CTA, segment) to the workspace, and records the
// first row of every segment it starts; a second launch (a programmatic
// dependent) sums the partials of each segment in virtual-CTA order, finding
// the segment's rows in that table or, when its grid fits one wave, in seg_id
// itself.  No floating-point atomics, no inter-CTA waits.
//
//   dx[t,d]      = rstd_t (g - mean_d g - xhat mean_d(g xhat)),  g = dy (1 + scale_b)
//   dscale[b,d]  = sum over rows of segment b of dy xhat
//   dshift[b,d]  = sum over rows of segment b of dy
//
// Partial slots: the (virtual CTA v, segment b) pairs met along the rows form
// a monotone path in which every step increases v, b or both, so slot v + b
// is unique per pair and G + nseg - 1 slots suffice (G virtual CTAs).
#include "ring.cuh"

namespace adaln {

// (1 + scale[b]) for this thread's columns, as fp32 pairs.
template <class E, int VPT>
__device__ __forceinline__ void load_one_plus_scale(const void* scale, int b, int j, int NT,
                                                    const bool (&valid)[VPT], int nvec,
                                                    float2 (&s1)[VPT][E::EPV / 2]) {
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    if (valid[q]) {
      E::unpack2(ld_global_v4(static_cast<const unsigned char*>(scale) +
                              ((size_t)b * nvec + j + q * NT) * 16), s1[q]);
#pragma unroll
      for (int e = 0; e < E::EPV / 2; ++e) s1[q][e] = add2(s1[q][e], splat2(1.0f));
    }
  }
}

// Write this thread's column sums as partial slot `slot`: [dscale | dshift].
template <class E, int VPT>
__device__ __forceinline__ void flush_partials(float* partials, int64_t slot, int D, int j,
                                               int NT, const bool (&valid)[VPT],
                                               const float2 (&acc_s)[VPT][E::EPV / 2],
                                               const float2 (&acc_b)[VPT][E::EPV / 2]) {
  float* ps = partials + (size_t)slot * 2 * D;
  float* pb = ps + D;
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    if (valid[q]) {
      const size_t c0 = (size_t)(j + q * NT) * E::EPV;
#pragma unroll
      for (int e = 0; e < E::EPV / 2; e += 2) {
        *reinterpret_cast<float4*>(ps + c0 + 2 * e) =
            make_float4(acc_s[q][e].x, acc_s[q][e].y, acc_s[q][e + 1].x, acc_s[q][e + 1].y);
        *reinterpret_cast<float4*>(pb + c0 + 2 * e) =
            make_float4(acc_b[q][e].x, acc_b[q][e].y, acc_b[q][e + 1].x, acc_b[q][e + 1].y);
      }
    }
  }
}

// Chunks of R rows per ring stage, R rows per reduction round.  Consumers
// walk the CTA's rows as runs of equal segment id: an inner loop over the
// chunks of one run (no flush inside, so the column accumulators stay in
// registers) and the flush of the run's partial between runs.  A chunk that
// a segment boundary splits is visited once per run, each visit handling its
// rows of that run; its stage is released after the last visit.
// NCX: 0 for the generic instantiation (warp count and row length at run
// time), else a consumer-warp count the row fills exactly (nvec = NCX x 32 x
// VPT; the counts compiled_exact lists), which makes both compile-time
// constants (offsets fold into immediates, no per-vector guards).
//
// A CTA holds `teams` teams (one per SM share of the variant); team k of CTA c
// owns the contiguous row range of virtual CTA v = c * teams + k, so the
// ranges, partial slots and sums are those of teams x grid independent CTAs,
// while the teams of one SM, being one CTA, get equal shares of it (two
// separate CTAs on an SM run up to a tenth apart).
template <class E, int VARIANT, int R, int NCX>
__global__ void __launch_bounds__(variant_min_blocks(VARIANT) * variant_max_threads(VARIANT), 1)
    adaln_bwd_rows_kernel(BwdArgs a, int nc_rt, int stages, int nvec_rt, int team_bytes) {
  constexpr int VPT = variant_vpt(VARIANT);
  constexpr bool EXACT = NCX != 0;
  const int nc = EXACT ? NCX : nc_rt;
  const int nvec = EXACT ? NCX * 32 * VPT : nvec_rt;
  constexpr int H = E::EPV / 2;
  extern __shared__ __align__(128) unsigned char smem[];
  const int team_threads = (nc + 1) * 32;
  const int teams = blockDim.x / team_threads;
  const int team = threadIdx.x / team_threads;
  const int lt = threadIdx.x - team * team_threads;  // thread index in the team
  const Ring rg = ring_layout(smem + team * team_bytes, stages, 1 + team, team * (nc + 1));
  if (lt == 0) ring_init_team(rg, nc);
  __syncthreads();
  // Launched as a programmatic dependent of the stream's previous kernel
  // (typically the forward that wrote mean and rstd): nothing in global
  // memory is read before that kernel has completed.  Only then may the
  // finalize be scheduled (as SMs free up): it reads seg_id before waiting
  // for this grid, so every kernel before this one must have completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int64_t G = (int64_t)gridDim.x * teams;  // virtual CTAs
  const int64_t v = (int64_t)blockIdx.x * teams + team;
  const int64_t r0 = part_begin(v, a.T, G);
  const int64_t nrows = part_begin(v + 1, a.T, G) - r0;
  const int row_bytes = nvec * 16;
  const int warp = lt >> 5;

  if (warp == nc) {  // producer warp: R rows of x, then R rows of dy, per stage
    if ((lt & 31) == 0) {
      const unsigned char* src[2] = {
          static_cast<const unsigned char*>(a.x) + (size_t)r0 * row_bytes,
          static_cast<const unsigned char*>(a.dy) + (size_t)r0 * row_bytes};
      ring_produce<R, 2>(rg, src, nrows, row_bytes, a.status);
    }
    return;
  }

  const int j = lt;
  const int NT = nc * 32;
  const int64_t nchunks = (nrows + R - 1) / R;
  const uint32_t ring0 = smem_addr(rg.ring);
  const uint32_t stage_bytes = (uint32_t)R * row_bytes * 2;
  bool valid[VPT];
#pragma unroll
  for (int q = 0; q < VPT; ++q) valid[q] = EXACT || j + q * NT < nvec;

  float2 acc_s[VPT][H], acc_b[VPT][H], s1[VPT][H];
  int s1_seg = -1;  // segment whose (1 + scale) is in s1
  // Clamped segment of the row before the current chunk (-1 before row 0).
  int prev_last = -1;
  if (r0 > 0) {
    int p = a.seg[r0 - 1];
    prev_last = p < 0 ? 0 : (p >= a.nseg ? a.nseg - 1 : p);
  }
  int phase = 0;
  bool aborted = false;

  // Row metadata of the current chunk (cb: clamped segment ids) and, loaded
  // one chunk ahead so the latency hides behind a chunk's work, of the next.
  int cb[R], nb[R];
  float cmu[R], crs[R], nmu[R], nrs[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool in = r < nrows;
    nb[r] = in ? __ldg(a.seg + r0 + r) : 0;
    nmu[r] = in ? __ldg(a.mean + r0 + r) : 0.0f;
    nrs[r] = in ? __ldg(a.rstd + r0 + r) : 0.0f;
  }
  // Move the prefetched metadata of chunk kk into cb/cmu/crs (checking the
  // segment ids), then start loading chunk kk + 1.
  auto advance = [&](int64_t kk) {
    const int rows = (int)min((int64_t)R, nrows - kk * R);
    int before = prev_last < 0 ? 0 : prev_last;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      cmu[r] = nmu[r];
      crs[r] = nrs[r];
      cb[r] = 0;
      if (r < rows) {
        cb[r] = checked_seg(nb[r], before, a.nseg, a.status);
        before = cb[r];
      }
      const int64_t u = (kk + 1) * R + r;
      const bool in = u < nrows;
      nb[r] = in ? __ldg(a.seg + r0 + u) : 0;
      nmu[r] = in ? __ldg(a.mean + r0 + u) : 0.0f;
      nrs[r] = in ? __ldg(a.rstd + r0 + u) : 0.0f;
    }
  };
  advance(0);

  int64_t k = 0;  // current chunk
  int ks = 0;     // its ring stage, k % stages (kept by increment: no 64-bit division)
  uint32_t kpar = 0;  // parity of its use of that stage, (k / stages) & 1
  int lo = 0;     // first row of chunk k not yet processed
  bool ok = true;
  while (k < nchunks && !aborted) {
    // Start a run at row (k, lo).  Its first row is recorded in the segment
    // start table, together with that of every empty segment between the
    // previous row's segment and this one (each entry has one writer: the CTA
    // owning the row).
    int run_seg = cb[0];
    int before = prev_last;
#pragma unroll
    for (int r = 1; r < R; ++r)
      if (r == lo) { run_seg = cb[r]; before = cb[r - 1]; }
    for (int b = before + 1 + j; b <= run_seg; b += NT)
      a.seg_start[b] = (int32_t)(r0 + k * R + lo);
#pragma unroll
    for (int q = 0; q < VPT; ++q)
#pragma unroll
      for (int e = 0; e < H; ++e) acc_s[q][e] = acc_b[q][e] = make_float2(0.f, 0.f);
    if (run_seg != s1_seg) {
      load_one_plus_scale<E, VPT>(a.scale, run_seg, j, NT, valid, nvec, s1);
      s1_seg = run_seg;
    }

    while (k < nchunks) {
      const int rows = (int)min((int64_t)R, nrows - k * R);
      // Rows [lo, hi) of this chunk belong to the run.
      int hi = lo;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r == hi && r < rows && cb[r] == run_seg) hi = r + 1;
      if (hi == lo) break;  // row lo starts the next run

      const int s = ks;
      if (lo == 0) ok = mbar_wait_bounded(rg.full(s), kpar, rg.abort);
      const uint32_t st0 = ring0 + s * stage_bytes;

      // Phase 1: xhat, g; column sums; the two row partials.
      float part[R][2];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        part[r][0] = part[r][1] = 0.0f;
        if (ok && r >= lo && r < hi) {
          // xhat = x rstd - mean rstd: one FMA per element.
          const float2 r2 = splat2(crs[r]), nmr = splat2(-cmu[r] * crs[r]);
          float2 p0 = make_float2(0.f, 0.f), p1 = p0;
#pragma unroll
          for (int q = 0; q < VPT; ++q) {
            if (valid[q]) {
              const int v = j + q * NT;
              float2 fx[H], fd[H];
              E::unpack2(ld_shared_v4(st0 + (uint32_t)(r * nvec + v) * 16), fx);
              E::unpack2(ld_shared_v4(st0 + (uint32_t)((R + r) * nvec + v) * 16), fd);
#pragma unroll
              for (int e = 0; e < H; ++e) {
                const float2 xh = fma2(fx[e], r2, nmr);
                const float2 g = mul2(fd[e], s1[q][e]);
                p0 = add2(p0, g);
                p1 = fma2(g, xh, p1);
                acc_s[q][e] = fma2(fd[e], xh, acc_s[q][e]);
                acc_b[q][e] = add2(acc_b[q][e], fd[e]);
              }
            }
          }
          part[r][0] = p0.x + p0.y;
          part[r][1] = p1.x + p1.y;
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

      // Phase 2: dx = rstd (g - mean g - xhat mean(g xhat)), rearranged as
      //   dx = dy (rstd (1 + scale)) + x k1 + (k0 - mean k1),
      //   k1 = -rstd^2 mean(g xhat),  k0 = -rstd mean(g)
      // (three packed operations per pair of elements).
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r >= lo && r < hi) {
          const int64_t t = r0 + k * R + r;
          const float2 r2 = splat2(crs[r]);
          const float k1s = -(crs[r] * crs[r]) * (part[r][1] * a.inv_d);
          const float2 k1 = splat2(k1s);
          const float2 k0 = splat2(fmaf(-cmu[r], k1s, -crs[r] * (part[r][0] * a.inv_d)));
#pragma unroll
          for (int q = 0; q < VPT; ++q) {
            if (valid[q]) {
              const int v = j + q * NT;
              float2 fx[H], fd[H];
              E::unpack2(ld_shared_v4(st0 + (uint32_t)(r * nvec + v) * 16), fx);
              E::unpack2(ld_shared_v4(st0 + (uint32_t)((R + r) * nvec + v) * 16), fd);
#pragma unroll
              for (int e = 0; e < H; ++e)
                fx[e] = fma2(fd[e], mul2(s1[q][e], r2), fma2(fx[e], k1, k0));
              st_global_cs_v4(static_cast<unsigned char*>(a.dx) + ((size_t)t * nvec + v) * 16,
                              E::pack2(fx));
            }
          }
        }
      }

      if (hi < rows) {  // a segment boundary inside the chunk: next run
        lo = hi;
        break;
      }
      __syncwarp();
      if ((lt & 31) == 0) mbar_arrive(rg.empty(s));
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r == rows - 1) prev_last = cb[r];
      ++k;
      if (++ks == stages) {
        ks = 0;
        kpar ^= 1;
      }
      lo = 0;
      if (k < nchunks) advance(k);
    }
    if (!aborted)
      flush_partials<E, VPT>(a.partials, v + run_seg, a.D, j, NT, valid, acc_s, acc_b);
  }
  // The CTA owning the last row closes the table: segments after the last
  // one present start (and end) at T.
  if (!aborted && r0 + nrows == a.T)
    for (int b = prev_last + 1 + j; b <= a.nseg; b += NT) a.seg_start[b] = (int32_t)a.T;
}

// Sum the partials of each segment in CTA order.  A slot holds 2D floats
// (dscale partial, then dshift partial), read as 2D/4 float4 columns.  A block
// of 256 threads covers CB = 256 / GPC consecutive float4 columns of one
// segment; each column is split over GPC slot groups (contiguous runs of the
// segment's CTAs, each summed in slot order with up to 8 loads in flight),
// and the group sums are combined by a fixed pairwise tree.  GPC follows the
// number of partials per segment: 1 when segments are short (each thread a
// column, blocks span 256 columns), up to 64 for a segment spanning every CTA.
// The order of every sum is fixed by (T, G, nseg), so results are bitwise
// reproducible.  Launched as a programmatic dependent of the row pass: it
// waits (griddepcontrol.wait) until the row pass has completed and its writes
// are visible, reading only seg_id (an input) before that.
constexpr int kFinalizeThreads = 256;

// First rows of segments b and b + 1 in the sorted seg_id (lower bounds of b
// and b + 1, T when absent), found by the whole block: each round probes 256
// evenly spaced rows of the remaining range and counts those below the
// target (__syncthreads_count), which narrows the range 256-fold, so T rows
// take ceil(log256 T) + 1 rounds of one load each.  On unsorted (invalid)
// input the results are some rows in [0, T].
__device__ __forceinline__ void segment_rows(const int32_t* seg, int64_t T, int b,
                                             int64_t& sb, int64_t& eb) {
  int64_t lo[2] = {0, 0}, hi[2] = {T, T};
  while (hi[0] > lo[0] || hi[1] > lo[1]) {
    int n[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t step = (hi[k] - lo[k] + kFinalizeThreads - 1) / kFinalizeThreads;
      const int64_t p = lo[k] + threadIdx.x * step;
      const bool below = hi[k] > lo[k] && p < hi[k] && __ldg(seg + p) < b + k;
      n[k] = __syncthreads_count(below);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (hi[k] <= lo[k]) continue;
      const int64_t step = (hi[k] - lo[k] + kFinalizeThreads - 1) / kFinalizeThreads;
      if (n[k] == 0) {
        hi[k] = lo[k];  // the first probe is not below: the bound is lo
      } else {
        // Probes 0 .. n-1 are below the target, probe n is not.
        const int64_t top = lo[k] + n[k] * step;
        lo[k] += (n[k] - 1) * step + 1;
        if (top < hi[k]) hi[k] = top;
      }
    }
  }
  sb = lo[0];
  eb = lo[1];
}

__global__ void __launch_bounds__(kFinalizeThreads, 4)
    adaln_bwd_finalize_kernel(BwdArgs a, int G, int gpc, int search) {
  __shared__ float4 sh[kFinalizeThreads];
  const int b = blockIdx.x;
  const int cb = kFinalizeThreads / gpc;   // columns per block
  const int ncol4 = a.D / 4;               // float4 columns of one half
  const int cl = threadIdx.x % cb, g = threadIdx.x / cb;
  const int col4 = blockIdx.y * cb + cl;   // in [0, 2 ncol4)

  // Rows of segment b, [sb, eb): with `search`, found in seg_id (an input)
  // while the row pass still runs; else from the segment start table the
  // row pass records.  Both agree on valid input.  Clamped so that
  // inconsistent input (reported in the status word) still reads inside the
  // workspace.
  int64_t sb = 0, eb = 0;
  if (search && a.T > 0) segment_rows(a.seg, a.T, b, sb, eb);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The stream's next kernel (this library's row kernels wait before
  // reading) may be scheduled as this grid's blocks finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!search && a.T > 0) {
    sb = a.seg_start[b];
    eb = a.seg_start[b + 1];
  }
  sb = sb < 0 ? 0 : (sb > a.T ? a.T : sb);
  eb = eb < 0 ? 0 : (eb > a.T ? a.T : eb);
  float4 ps = make_float4(0.f, 0.f, 0.f, 0.f);
  if (eb > sb && col4 < 2 * ncol4) {
    const int64_t c0 = part_owner(sb, a.T, G), c1 = part_owner(eb - 1, a.T, G);
    const int64_t n = c1 - c0 + 1;
    const int64_t lo = c0 + (n * g) / gpc, hi = c0 + (n * (g + 1)) / gpc;
    const size_t row4 = 2 * (size_t)ncol4;  // float4 per slot
    const float4* base = reinterpret_cast<const float4*>(a.partials) + col4;
    for (int64_t c = lo; c < hi; c += 8) {
      float4 u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c + i < hi) u[i] = __ldcs(base + (size_t)(c + i + b) * row4);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c + i < hi) {
          ps.x += u[i].x; ps.y += u[i].y; ps.z += u[i].z; ps.w += u[i].w;
        }
      }
    }
  }
  if (gpc > 1) {
    sh[threadIdx.x] = ps;
    __syncthreads();
    // Fixed pairwise tree over the groups: group g absorbs group g + h.
    for (int h = gpc / 2; h >= 1; h >>= 1) {
      if (g < h) {
        const float4 u = sh[threadIdx.x + h * cb];
        ps.x += u.x; ps.y += u.y; ps.z += u.z; ps.w += u.w;
        sh[threadIdx.x] = ps;
      }
      __syncthreads();
    }
  }
  if (g == 0 && col4 < 2 * ncol4) {
    float4* o = col4 < ncol4
                    ? reinterpret_cast<float4*>(a.dscale + (size_t)b * a.D) + col4
                    : reinterpret_cast<float4*>(a.dshift + (size_t)b * a.D) + (col4 - ncol4);
    if (!a.accumulate) {
      *o = ps;
    } else if (eb > sb) {  // a chunk of a row-chunked call: add, in chunk order
      const float4 u = *o;
      *o = make_float4(u.x + ps.x, u.y + ps.y, u.z + ps.z, u.w + ps.w);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
cudaError_t staging_shape(void* kernel, int64_t T, int32_t D, adaln_dtype_t dt,
                          int ntensors, int rows_per_round, int variant, int teams,
                          int cta_header, Shape* s);

namespace {

template <class E, int V, int NCX>
void* rows_inst() {
  return reinterpret_cast<void*>(&adaln_bwd_rows_kernel<E, V, bwd_rows(V), NCX>);
}

// The instantiation for (variant, fixed warp count or 0); compiled_exact lists
// the fixed counts.
template <class E>
void* rows_kernel_for(int variant, int ncx) {
  switch (variant) {
    case 6: return ncx == 1 ? rows_inst<E, 6, 1>() : ncx == 2 ? rows_inst<E, 6, 2>()
                 : ncx == 3 ? rows_inst<E, 6, 3>() : rows_inst<E, 6, 0>();
    case 4: return ncx == 2 ? rows_inst<E, 4, 2>() : ncx == 3 ? rows_inst<E, 4, 3>()
                 : rows_inst<E, 4, 0>();
    case 2: return ncx == 4 ? rows_inst<E, 2, 4>() : ncx == 5 ? rows_inst<E, 2, 5>()
                 : rows_inst<E, 2, 0>();
    default: return ncx == 6 ? rows_inst<E, 3, 6>() : ncx == 8 ? rows_inst<E, 3, 8>()
                  : rows_inst<E, 3, 0>();
  }
}

void* pick_rows(adaln_dtype_t dt, int variant, int ncx) {
  return dt == ADALN_BF16 ? rows_kernel_for<BF16>(variant, ncx) : rows_kernel_for<F32>(variant, ncx);
}

}  // namespace

cudaError_t bwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  const int nvec = D * esize / 16;
  const int v = choose_bwd_variant(nvec);
  return staging_shape(pick_rows(dt, v, exact_warps(v, nvec)), T, D, dt, 2, bwd_rows(v), v,
                       variant_min_blocks(v), 0, s);
}

cudaError_t launch_bwd_rows(const BwdArgs& a, adaln_dtype_t dt, const Shape& s,
                            cudaStream_t st) {
  void* k = pick_rows(dt, s.variant, s.ncx);
  int nc = s.nc, stages = s.stages, nvec = s.nvec, team_bytes = s.team_bytes;
  BwdArgs args = a;
  void* params[] = {&args, &nc, &stages, &nvec, &team_bytes};
  return launch_dependent(k, s, params, st);
}

cudaError_t launch_bwd_finalize(const BwdArgs& a, const Shape& s, cudaStream_t st) {
  // Slot groups per column: about 4-8 partials per group for the longest
  // segments (power of two, 1..64; one round of 8 loads in flight per
  // thread), a single group when segments are short.
  const int64_t per_seg = (virtual_ctas(s) + a.nseg - 1) / a.nseg;
  int gpc = 1;
  while (gpc < 64 && per_seg > 8 * gpc) gpc *= 2;
  // The blocks start only as the row pass frees SMs, 4 per SM: when the grid
  // would need a second wave, and half the groups (two rounds of loads per
  // thread) would not, take half.
  auto blocks = [&](int g) {
    const int64_t cb = kFinalizeThreads / g;
    return (int64_t)a.nseg * ((2 * (a.D / 4) + cb - 1) / cb);
  };
  if (gpc > 1 && blocks(gpc) > 4 * (int64_t)s.sms && blocks(gpc / 2) <= 4 * (int64_t)s.sms)
    gpc /= 2;
  int G = (int)virtual_ctas(s);
  // One wave of blocks starts while the row pass ends: they find their
  // segment's rows in seg_id meanwhile.  With more blocks, the later ones
  // start after the row pass and read the recorded table instead.
  int search = blocks(gpc) <= 4 * (int64_t)s.sms ? 1 : 0;
  BwdArgs args = a;
  void* params[] = {&args, &G, &gpc, &search};
  cudaLaunchConfig_t cfg = {};
  const int cb = kFinalizeThreads / gpc;
  cfg.gridDim = dim3((unsigned)a.nseg, (unsigned)((2 * (a.D / 4) + cb - 1) / cb));
  cfg.blockDim = dim3(kFinalizeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // Programmatic dependent launch: the launch overlaps the row pass's tail;
  // the kernel itself waits for the row pass's results.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&adaln_bwd_finalize_kernel),
                             params);
}

}  // namespace adaln
