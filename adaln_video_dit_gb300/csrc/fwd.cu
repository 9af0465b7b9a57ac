// Fused AdaLN forward: y = (x - mean) * rstd * (1 + scale[b]) + shift[b].
//
// AdaptiveLoad, Technical summary section 2.B, forward pass: statistics are
// reduced on chip in two stages (warp shuffles, then across warps) and the
// modulation is applied in the same launch, so x is read from HBM once and y
// written once.  Here persistent teams (consumer warps + a producer warp,
// one to four per CTA, one CTA per SM) claim units of R rows and stream them
// through their shared-memory rings (bulk async copies issued by one producer
// lane); for each round of R rows the consumer threads read their column
// slice from the stage three times (row sums -> mean; centred sum of squares
// -> rstd, the two-pass definition of the biased variance; modulate) and
// write y with 16-byte streaming stores, keeping only the segment's
// (1 + scale) and shift in registers.  Element arithmetic uses packed fp32x2
// instructions.
#include <cstdlib>
#include <mutex>

#include "ring.cuh"

namespace adaln {

// One CTA per SM holds `teams` teams (consumer warps + a producer warp, each
// with its own ring); teams claim units of R rows.  With a device-wide
// counter (a.ticket) all teams share all rows, so SMs that stream faster take
// more rows (SMs differ by up to a fifth in throughput); without one the
// CTAs split the rows into contiguous ranges and the teams of a CTA share
// its range through a shared-memory counter (then a segment's modulation
// rows are loaded once per team, not once per unit: the mode for many short
// segments, and for launches captured into CUDA graphs).  In between, the
// CTAs share the first rows in contiguous ranges and all teams share a
// device-wide tail (a.tail_rows).  Every row's result is independent of
// which team computes it.
// NCX: 0 for the generic instantiation (warp count and row length at run
// time), else a consumer-warp count the row fills exactly (nvec = NCX x 32 x
// VPT; the counts compiled_exact lists), which makes both compile-time
// constants (offsets fold into immediates, no per-vector guards).
template <class E, int VARIANT, int R, int NCX>
__global__ void __launch_bounds__(variant_min_blocks(VARIANT) * variant_max_threads(VARIANT), 1)
    adaln_fwd_kernel(FwdArgs a, int nc_rt, int stages, int nvec_rt, int team_bytes) {
  constexpr int VPT = variant_vpt(VARIANT);
  constexpr bool EXACT = NCX != 0;
  const int nc = EXACT ? NCX : nc_rt;
  const int nvec = EXACT ? NCX * 32 * VPT : nvec_rt;
  constexpr int H = E::EPV / 2;  // float2 pairs per vector
  extern __shared__ __align__(128) unsigned char smem[];
  const int team_threads = (nc + 1) * 32;
  const int team = threadIdx.x / team_threads;
  const int lt = threadIdx.x - team * team_threads;  // thread index in the team
  int* next_unit = reinterpret_cast<int*>(smem);
  const Ring rg = ring_layout(smem + kCtaHeaderBytes + team * team_bytes, stages, 1 + team,
                              team * (nc + 1));
  if (lt == 0) ring_init_team(rg, nc);
  if (threadIdx.x == 0) *next_unit = 0;
  __syncthreads();
  // Launched as a programmatic dependent of the stream's previous kernel: the
  // set-up above may overlap that kernel's end, nothing in global memory is
  // read before it has completed.  The next kernel may then be scheduled as
  // SMs free up (this library's kernels wait the same way before reading).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int64_t G = gridDim.x;
  const int64_t r0 = part_begin(blockIdx.x, a.T, G);
  const int64_t nrows = part_begin(blockIdx.x + 1, a.T, G) - r0;
  const int row_bytes = nvec * 16;
  const int warp = lt >> 5;

  if (warp == nc) {  // producer warp
    if ((lt & 31) == 0) {
      const unsigned char* src[1] = {static_cast<const unsigned char*>(a.x)};
      if (a.ticket != nullptr) {
        if (a.tail_rows > 0) {
          // The CTA's share of the first T - tail rows through the CTA's
          // counter, then the last tail rows device-wide.
          const int64_t TL = a.T - a.tail_rows;
          const int64_t l0 = part_begin(blockIdx.x, TL, G);
          ring_produce_units<R, 1>(rg, src, l0, part_begin(blockIdx.x + 1, TL, G) - l0,
                                   next_unit, TL, a.tail_rows, a.ticket, R, row_bytes, a.seg,
                                   a.status);
        } else {
          // All rows, units claimed device-wide.
          ring_produce_units<R, 1>(rg, src, 0, 0, nullptr, 0, a.T, a.ticket, R, row_bytes,
                                   a.seg, a.status);
        }
        // The last producer to finish (every claim of every producer is done
        // by then) zeroes the counter pair for the next launch given it.
        __threadfence();
        const int producers = (int)gridDim.x * (int)(blockDim.x / team_threads);
        if (atomicAdd(a.ticket + 1, 1) == producers - 1) {
          a.ticket[0] = 0;
          __threadfence();
          a.ticket[1] = 0;
        }
      } else {
        ring_produce_units<R, 1>(rg, src, r0, nrows, next_unit, 0, 0, nullptr, R, row_bytes,
                                 a.seg, a.status);
      }
    }
    return;
  }

  const int j = lt;
  const int NT = nc * 32;
  const uint32_t ring0 = smem_addr(rg.ring);
  const uint32_t stage_bytes = (uint32_t)R * row_bytes;
  bool valid[VPT];
#pragma unroll
  for (int q = 0; q < VPT; ++q) valid[q] = EXACT || j + q * NT < nvec;

  // (1 + scale) and shift of the current segment for this thread's columns.
  float2 s1[VPT][H], sh[VPT][H];
  int cur_b = -1;
  int phase = 0;

  // Every thread's vectors are all in the row when nvec is a multiple of the
  // consumer thread count times VPT (true for D = 1536, 3072, 5120 bf16).
  const bool all_valid = EXACT || nvec == NT * VPT;

  int s = 0;          // ring stage of this round (advanced by increment)
  uint32_t par = 0;   // parity of this use of the stage
  for (;; s = (s + 1 == stages ? 0 : s + 1), par ^= (s == 0 ? 1u : 0u)) {
    // The stage's data and meta (unit, segment ids) arrive together.
    const bool ok = mbar_wait_bounded(rg.full(s), par, rg.abort);
    const int* m = rg.meta + s * kMetaInts;
    const int mrows = ok ? m[0] : 0;
    const bool end = ok && mrows < 0;  // no work left (the same for every warp)
    const int rows = mrows > 0 ? mrows : 0;
    const int64_t t0 = rows > 0 ? (int64_t)(uint32_t)m[2] | ((int64_t)m[3] << 32) : 0;
    int sg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sg[r] = r < rows ? m[4 + r] : 0;
    int prev_b = 0;
    if (rows > 0 && m[1] >= 0) prev_b = m[1] >= a.nseg ? a.nseg - 1 : m[1];

    // x stays in the stage until the outputs are written: each pass reads
    // its rows from shared memory (registers hold only column state).
    const uint32_t st0 = ring0 + s * stage_bytes;

    // One round over the unit's rows: 0 = done, 1 = no unit left, 2 = abort.
    // FULL (all R rows present, every vector of this thread in the row,
    // pipeline ok) drops the per-row and per-vector guards, so the rows' work
    // interleaves freely.  The last round (rows = 0) still takes part in the
    // first team reduction, so that all warps leave the loop together.
    auto round = [&](auto full_tag) -> int {
      constexpr bool FULL = decltype(full_tag)::value;
      // Pass 1: row sums -> mean.
      float acc[R][1];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float2 t[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if (FULL || r < rows) {
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
      if (!team_sum<R, 1>(acc, ok, rg, nc, phase)) return 2;
      phase ^= 1;
      if (end) return 1;
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

      // Segment bookkeeping for the unit's rows, then the modulated outputs.
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
      return 0;
    };
    const bool full = ok && rows == R && all_valid;
    const int rc = full ? round(Tag<true>()) : round(Tag<false>());
    if (rc == 1) break;
    if (rc == 2) {
      if (j == 0) {
        atomicOr(a.status, ADALN_DEV_TIMEOUT);
        *rg.abort = 1;
      }
      break;
    }
    __syncwarp();
    if ((lt & 31) == 0) mbar_arrive(rg.empty(s));
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {

template <class E, int V, int NCX>
void* fwd_inst() {
  return reinterpret_cast<void*>(&adaln_fwd_kernel<E, V, fwd_rows(V), NCX>);
}

// The instantiation for (variant, fixed warp count or 0); compiled_exact lists
// the fixed counts.
template <class E>
void* fwd_kernel_for(int variant, int ncx) {
  switch (variant) {
    case 5: return ncx == 1 ? fwd_inst<E, 5, 1>() : ncx == 2 ? fwd_inst<E, 5, 2>()
                 : ncx == 3 ? fwd_inst<E, 5, 3>() : fwd_inst<E, 5, 0>();
    case 1: return fwd_inst<E, 1, 6>();
    case 4: return ncx == 2 ? fwd_inst<E, 4, 2>() : ncx == 3 ? fwd_inst<E, 4, 3>()
                 : fwd_inst<E, 4, 0>();
    case 2: return ncx == 4 ? fwd_inst<E, 2, 4>() : ncx == 5 ? fwd_inst<E, 2, 5>()
                 : fwd_inst<E, 2, 0>();
    default: return ncx == 6 ? fwd_inst<E, 3, 6>() : ncx == 8 ? fwd_inst<E, 3, 8>()
                  : fwd_inst<E, 3, 0>();
  }
}

void* pick_fwd(adaln_dtype_t dt, int variant, int ncx) {
  return dt == ADALN_BF16 ? fwd_kernel_for<BF16>(variant, ncx) : fwd_kernel_for<F32>(variant, ncx);
}

}  // namespace

// Common shape rule of the staging kernels: the compiled variant for the row
// length, consumer warps to cover the row, `teams` teams per CTA (the
// variant's count, or more when smaller teams fit its thread budget) after a
// `cta_header`-byte CTA header, ring depth sized for about 160 KB of staged
// rows per SM over those teams, and persistent CTAs = SMs x resident CTAs per
// SM (at most T).
cudaError_t staging_shape(void* kernel, int64_t T, int32_t D, adaln_dtype_t dt,
                          int ntensors, int rows_per_round, int variant, int teams,
                          int cta_header, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  s->row_bytes = D * esize;
  s->nvec = s->row_bytes / 16;
  s->variant = variant;
  s->ncx = exact_warps(variant, s->nvec);
  s->vpt = variant_vpt(s->variant);
  s->nc = (s->nvec + 32 * s->vpt - 1) / (32 * s->vpt);
  // The kernel is compiled for `teams` teams of the variant's largest warp
  // count; rows that need fewer consumer warps run more teams in the same
  // thread (and register) budget, up to kMaxTeams, so that an SM keeps about
  // as many warps, and rows, in flight.
  const int fit = teams * variant_max_threads(variant) / ((s->nc + 1) * 32);
  if (fit > teams) teams = fit < kMaxTeams ? fit : kMaxTeams;
  s->teams = teams;
  s->threads = teams * (s->nc + 1) * 32;

  int dev = 0, sms = 0, optin = 0, smem_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;

  // Ring depth: about 160 KB of staged rows per SM, split over the teams,
  // and no more than fits beside them.
  const int units = teams;  // teams per SM (one CTA per SM)
  const int ctas = 1;
  const int stage_bytes = rows_per_round * s->row_bytes * ntensors;
  const int per_cta = smem_sm / ctas - 2048;  // room for the per-CTA reserve
  const int per_team = (per_cta - cta_header) / teams;
  int ring_kb = 160;
#ifdef ADALN_TUNING
  // Tuning builds only (build.py --tuning): launch-shape sweeps.  The
  // release library reads no environment variable.
  if (const char* env = getenv("ADALN_RING_KB")) {
    const int v = atoi(env);
    if (v >= 16 && v <= 256) ring_kb = v;
  }
#endif
  int budget = ring_kb * 1024 / units;
  if (budget > per_team) budget = per_team;
  int stages = budget / stage_bytes;
  stages = stages < 2 ? 2 : (stages > 16 ? 16 : stages);
  auto team_bytes = [&](int st) {
    return (ring_header_bytes(st) + st * stage_bytes + 127) & ~127;
  };
  while (stages > 2 && team_bytes(stages) > per_team) --stages;
  s->stages = stages;
  s->team_bytes = team_bytes(stages);
  s->smem = cta_header + teams * s->team_bytes;
  if (s->smem > optin) return cudaErrorInvalidValue;

  // Allow the device maximum: other D values reuse this template instance
  // with larger rings.
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, s->threads, s->smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
#ifdef ADALN_TUNING
  // Tuning builds only: fewer resident CTAs per SM (launch-shape sweeps).
  if (const char* env = getenv("ADALN_CTAS_PER_SM")) {
    const int v = atoi(env);
    if (v >= 1 && v < per_sm) per_sm = v;
  }
#endif
  int64_t g = (int64_t)sms * per_sm;
  if (g > T) g = T;
  s->grid = (int)(g < 1 ? 1 : g);
  s->sms = sms;
  return cudaSuccess;
}

cudaError_t fwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, int v, Shape* s) {
  const int esize = dt == ADALN_BF16 ? 2 : 4;
  const int nvec = D * esize / 16;
  return staging_shape(pick_fwd(dt, v, exact_warps(v, nvec)), T, D, dt, 1, fwd_rows(v), v,
                       variant_min_blocks(v), kCtaHeaderBytes, s);
}

// Device-wide unit counters {next unit, producers done}, one per launch slot
// (internal.h): zero at module load; the last producer of a launch zeroes its
// counters again, and a slot is handed to a launch only when the launch that
// used it before has completed.
__device__ int g_fwd_tickets[kLaunchSlots][2];

namespace {

// Device address of g_fwd_tickets on the current device (looked up once per
// device), or nullptr.
int* fwd_tickets_base() {
  constexpr int kDevices = 64;
  static std::mutex mu;
  static int* base[kDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!base[dev]) {
    void* b = nullptr;
    if (cudaGetSymbolAddress(&b, g_fwd_tickets) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    base[dev] = static_cast<int*>(b);
  }
  return base[dev];
}

// How the forward's teams get their rows.  Device-wide units balance the
// SMs' unequal speeds but make a team's consecutive units often change
// segment, which reloads the segment's modulation rows: all rows go
// device-wide when segments are at least 4 rounds of all teams long.
// Otherwise each CTA's teams share the CTA's contiguous range, and, when
// there are at least 10 rounds of rows and segments of at least one round,
// the last tenth of the rows is shared device-wide, so that teams on faster
// SMs take the tail (a reload at each of those few units): mmdit_joint's
// forward 80.2 vs 78.0 us; with fewer rows the tail is too large a share
// (wan13b +0.5 us), with shorter segments the reloads cost more than the
// balance gains (mixed_varlen +0.2 %).  Returns the rows of that device-wide
// tail, 0 for all rows device-wide, -1 for CTA ranges only.
int64_t device_rows_plan(const FwdArgs& a, const Shape& s, int R) {
  const int64_t round_rows = (int64_t)s.grid * s.teams * R;
  int mode = 0;
  if (a.T >= 2 * round_rows && a.T / a.nseg >= 4 * round_rows) mode = 1;
  else if (a.T >= 10 * round_rows && a.T / a.nseg >= round_rows) mode = 2;
#ifdef ADALN_TUNING
  // Tuning builds only: ADALN_FWD_SCHED = "cta", "device" or "hybrid".
  if (const char* env = getenv("ADALN_FWD_SCHED")) {
    if (env[0] == 'c') mode = 0;
    if (env[0] == 'd') mode = 1;
    if (env[0] == 'h') mode = 2;
  }
#endif
  if (mode == 0 || a.T < 2 * round_rows) return -1;
  if (mode == 1) return 0;
  int64_t tail = a.T / 10 / R * R;
  if (tail < round_rows) tail = round_rows;
  return tail < a.T / 2 ? tail : -1;
}}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, adaln_dtype_t dt, const Shape& s,
                       cudaStream_t st) {
  void* k = pick_fwd(dt, s.variant, s.ncx);
  int nc = s.nc, stages = s.stages, nvec = s.nvec, team_bytes = s.team_bytes;
  FwdArgs args = a;
  args.ticket = nullptr;
  args.tail_rows = 0;
  int slot = -1;
  const int64_t plan = device_rows_plan(a, s, fwd_rows(s.variant));
  if (plan >= 0) {
    int* base = fwd_tickets_base();
    if (base) slot = launch_slot_acquire(kPoolFwdUnits, st);
    if (slot >= 0) {
      args.ticket = base + 2 * slot;
      args.tail_rows = plan;
    }
  }
  void* params[] = {&args, &nc, &stages, &nvec, &team_bytes};
  const cudaError_t e = launch_dependent(k, s, params, st);
  if (slot >= 0) {
    const cudaError_t r = launch_slot_release(kPoolFwdUnits, slot, st, e == cudaSuccess);
    if (e == cudaSuccess && r != cudaSuccess) return r;
  }
  return e;
}

}  // namespace adaln
