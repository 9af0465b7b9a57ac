// Host-side interface between the C ABI (api.cu) and the kernel launchers
// (fwd.cu, bwd.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/adaln.h"

#ifdef __CUDACC__
#define ADALN_HD __host__ __device__
#else
#define ADALN_HD
#endif

namespace adaln {

// Most rows handled per reduction round (sizes the reduction scratch).
constexpr int kRowsPerRound = 8;
// Largest number of consumer warps in a team (any variant).
constexpr int kMaxConsumerWarps = 8;
// Most teams in one CTA (each uses named barrier 1 + its index).
constexpr int kMaxTeams = 8;
// Ints of stage meta per ring stage: rows in the stage (-1: no work left),
// raw segment id of the row before it, first row (low, high 32 bits), then
// kRowsPerRound segment ids.
constexpr int kMetaInts = 4 + kRowsPerRound;
// Bytes before the teams' regions in a staging kernel's shared memory (the
// unit counter of the teams).
constexpr int kCtaHeaderBytes = 128;

// Compiled variants of the staging kernels, chosen by the row length in
// 16-byte vectors (nvec): vectors per thread (VPT), the largest consumer-warp
// count, and the teams per SM the register budget is sized for (one CTA per
// SM holds them).  At most 8 consumer warps share a row, so the per-row
// reduction work (shuffles, one shared-memory exchange, scalar statistics) is
// repeated by few warps; short rows use few warps per row and more teams, so
// that per-row overheads are shared by more elements.  The register cap
// follows from the warps per SM: 12 or 9 warps allow 168 registers a thread,
// 16 allow 128.
//   variant 5: nvec <=  192  VPT 2, <= 3 warps, 4 teams (forward)
//   variant 6: nvec <=  192  VPT 2, <= 3 warps, 3 teams (backward)
//   variant 1: nvec  =  384  VPT 2,    6 warps, 2 teams (forward)
//   variant 4: nvec <=  384  VPT 4, <= 3 warps, 3 teams (backward: its column
//              sums favour few warps per row, many rows per SM; forward below
//              384 vectors, where 2-warp teams fit four to an SM)
//   variant 2: nvec <=  640  VPT 4, <= 5 warps, 2 teams
//   variant 3: nvec <= 1024  VPT 4, <= 8 warps, 1 team
// A row that needs fewer warps than the variant's largest count runs more,
// smaller teams in the same thread budget (staging_shape).
ADALN_HD inline int choose_variant(int nvec) {
  return nvec <= 192 ? 5 : (nvec < 384 ? 4 : (nvec == 384 ? 1 : (nvec <= 640 ? 2 : 3)));
}
// The forward of 384 vectors (D = 3072 bf16, 1536 fp32) has two compiled
// shapes: variant 1 (two teams of 6 warps) and variant 4 (three teams of 3
// warps, 4 vectors a thread).  Variant 4 is faster when segments are long
// (T = 36864 in 16 segments, the MMDiT joint layer: 73.7 vs 77.8 us; every
// T from 8192 to 262144 with 2300 or more rows a segment: 2-15 % faster)
// and slower when they are short (about 640 rows: 6-8 % slower from
// T = 65536 on), so it takes the rows per segment into account.
ADALN_HD inline int choose_fwd_variant(int nvec, int64_t rows_per_segment) {
  return nvec == 384 && rows_per_segment >= 1024 ? 4 : choose_variant(nvec);
}
ADALN_HD inline int choose_bwd_variant(int nvec) {
  return nvec <= 192 ? 6 : (nvec <= 384 ? 4 : (nvec <= 640 ? 2 : 3));
}
ADALN_HD constexpr int variant_vpt(int v) { return (v == 1 || v == 5 || v == 6) ? 2 : 4; }
ADALN_HD constexpr int variant_max_warps(int v) {
  return v == 2 ? 5 : (v == 3 ? 8 : ((v == 4 || v == 5 || v == 6) ? 3 : 6));
}
ADALN_HD constexpr int variant_min_blocks(int v) {
  return v == 3 ? 1 : ((v == 4 || v == 6) ? 3 : (v == 5 ? 4 : 2));
}
ADALN_HD constexpr int variant_max_threads(int v) { return (variant_max_warps(v) + 1) * 32; }
// Rows per reduction round (and per ring stage).  The forward takes 4 in
// every variant: for short rows 8 made a round long and split a CTA's rows
// unevenly over its 4 teams (wan13b forward 20.9 vs 18.4 us).  The backward
// takes 4 for short rows, 2 otherwise (two tensors per stage).
ADALN_HD constexpr int fwd_rows(int v) { return (void)v, 4; }
ADALN_HD constexpr int bwd_rows(int v) { return v == 6 ? 4 : 2; }
// Consumer-warp counts with a compiled fixed-width instantiation per variant
// (forward and backward alike; variant 1 serves the forward only at 6): the
// variant's largest count and the counts of the common power-of-two widths
// (bf16 D = 512, 1024, 2048, 4096, 6144; fp32 half those).
ADALN_HD constexpr bool compiled_exact(int v, int nc) {
  return v == 5 || v == 6 ? (nc >= 1 && nc <= 3)
         : v == 1         ? nc == 6
         : v == 4         ? (nc == 2 || nc == 3)
         : v == 2         ? (nc == 4 || nc == 5)
                          : (nc == 6 || nc == 8);
}
// The fixed-width instantiation for a row of nvec vectors: its consumer-warp
// count when the row fills that many warps exactly and it is compiled, else
// 0 (the generic instantiation, warp count and row length at run time).
ADALN_HD inline int exact_warps(int v, int nvec) {
  const int per_warp = 32 * variant_vpt(v);
  const int nc = nvec / per_warp;
  return nc * per_warp == nvec && compiled_exact(v, nc) ? nc : 0;
}

struct Shape {
  int variant;    // compiled variant (choose_variant)
  int ncx;        // fixed-width instantiation's warp count (exact_warps), or 0
  int vpt;        // 16-byte vectors per thread per row (1, 2 or 4)
  int nc;         // consumer warps of a team
  int teams;      // teams per CTA (a team: nc consumer warps + a producer warp)
  int threads;    // teams * (nc + 1) * 32
  int team_bytes; // shared memory of one team (header + ring, 128-byte multiple)
  int stages;     // depth of the shared-memory ring
  int smem;       // dynamic shared memory bytes
  int grid;       // persistent CTAs
  int sms;        // SMs of the device
  int nvec;       // 16-byte vectors per row
  int row_bytes;  // bytes of one row of x
};

struct FwdArgs {
  const void* x;
  const void* shift;
  const void* scale;
  const int32_t* seg;
  void* y;
  float* mean;
  float* rstd;
  int64_t T;
  int32_t D;
  int32_t nseg;
  float eps;
  float inv_d;  // 1 / D rounded to fp32
  unsigned* status;
  // Device-wide unit counter {next unit, producers done} of this launch, or
  // nullptr: the teams then share their CTA's contiguous row range only.
  int* ticket;
  // With a ticket: 0 = all rows in device-wide units; > 0 = the CTAs share
  // the first T - tail_rows rows in contiguous ranges and the last tail_rows
  // go device-wide.
  int64_t tail_rows;
};

struct BwdArgs {
  const void* dy;
  const void* x;
  const float* mean;
  const float* rstd;
  const void* scale;
  const int32_t* seg;
  void* dx;
  float* dshift;
  float* dscale;
  float* partials;  // [G + nseg - 1][2][D] fp32: (dscale, dshift) partials
  int32_t* seg_start;  // [nseg + 1]: first row of each segment (T at the end)
  int64_t T;
  int32_t D;
  int32_t nseg;
  float inv_d;  // 1 / D rounded to fp32
  unsigned* status;
  int accumulate;  // finalize adds its sums to dshift/dscale (row-chunked calls)
};

// Launch shapes (depend on the current device).  Return cudaSuccess or the
// error of the device query.
cudaError_t fwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, int variant, Shape* s);
cudaError_t bwd_shape(int64_t T, int32_t D, adaln_dtype_t dt, Shape* s);

// Number of fp32 partial slots of the backward: G + nseg - 1.
// Row ranges of the staging kernels are owned by teams: team k of CTA c is
// virtual CTA c * teams + k of grid * teams.
inline int64_t virtual_ctas(const Shape& s) { return (int64_t)s.grid * s.teams; }
inline int64_t bwd_slots(const Shape& s, int32_t nseg) {
  return virtual_ctas(s) + nseg - 1;
}

// Backward workspace: the partial slots, then the segment start table.
inline size_t bwd_partials_bytes(const Shape& s, int32_t D, int32_t nseg) {
  return (size_t)bwd_slots(s, nseg) * 2 * (size_t)D * sizeof(float);
}
inline size_t bwd_workspace_bytes(const Shape& s, int32_t D, int32_t nseg) {
  return bwd_partials_bytes(s, D, nseg) + ((size_t)nseg + 1) * sizeof(int32_t);
}

// Launch a row kernel of shape s as a programmatic dependent of the previous
// kernel on st (the kernel waits, griddepcontrol.wait, before reading global
// memory).
inline cudaError_t launch_dependent(void* kernel, const Shape& s, void** params,
                                    cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s.grid);
  cfg.blockDim = dim3((unsigned)s.threads);
  cfg.dynamicSmemBytes = (size_t)s.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, params);
}

cudaError_t launch_fwd(const FwdArgs& a, adaln_dtype_t dt, const Shape& s,
                       cudaStream_t st);
cudaError_t launch_bwd_rows(const BwdArgs& a, adaln_dtype_t dt,
                            const Shape& s, cudaStream_t st);
cudaError_t launch_bwd_finalize(const BwdArgs& a, const Shape& s,
                                cudaStream_t st);

// Launch parts of the C entry points (api.cu), without argument checks; the
// backward can add its sums into dshift/dscale (accumulate = 1) for callers
// that process the rows in chunks, and the forward takes the rows per
// segment of the whole batch (seg_rows: its variant choice, so that a chunk
// computes what the whole call would).
int run_fwd(const void* x, const void* shift, const void* scale, const int32_t* seg_id,
            int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype, float eps, void* y,
            float* mean, float* rstd, cudaStream_t st, int64_t seg_rows);
int run_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
            const void* scale, const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
            adaln_dtype_t dtype, void* dx, float* dshift, float* dscale, void* workspace,
            size_t workspace_bytes, cudaStream_t st, int accumulate);
size_t bwd_workspace_need(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype, int* rc);
int check_dims_public(int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dt);

// Launch slots (api.cu).  A launch that needs device-wide state of its own
// (the forward's unit counters) takes one of kLaunchSlots slots of a pool and
// indexes a static device array with it.  A slot is handed out only when the
// launch that used it before has completed (a CUDA event per slot), so no two
// launches in flight share one; launches being captured into a CUDA graph get
// none (a graph may be replayed while other work runs).
constexpr int kLaunchSlots = 256;
enum { kPoolFwdUnits = 0, kNumSlotPools = 1 };
// A slot index, or -1 when none is free (or the stream is capturing).
int launch_slot_acquire(int pool, cudaStream_t st);
// After the launch: the slot stays busy until the work queued on `st` ends.
cudaError_t launch_slot_release(int pool, int slot, cudaStream_t st, bool launched);

// Bounded-wait self-test (selftest.cu).
cudaError_t launch_wait_timeout_probe(unsigned* status, uint64_t limit_ns, cudaStream_t st);

// Shared-memory header of the staging kernels (barriers, flags, reduction
// scratch), before the 128-byte aligned ring.
ADALN_HD inline int ring_header_bytes(int stages) {
  int b = 16 * stages            // full[] and empty[] mbarriers
          + 16                   // abort flag (+ pad)
          + 2 * kMaxConsumerWarps * kRowsPerRound * 2 * 4  // reduction values
          + 2 * kMaxConsumerWarps * 4                      // ok flags
          + stages * kMetaInts * 4;                        // stage meta
  return (b + 127) & ~127;
}

}  // namespace adaln
