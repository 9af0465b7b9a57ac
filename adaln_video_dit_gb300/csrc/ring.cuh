// Shared-memory staging ring used by the forward and backward row kernels.
//
// A team = nc consumer warps + 1 producer warp, with its own ring; a CTA
// holds one team (backward) or several that share the CTA's rows (forward,
// ring_produce_units).  The producer (one lane) of a team
// streams chunks of R consecutive rows from global memory into S ring stages
// with bulk asynchronous copies, each completing on the stage's "full"
// mbarrier; consumer warps read the rows from shared memory as often as
// their passes need and release the stage on its "empty" mbarrier when they
// are done with it.  Consumer thread j owns the
// 16-byte column vectors j, j + 32 nc, ... of every row, so column state
// (modulation vectors, gradient accumulators) stays in its registers for the
// whole row range, and row sums are finished with a warp butterfly plus one
// exchange through shared memory per round of R rows.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace adaln {

struct Ring {
  uint32_t base;   // shared address of this team's header
  int stages;
  int bar_id;      // named barrier of the team's consumer warps
  int warp0;       // CTA warp index of the team's first warp
  volatile int* abort;
  float* red;      // [2][kMaxConsumerWarps][R][2]
  int* okf;        // [2][kMaxConsumerWarps]
  int* meta;       // [stages][kMetaInts]: unit, segment before it, its segments
  unsigned char* ring;

  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (stages + s); }
};

// Layout of one team's region (header, then the 128-byte aligned stages).
__device__ __forceinline__ Ring ring_layout(unsigned char* smem, int stages, int bar_id = 1,
                                            int warp0 = 0) {
  Ring r;
  r.base = smem_addr(smem);
  r.stages = stages;
  r.bar_id = bar_id;
  r.warp0 = warp0;
  unsigned char* p = smem + 16 * stages;
  r.abort = reinterpret_cast<volatile int*>(p);
  p += 16;
  r.red = reinterpret_cast<float*>(p);
  p += 2 * kMaxConsumerWarps * kRowsPerRound * 2 * 4;
  r.okf = reinterpret_cast<int*>(p);
  p += 2 * kMaxConsumerWarps * 4;
  r.meta = reinterpret_cast<int*>(p);
  r.ring = smem + ring_header_bytes(stages);
  return r;
}

// One thread initialises a team's barriers and abort flag (no CTA sync: the
// caller follows with __syncthreads before the role split).
__device__ __forceinline__ void ring_init_team(const Ring& rg, int nc) {
  for (int s = 0; s < rg.stages; ++s) {
    mbar_init(rg.full(s), 1);
    mbar_init(rg.empty(s), nc);
  }
  *rg.abort = 0;
  mbar_init_fence();
}

// Thread 0 initialises the barriers; everyone syncs.  Must run before the
// role split (it uses __syncthreads).
__device__ __forceinline__ void ring_init(const Ring& rg, int nc) {
  if (threadIdx.x == 0) ring_init_team(rg, nc);
  __syncthreads();
}

// Producer loop (one lane).  Streams `nchunks` chunks of up to R rows of each
// of NT tensors (src[i] + row offset) into the ring.  Before returning it
// waits for the last copy issued into every stage, so that no copy into this
// CTA's shared memory is still in flight when the CTA exits.
template <int R, int NT>
__device__ __forceinline__ void ring_produce(const Ring& rg,
                                             const unsigned char* const (&src)[NT],
                                             int64_t nrows, int row_bytes,
                                             unsigned* status) {
  const uint64_t policy = l2_evict_first_policy();
  const int64_t nchunks = (nrows + R - 1) / R;
  const int S = rg.stages;
  const uint32_t stage_bytes = (uint32_t)R * row_bytes * NT;
  int64_t issued = 0;
  int s = 0;        // stage of chunk k (k % S, advanced by increment)
  uint32_t it = 0;  // use of that stage (k / S), for the "empty" parity
  for (int64_t k = 0; k < nchunks; ++k, it += (s + 1 == S), s = (s + 1 == S ? 0 : s + 1)) {
    if (it > 0 && !mbar_wait_bounded(rg.empty(s), (it - 1) & 1, rg.abort)) {
      if (!*rg.abort) atomicOr(status, ADALN_DEV_TIMEOUT);
      *rg.abort = 1;
      break;
    }
    if (*rg.abort) break;
    const int rows = (int)min((int64_t)R, nrows - k * R);
    const uint32_t bytes = (uint32_t)rows * row_bytes;
    mbar_arrive_expect_tx(rg.full(s), bytes * NT);
    const uint32_t dst = smem_addr(rg.ring) + (uint32_t)s * stage_bytes;
#pragma unroll
    for (int i = 0; i < NT; ++i)
      bulk_g2s(dst + (uint32_t)i * R * row_bytes,
               src[i] + (size_t)k * R * row_bytes, bytes, rg.full(s), policy);
    issued = k + 1;
    if (k == 0) {
      // Every team issues its whole ring at once at the start; let the first
      // stage's copies go ahead of the next ones, so that the first round can
      // start early: wait, briefly and bounded, for them to land.
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(rg.full(0), 0) && globaltimer_ns() - t0 < kFirstStageHeadNs) {
      }
    }
  }
  // Drain: the newest chunk of each stage is the only one possibly in flight.
  for (int s = 0; s < S; ++s) {
    if (issued <= s) break;
    const int64_t last = s + ((issued - 1 - s) / S) * S;
    if (!mbar_wait_bounded(rg.full(s), (uint32_t)((last / S) & 1), nullptr))
      atomicOr(status, ADALN_DEV_TIMEOUT);
  }
}

// Producer loop of a team that claims its work (one lane).  Work comes from
// up to two sources, taken in order: rows [l0, l0 + nl) cut into units of U
// rows (a multiple of R) claimed from the counter *lctr, then rows
// [g0, g0 + ng) in units claimed from *gctr (a null counter: no such
// source).  A counter in shared memory lets the teams of one CTA share the
// CTA's rows; one in global memory lets all teams share the rows, so a team
// that runs faster takes more and all finish together.  The next unit is
// claimed while the current one streams, hiding the counter's latency.  A
// unit goes through the ring in stages of up to R rows; each stage's meta
// (rows, raw segment id of the row before it or -1, first row, segment ids of
// its rows) is written before the producer's arrival on the stage's "full"
// barrier, which releases it with the data.  When no unit is left the stage
// gets rows = -1 and no data.  `src` holds the tensors' base addresses (rows
// are absolute).  Before returning it waits for the newest copy into every
// stage, so that no copy into this CTA's shared memory is still in flight
// when the CTA exits.
template <int R, int NT>
__device__ __forceinline__ void ring_produce_units(const Ring& rg,
                                                   const unsigned char* const (&src)[NT],
                                                   int64_t l0, int64_t nl, int* lctr,
                                                   int64_t g0, int64_t ng, int* gctr, int U,
                                                   int row_bytes, const int32_t* seg,
                                                   unsigned* status) {
  const uint64_t policy = l2_evict_first_policy();
  const int S = rg.stages;
  const uint32_t stage_bytes = (uint32_t)R * row_bytes * NT;
  int64_t issued = 0;
  int source = lctr != nullptr ? 0 : 1;  // 0: first source, 1: second, 2: none left
  // Claim the next unit: its rows [*a, *b), or false when both sources are done.
  auto claim = [&](int64_t* a, int64_t* b) -> bool {
    if (source == 0) {
      const int64_t u = atomicAdd(lctr, 1);
      if (u * U < nl) {
        *a = l0 + u * U;
        *b = min(*a + U, l0 + nl);
        return true;
      }
      source = 1;
    }
    if (source == 1 && gctr != nullptr) {
      const int64_t u = atomicAdd(gctr, 1);
      if (u * U < ng) {
        *a = g0 + u * U;
        *b = min(*a + U, g0 + ng);
        return true;
      }
    }
    source = 2;
    return false;
  };
  int64_t cur = 0, cur_end = 0;  // rows of the current unit not yet staged
  int64_t na = 0, nb = 0;        // the unit claimed ahead
  bool ahead = claim(&na, &nb);
  int s = 0;        // stage of claim k (k % S, advanced by increment)
  uint32_t it = 0;  // use of that stage (k / S), for the "empty" parity
  for (int64_t k = 0;; ++k, it += (s + 1 == S), s = (s + 1 == S ? 0 : s + 1)) {
    if (it > 0 && !mbar_wait_bounded(rg.empty(s), (it - 1) & 1, rg.abort)) {
      if (!*rg.abort) atomicOr(status, ADALN_DEV_TIMEOUT);
      *rg.abort = 1;
      break;
    }
    if (*rg.abort) break;
    int* m = rg.meta + s * kMetaInts;
    if (cur == cur_end) {
      if (!ahead) {
        m[0] = -1;
        mbar_arrive(rg.full(s));
        issued = k + 1;
        break;
      }
      cur = na;
      cur_end = nb;
      ahead = claim(&na, &nb);
    }
    const int rows = (int)min((int64_t)R, cur_end - cur);
    const uint32_t bytes = (uint32_t)rows * row_bytes;
    mbar_expect_tx(rg.full(s), bytes * NT);
    const uint32_t dst = smem_addr(rg.ring) + (uint32_t)s * stage_bytes;
#pragma unroll
    for (int i = 0; i < NT; ++i)
      bulk_g2s(dst + (uint32_t)i * R * row_bytes, src[i] + (size_t)cur * row_bytes, bytes,
               rg.full(s), policy);
    // Segment ids load while the copies are in flight.
    const int64_t t = cur;
    int sg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sg[r] = r < rows ? __ldg(seg + t + r) : 0;
    m[1] = t > 0 ? __ldg(seg + t - 1) : -1;
    m[2] = (int)(t & 0xffffffff);
    m[3] = (int)(t >> 32);
#pragma unroll
    for (int r = 0; r < R; ++r) m[4 + r] = sg[r];
    m[0] = rows;
    mbar_arrive(rg.full(s));
    cur += rows;
    issued = k + 1;
  }
  for (int s = 0; s < S; ++s) {
    if (issued <= s) break;
    const int64_t last = s + ((issued - 1 - s) / S) * S;
    if (!mbar_wait_bounded(rg.full(s), (uint32_t)((last / S) & 1), nullptr))
      atomicOr(status, ADALN_DEV_TIMEOUT);
  }
}

// Sum K values per row over the consumer team, for R rows at once.  Every
// consumer thread gets bitwise identical sums (butterflies of commutative
// adds, fixed shape).  `ok` is this thread's pipeline status; the returned
// flag is true only if every consumer warp was ok, so all consumers take the
// same branch after the exchange.  `phase` alternates the shared buffers.
template <int R, int K>
__device__ __forceinline__ bool team_sum(float (&v)[R][K], bool ok,
                                         const Ring& rg, int nc, int phase) {
  static_assert(R <= kRowsPerRound && K <= 2, "reduction buffer too small");
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - rg.warp0;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int q = 0; q < K; ++q) {
      float a = v[r][q];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      v[r][q] = a;
    }
  const bool warp_ok = __all_sync(0xffffffffu, ok);
  float* red = rg.red + phase * (kMaxConsumerWarps * kRowsPerRound * 2);
  int* okf = rg.okf + phase * kMaxConsumerWarps;
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int q = 0; q < K; ++q) red[(w * kRowsPerRound + r) * 2 + q] = v[r][q];
    okf[w] = warp_ok ? 1 : 0;
  }
  named_barrier_sync(rg.bar_id, nc * 32);
  // nc <= 8: every group of 8 lanes reduces the nc warp sums (the same
  // values in the same order), so all lanes end with identical bits.
  const int src = lane & 7;
  const bool mine = src < nc;
  bool all_ok = __all_sync(0xffffffffu, mine ? okf[src] != 0 : true);
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int q = 0; q < K; ++q) {
      float a = mine ? red[(src * kRowsPerRound + r) * 2 + q] : 0.0f;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      v[r][q] = a;
    }
  return all_ok;
}

// Read a row's segment id, clamp it into [0, nseg) and record range / order
// violations (lane 0 of each warp reports; errors only, so the extra atomics
// cost nothing on valid input).
__device__ __forceinline__ int checked_seg(int raw, int prev, int nseg,
                                           unsigned* status) {
  int b = raw;
  unsigned bad = 0;
  if (b < 0 || b >= nseg) {
    bad |= ADALN_DEV_SEG_RANGE;
    b = b < 0 ? 0 : nseg - 1;
  }
  if (b < prev) bad |= ADALN_DEV_SEG_ORDER;
  if (bad && (threadIdx.x & 31) == 0) atomicOr(status, bad);
  return b;
}

}  // namespace adaln
