// Device-side building blocks shared by the forward and backward kernels:
// element traits for 16-byte vectors, mbarrier / bulk-copy PTX wrappers for
// the shared-memory staging ring, bounded waits, and the launch-shape rules.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/adaln.h"

namespace adaln {

// ---------------------------------------------------------------------------
// Element traits.  A "vector" is 16 bytes: 8 bf16 or 4 fp32 values.
// ---------------------------------------------------------------------------
struct BF16 {
  static constexpr int EPV = 8;  // elements per 16-byte vector
  static constexpr int SIZE = 2;
  // Exact widening: a bf16 value is the upper half of an fp32 bit pattern.
  // Element 2i is the low half of word i.
  __device__ static __forceinline__ void unpack2(const uint4& v, float2 (&f)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  // Round to nearest even, once.
  __device__ static __forceinline__ uint4 pack2(const float2 (&f)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[i].x, f[i].y);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

struct F32 {
  static constexpr int EPV = 4;
  static constexpr int SIZE = 4;
  __device__ static __forceinline__ void unpack2(const uint4& v, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ static __forceinline__ uint4 pack2(const float2 (&f)[2]) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                      __float_as_uint(f[1].x), __float_as_uint(f[1].y));
  }
};

// Compile-time flag carried into generic lambdas.
template <bool B>
struct Tag {
  static constexpr bool value = B;
};

// Packed fp32x2 arithmetic (one instruction per pair on sm_100 and later).
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ---------------------------------------------------------------------------
// Plain memory helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Streaming 16-byte global store (written once, not re-read by this kernel).
__device__ __forceinline__ void st_global_cs_v4(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier and bulk asynchronous copy (global -> shared).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the other threads and to the async
// (bulk-copy) proxy before first use.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Announce `bytes` more transaction bytes for the current phase, without
// arriving (the arrival follows separately).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Upper bound on any single wait of a staging pipeline.  Legitimate waits
// last microseconds; the bound only turns an internal error into a status
// bit and an orderly exit instead of a hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// As mbar_try_wait, but the thread may be suspended (instead of spinning)
// until the phase completes or about `hint_ns` nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Longest wait of a producer for its first stage's copies to land before it
// issues the next stage's (a head start for the first stages of all teams).
constexpr uint64_t kFirstStageHeadNs = 3000;

// Suspend hint of the waits below: long enough that a waiting thread sleeps
// instead of spinning (taking issue slots from the other warps), short
// enough that the abort flag and the time bound are still polled.
constexpr uint32_t kWaitSleepHintNs = 20000;

// Wait for phase `parity` of barrier `bar` to complete.  Gives up (returns
// false) after `limit_ns` (default kWaitLimitNs), or early once *abort is set.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepHintNs)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; completion is signalled
// to barrier `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src,
                                         uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data streamed through once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Row partition shared by the backward row pass and its finalize: CTA c of G
// owns rows [floor(c T / G), floor((c+1) T / G)).  With G <= T every range is
// non-empty, and the CTA owning row t is floor(((t+1) G - 1) / T).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t part_begin(int64_t c, int64_t T,
                                                       int64_t G) {
  return (c * T) / G;
}
__host__ __device__ __forceinline__ int64_t part_owner(int64_t t, int64_t T,
                                                       int64_t G) {
  return ((t + 1) * G - 1) / T;
}

}  // namespace adaln
