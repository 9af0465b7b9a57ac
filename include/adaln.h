/*
 * libadaln -- fused AdaLN LayerNorm-Modulate for GB300 (sm_103a).
 *
 * The operator is the fused adaptive LayerNorm of video / MMDiT diffusion
 * transformers described in "AdaptiveLoad: Towards Efficient Video Diffusion
 * Transformer Training", Technical summary, section 2.B ("Fused
 * LayerNorm-Modulate CUDA kernels"): normalisation and modulation in a single
 * kernel launch (forward), and a backward whose modulation-gradient reduction
 * along the sequence dimension is laid out so that each thread owns a feature
 * column d and accumulates down the sequence (the "D-tile coalesced
 * reduction").  The pages give no formula; this library computes, for every
 * token row t of a packed variable-length batch with b = seg_id[t]:
 *
 *   mean[t] = (1/D) sum_d x[t,d]
 *   var[t]  = (1/D) sum_d (x[t,d] - mean[t])^2         (biased)
 *   rstd[t] = 1 / sqrt(var[t] + eps)
 *   xhat    = (x - mean[t]) * rstd[t]
 *   y       = xhat * (1 + scale[b,d]) + shift[b,d]
 *   g       = dy * (1 + scale[b,d])
 *   dx      = rstd[t] * (g - mean_d(g) - xhat * mean_d(g * xhat))
 *   dscale[b,d] = sum_{t: seg_id[t]=b} dy[t,d] * xhat[t,d]
 *   dshift[b,d] = sum_{t: seg_id[t]=b} dy[t,d]
 *
 * Layout: all tensors row-major and contiguous.  x, y, dy, dx are [T, D];
 * shift, scale are [nseg, D]; all of these have the element type `dtype`.
 * seg_id is int32 [T]; mean, rstd are fp32 [T]; dshift, dscale are fp32
 * [nseg, D].  Arithmetic is fp32; bf16 outputs are rounded once (to nearest
 * even) at the store.
 *
 * Ownership: every pointer is owned by the caller and must point to device
 * memory of the current CUDA device (except host_* arguments).  The library
 * never allocates, frees or retains caller memory.
 *
 * Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 * default stream) and the calls return without synchronising.  The kernels
 * are launched as programmatic dependents of the stream's previous kernel:
 * they may be scheduled while it ends, but read nothing before it has
 * completed.  They also let the stream's next kernel be scheduled before they
 * complete; a kernel launched after them with programmatic stream
 * serialization must wait (cudaGridDependencySynchronize) before reading
 * their outputs, as that launch mode requires anyway.  Ordinary launches,
 * copies and events see the usual stream order.  Return codes
 * report errors detectable on the host before launch, and launch failures.
 * Data errors found on the device (a seg_id outside [0, nseg) or decreasing
 * along the rows) are clamped so that every access stays in bounds, and are
 * recorded in a status word read by adaln_get_status() (per device, or one the
 * calling thread bound with adaln_status_bind()); outputs of such a call are
 * unspecified.
 *
 * Preconditions (checked, ADALN_ERR_* on violation):
 *   - T >= 0 (T = 0 does nothing, except that adaln_bwd zeroes dshift/dscale);
 *   - D >= 1, D * sizeof(element) a multiple of 16 bytes (D % 8 == 0 for bf16,
 *     D % 4 == 0 for fp32), D <= ADALN_MAX_D_BF16 / ADALN_MAX_D_F32;
 *   - 1 <= nseg <= ADALN_MAX_NSEG;
 *   - x, y, dy, dx, shift, scale, dshift, dscale and the workspace 16-byte
 *     aligned; seg_id, mean, rstd 4-byte aligned;
 *   - eps finite and >= 0;
 *   - seg_id non-decreasing along rows (segments packed contiguously), values
 *     in [0, nseg).  Segments may be empty.
 */
#ifndef ADALN_H
#define ADALN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbol visibility of the exported entry points. */
#if defined(__GNUC__)
#define ADALN_API __attribute__((visibility("default")))
#else
#define ADALN_API
#endif

#define ADALN_MAX_D_BF16 8192
#define ADALN_MAX_D_F32 4096
#define ADALN_MAX_NSEG (1 << 24)

typedef enum {
  ADALN_F32 = 0,  /* IEEE binary32 */
  ADALN_BF16 = 1  /* bfloat16 */
} adaln_dtype_t;

typedef enum {
  ADALN_OK = 0,
  ADALN_ERR_NULL = 1,      /* a required pointer is NULL */
  ADALN_ERR_DIM = 2,       /* T, D or nseg outside the supported range */
  ADALN_ERR_ALIGN = 3,     /* a pointer is not aligned as required */
  ADALN_ERR_DTYPE = 4,     /* unknown dtype */
  ADALN_ERR_SEG = 5,       /* device status: seg_id out of range or decreasing */
  ADALN_ERR_WORKSPACE = 6, /* workspace smaller than required */
  ADALN_ERR_CUDA = 7,      /* a CUDA runtime call or launch failed */
  ADALN_ERR_ARG = 8,       /* eps negative or not finite; bad trace argument */
  ADALN_ERR_TIMEOUT = 9    /* device status: an internal pipeline wait gave up */
} adaln_status_t;

/* Bits of the device status word (adaln_get_status). */
#define ADALN_DEV_SEG_RANGE 1u   /* a seg_id was outside [0, nseg) */
#define ADALN_DEV_SEG_ORDER 2u   /* seg_id decreased from one row to the next */
#define ADALN_DEV_TIMEOUT 4u     /* a bounded wait on a copy pipeline expired */

/*
 * Forward (section 2.B, forward pass): per-row statistics reduced on chip and
 * the modulation applied in the same launch.  Reads x once, writes y, mean,
 * rstd.  One kernel launch on `stream`.
 */
ADALN_API int adaln_fwd(const void* x, const void* shift, const void* scale,
              const int32_t* seg_id, int64_t T, int32_t D, int32_t nseg,
              adaln_dtype_t dtype, float eps, void* y, float* mean,
              float* rstd, void* stream);

/*
 * Bytes of device workspace adaln_bwd needs for these sizes on the current
 * device (it depends on the device's SM count).  Written to *bytes.
 */
ADALN_API int adaln_bwd_workspace_size(int64_t T, int32_t D, int32_t nseg,
                             adaln_dtype_t dtype, size_t* bytes);

/*
 * Backward (section 2.B, backward pass with the D-tile coalesced reduction).
 * Reads dy and x once (plus the saved mean/rstd), writes dx [T, D] and the
 * fp32 sequence reductions dshift, dscale [nseg, D].  Two kernel launches on
 * `stream`: a row pass that also accumulates per-(CTA, segment) column
 * partials into `workspace`, then a fixed-order reduction of those partials.
 * No floating-point atomics: for a given device and sizes the results of
 * valid input are bitwise reproducible.  (With an invalid seg_id the outputs
 * are unspecified and may differ between runs: teams whose clamped segment
 * paths cross can share a partial slot.)  `workspace` (at least
 * adaln_bwd_workspace_size bytes, 16-byte aligned) is scratch owned by the
 * caller; its contents on entry do not matter.  Calls sharing one workspace
 * must not overlap on the device.  A NULL workspace is ADALN_ERR_NULL
 * (adaln_bwd_noalloc serves callers without one); a short one is
 * ADALN_ERR_WORKSPACE.
 */
ADALN_API int adaln_bwd(const void* dy, const void* x, const float* mean,
              const float* rstd, const void* scale, const int32_t* seg_id,
              int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype,
              void* dx, float* dshift, float* dscale, void* workspace,
              size_t workspace_bytes, void* stream);

/*
 * Backward that allocates nothing, for callers that cannot call cudaMalloc
 * (for example code inside a host framework whose allocator owns all device
 * memory, or code on a latency-critical path where allocating would
 * synchronise the device).  The paper has no counterpart: this is a
 * deployment variant of adaln_bwd.  Same arguments, results and launches as
 * adaln_bwd, minus the workspace: the scratch is a fixed file-scope device
 * array of ADALN_NOALLOC_SCRATCH_BYTES.  A device holds it from the first
 * adaln_bwd_noalloc call on it (under CUDA's default lazy module loading;
 * from the library's first use there under eager loading) until the process
 * exits.  The partials grow with the SM count (G = SMs x teams per SM):
 * 3072-wide bf16 rows with 822 segments fit up to 181 SMs.  Sizes whose
 * adaln_bwd_workspace_size exceeds it are rejected with ADALN_ERR_WORKSPACE
 * before anything is launched.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  All calls on a device share the array and it
 * keeps the last call's contents (nothing in it needs to start at zero);
 * calls that overlap on the GPU race on it.  No cudaMalloc, cudaFree or other
 * allocating routine is called.
 */
#define ADALN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
ADALN_API int adaln_bwd_noalloc(const void* dy, const void* x, const float* mean,
              const float* rstd, const void* scale, const int32_t* seg_id,
              int64_t T, int32_t D, int32_t nseg, adaln_dtype_t dtype,
              void* dx, float* dshift, float* dscale, void* stream);

/*
 * One forward + backward step on HOST-resident tensors: the operator of
 * section 2.B of the AdaptiveLoad technical summary, as adaln_fwd followed by
 * adaln_bwd (the formulas at the top of this file), for training steps whose
 * tensors live in host memory.  The pages describe no host pipeline; this
 * entry point is this library's own.
 *
 * Rows are processed in chunks of at most `chunk_rows` (0 = about 32 MB per
 * [rows, D] tensor and chunk; shorter chunks at both ends shorten the time
 * the link carries one direction only): the copies of chunk i + 1 in and of
 * chunk i - 1 out overlap the kernels of chunk i, on three internal streams
 * of the current device.  The step starts after the work already queued on
 * `stream` and after the previous call of this function on the device;
 * `stream` waits for the whole step (the host buffers may be read once it
 * has drained).
 *
 * Arguments: x, dy, shift, scale, seg_id are HOST pointers read by the step;
 * y, mean, rstd, dx, dshift, dscale are HOST pointers it writes; shapes and
 * element types as above.  Page-locked (pinned) host memory lets the copies
 * run asynchronously; pageable memory works but serialises them.  `scratch`
 * is DEVICE memory of at least adaln_fwd_bwd_host_scratch_size(T, D, nseg,
 * dtype, chunk_rows) bytes, 256-byte aligned, owned by the caller; calls on
 * different scratch buffers may share none of them while in flight.
 *
 * Results: y, mean, rstd, dx equal those of the device calls bit for bit;
 * dshift, dscale add the chunks' per-segment sums in chunk order (a fixed
 * association, deterministic for a given chunk size).
 *
 * Errors: ADALN_ERR_DIM, _DTYPE as for adaln_fwd; ADALN_ERR_NULL for a NULL
 * pointer (row pointers may be NULL when T = 0); ADALN_ERR_ARG for a bad eps
 * or a negative chunk_rows; ADALN_ERR_ALIGN when scratch is not 256-byte
 * aligned; ADALN_ERR_WORKSPACE when scratch_bytes is too small;
 * ADALN_ERR_CUDA when a copy or launch fails
 * (work enqueued before the failure may still run).  Device data errors go
 * to the status word as for the device calls.
 */
ADALN_API int adaln_fwd_bwd_host_scratch_size(int64_t T, int32_t D, int32_t nseg,
              adaln_dtype_t dtype, int64_t chunk_rows, size_t* bytes);
ADALN_API int adaln_fwd_bwd_host(const void* x, const void* dy, const void* shift,
              const void* scale, const int32_t* seg_id, int64_t T, int32_t D,
              int32_t nseg, adaln_dtype_t dtype, float eps, void* y, float* mean,
              float* rstd, void* dx, float* dshift, float* dscale,
              int64_t chunk_rows, void* scratch, size_t scratch_bytes, void* stream);

/*
 * Synchronise `stream`, then read and clear the status word: the one the
 * calling thread bound (adaln_status_bind), else the current device's.
 * *host_bits (if non-NULL) receives the ADALN_DEV_* bits.  Returns ADALN_OK,
 * ADALN_ERR_SEG, ADALN_ERR_TIMEOUT or ADALN_ERR_CUDA.  The device's word is
 * shared by all calls on the device that use it since it was last cleared.
 */
ADALN_API int adaln_get_status(uint32_t* host_bits, void* stream);

/*
 * Bind a caller-owned device status word for the calls the calling host
 * thread makes from now on (its kernels OR ADALN_DEV_* bits into it, and
 * adaln_get_status() reads and clears it), instead of the device's shared
 * word; NULL returns to the shared word.  For callers that drive several
 * streams: with one word per stream (bound by the thread issuing that
 * stream's calls), a data error is reported to the caller whose call caused
 * it.  `device_word` is a 4-byte aligned uint32 in device memory of the
 * device the calls run on, owned by the caller, zeroed by the caller before
 * first use, and left bound until unbound or the thread exits (the library
 * keeps only the pointer).  Returns ADALN_OK or ADALN_ERR_ALIGN.  The paper
 * describes no status reporting; this is the library's own.
 */
ADALN_API int adaln_status_bind(uint32_t* device_word);

/* Static description of a status code. */
ADALN_API const char* adaln_strerror(int code);

/*
 * Kernel timing trace.  Between adaln_trace_begin(capacity) and
 * adaln_trace_end(), every kernel launch made by this library (from any
 * thread) is bracketed by a pair of CUDA events recorded on its stream, up to
 * `capacity` launches.  adaln_trace_end() synchronises those events and sums
 * the elapsed time per kernel; adaln_trace_get() reads the sums.
 * Kernel ids: ADALN_KERNEL_FWD, ADALN_KERNEL_BWD_ROWS, ADALN_KERNEL_BWD_FINALIZE.
 */
#define ADALN_KERNEL_FWD 0
#define ADALN_KERNEL_BWD_ROWS 1
#define ADALN_KERNEL_BWD_FINALIZE 2
#define ADALN_NUM_KERNELS 3
ADALN_API int adaln_trace_begin(int capacity);
ADALN_API int adaln_trace_end(void);
ADALN_API int adaln_trace_get(int kernel_id, int64_t* launches, double* total_ms);

/*
 * Self-test of failure detection: launches one thread that waits, through the
 * bounded wait the staging pipelines use, on an mbarrier that nothing ever
 * completes, giving up after limit_us microseconds (1..100000).  On return of
 * the next adaln_get_status() the device status word must hold
 * ADALN_DEV_TIMEOUT (ADALN_ERR_TIMEOUT), and the device must remain usable.
 * The pipelines' own limit is 2 s; the staging kernels never wait unbounded.
 */
ADALN_API int adaln_selftest_wait_timeout(uint32_t limit_us, void* stream);

/*
 * Launch shape chosen for these sizes on the current device: grid (CTAs),
 * threads per CTA, ring stages, dynamic shared memory bytes.  `which` is
 * ADALN_KERNEL_FWD or ADALN_KERNEL_BWD_ROWS.  For reports and tests.
 */
ADALN_API int adaln_launch_shape(int which, int64_t T, int32_t D, int32_t nseg,
                       adaln_dtype_t dtype, int32_t* grid, int32_t* threads,
                       int32_t* stages, int32_t* smem_bytes);

#ifdef __cplusplus
}
#endif
#endif /* ADALN_H */
