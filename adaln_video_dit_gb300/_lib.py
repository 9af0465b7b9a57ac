"""ctypes binding of libadaln.so (C ABI: include/adaln.h).

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels.  torch supplies device memory, streams and output allocation.
The functions carry the C names.  There is no fallback: if libadaln.so is
missing or a call fails, an exception is raised.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libadaln.so")

ADALN_F32, ADALN_BF16 = 0, 1
(ADALN_OK, ADALN_ERR_NULL, ADALN_ERR_DIM, ADALN_ERR_ALIGN, ADALN_ERR_DTYPE,
 ADALN_ERR_SEG, ADALN_ERR_WORKSPACE, ADALN_ERR_CUDA, ADALN_ERR_ARG,
 ADALN_ERR_TIMEOUT) = range(10)
ADALN_DEV_SEG_RANGE, ADALN_DEV_SEG_ORDER, ADALN_DEV_TIMEOUT = 1, 2, 4
ADALN_KERNEL_FWD, ADALN_KERNEL_BWD_ROWS, ADALN_KERNEL_BWD_FINALIZE = 0, 1, 2
KERNEL_NAMES = {0: "adaln_fwd_kernel", 1: "adaln_bwd_rows_kernel",
                2: "adaln_bwd_finalize_kernel"}

NOALLOC_SCRATCH_BYTES = 32 << 20

EXPORTS = ["adaln_fwd", "adaln_bwd_workspace_size", "adaln_bwd", "adaln_bwd_noalloc",
           "adaln_get_status", "adaln_status_bind", "adaln_strerror", "adaln_trace_begin",
           "adaln_trace_end", "adaln_trace_get", "adaln_launch_shape",
           "adaln_selftest_wait_timeout", "adaln_fwd_bwd_host_scratch_size",
           "adaln_fwd_bwd_host"]


class AdalnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libadaln.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, ci, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                             ctypes.c_int, ctypes.c_float)
    lib.adaln_fwd.restype = ci
    lib.adaln_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, ci, f32, vp, vp, vp, vp]
    lib.adaln_bwd_workspace_size.restype = ci
    lib.adaln_bwd_workspace_size.argtypes = [i64, i32, i32, ci, ctypes.POINTER(ctypes.c_size_t)]
    lib.adaln_bwd.restype = ci
    lib.adaln_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, ci, vp, vp, vp,
                              vp, ctypes.c_size_t, vp]
    lib.adaln_bwd_noalloc.restype = ci
    lib.adaln_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, ci, vp, vp, vp, vp]
    lib.adaln_get_status.restype = ci
    lib.adaln_get_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.adaln_status_bind.restype = ci
    lib.adaln_status_bind.argtypes = [vp]
    lib.adaln_strerror.restype = ctypes.c_char_p
    lib.adaln_strerror.argtypes = [ci]
    lib.adaln_trace_begin.restype = ci
    lib.adaln_trace_begin.argtypes = [ci]
    lib.adaln_trace_end.restype = ci
    lib.adaln_trace_end.argtypes = []
    lib.adaln_trace_get.restype = ci
    lib.adaln_trace_get.argtypes = [ci, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.adaln_fwd_bwd_host_scratch_size.restype = ci
    lib.adaln_fwd_bwd_host_scratch_size.argtypes = [i64, i32, i32, ci, i64,
                                                    ctypes.POINTER(ctypes.c_size_t)]
    lib.adaln_fwd_bwd_host.restype = ci
    lib.adaln_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, ci, f32, vp, vp, vp,
                                       vp, vp, vp, i64, vp, ctypes.c_size_t, vp]
    lib.adaln_selftest_wait_timeout.restype = ci
    lib.adaln_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    lib.adaln_launch_shape.restype = ci
    lib.adaln_launch_shape.argtypes = [ci, i64, i32, i32, ci] + [ctypes.POINTER(i32)] * 4
    return lib


raw = _load()


def strerror(code):
    return raw.adaln_strerror(int(code)).decode()


def _check(rc, what):
    if rc != ADALN_OK:
        raise AdalnError(rc, what)


def dtype_code(t):
    if t == torch.bfloat16:
        return ADALN_BF16
    if t == torch.float32:
        return ADALN_F32
    raise TypeError(f"libadaln supports bfloat16 and float32, not {t}")


def _stream_ptr(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t, name, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def adaln_fwd(x, shift, scale, seg_id, eps, y=None, mean=None, rstd=None, stream=None):
    """y = (x - mean) * rstd * (1 + scale[seg_id]) + shift[seg_id].

    x [T, D]; shift, scale [nseg, D] (x's dtype); seg_id int32 [T].
    Returns (y, mean, rstd); outputs are allocated when not given."""
    T, D = x.shape
    nseg = shift.shape[0]
    dt = x.dtype
    _dev(x, "x", dt)
    _dev(shift, "shift", dt, (nseg, D))
    _dev(scale, "scale", dt, (nseg, D))
    _dev(seg_id, "seg_id", torch.int32, (T,))
    y = torch.empty_like(x) if y is None else _dev(y, "y", dt, (T, D))
    mean = torch.empty(T, device=x.device, dtype=torch.float32) if mean is None else _dev(mean, "mean", torch.float32, (T,))
    rstd = torch.empty(T, device=x.device, dtype=torch.float32) if rstd is None else _dev(rstd, "rstd", torch.float32, (T,))
    rc = raw.adaln_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(seg_id), T, D, nseg,
                       dtype_code(dt), float(eps), _ptr(y), _ptr(mean), _ptr(rstd),
                       _stream_ptr(stream, x.device))
    _check(rc, "adaln_fwd")
    return y, mean, rstd


def adaln_bwd_workspace_size(T, D, nseg, dtype):
    """Workspace bytes adaln_bwd needs on the current device."""
    n = ctypes.c_size_t(0)
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    _check(raw.adaln_bwd_workspace_size(int(T), int(D), int(nseg), code, ctypes.byref(n)),
           "adaln_bwd_workspace_size")
    return n.value


def adaln_bwd(dy, x, mean, rstd, scale, seg_id, dx=None, dshift=None, dscale=None,
              workspace=None, stream=None):
    """Backward of adaln_fwd.  Returns (dx [T, D] in x's dtype, dshift, dscale
    [nseg, D] fp32).  `workspace` is a uint8 CUDA tensor of at least
    adaln_bwd_workspace_size bytes (allocated when not given)."""
    T, D = x.shape
    nseg = scale.shape[0]
    dt = x.dtype
    _dev(dy, "dy", dt, (T, D))
    _dev(x, "x", dt)
    _dev(mean, "mean", torch.float32, (T,))
    _dev(rstd, "rstd", torch.float32, (T,))
    _dev(scale, "scale", dt, (nseg, D))
    _dev(seg_id, "seg_id", torch.int32, (T,))
    dx = torch.empty_like(x) if dx is None else _dev(dx, "dx", dt, (T, D))
    dshift = (torch.empty(nseg, D, device=x.device, dtype=torch.float32) if dshift is None
              else _dev(dshift, "dshift", torch.float32, (nseg, D)))
    dscale = (torch.empty(nseg, D, device=x.device, dtype=torch.float32) if dscale is None
              else _dev(dscale, "dscale", torch.float32, (nseg, D)))
    need = adaln_bwd_workspace_size(T, D, nseg, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    _dev(workspace, "workspace")
    rc = raw.adaln_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(seg_id),
                       T, D, nseg, dtype_code(dt), _ptr(dx), _ptr(dshift), _ptr(dscale),
                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                       _stream_ptr(stream, x.device))
    _check(rc, "adaln_bwd")
    return dx, dshift, dscale


def adaln_bwd_noalloc(dy, x, mean, rstd, scale, seg_id, dx=None, dshift=None, dscale=None,
                      stream=None):
    """adaln_bwd without a workspace argument: for callers that cannot
    allocate device memory, the library uses its fixed static scratch array
    (ADALN_NOALLOC_SCRATCH_BYTES per device, shared by all calls; calls that
    overlap on the GPU race).  Outputs are allocated here only when not
    given; pass them in to allocate nothing."""
    T, D = x.shape
    nseg = scale.shape[0]
    dt = x.dtype
    _dev(dy, "dy", dt, (T, D))
    _dev(x, "x", dt)
    _dev(mean, "mean", torch.float32, (T,))
    _dev(rstd, "rstd", torch.float32, (T,))
    _dev(scale, "scale", dt, (nseg, D))
    _dev(seg_id, "seg_id", torch.int32, (T,))
    dx = torch.empty_like(x) if dx is None else _dev(dx, "dx", dt, (T, D))
    dshift = (torch.empty(nseg, D, device=x.device, dtype=torch.float32) if dshift is None
              else _dev(dshift, "dshift", torch.float32, (nseg, D)))
    dscale = (torch.empty(nseg, D, device=x.device, dtype=torch.float32) if dscale is None
              else _dev(dscale, "dscale", torch.float32, (nseg, D)))
    rc = raw.adaln_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale),
                               _ptr(seg_id), T, D, nseg, dtype_code(dt), _ptr(dx),
                               _ptr(dshift), _ptr(dscale), _stream_ptr(stream, x.device))
    _check(rc, "adaln_bwd_noalloc")
    return dx, dshift, dscale


def adaln_fwd_bwd_host_scratch_size(T, D, nseg, dtype, chunk_rows=0):
    """Device scratch bytes adaln_fwd_bwd_host needs."""
    n = ctypes.c_size_t(0)
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    _check(raw.adaln_fwd_bwd_host_scratch_size(int(T), int(D), int(nseg), code, int(chunk_rows),
                                               ctypes.byref(n)), "adaln_fwd_bwd_host_scratch_size")
    return n.value


def _host(t, name, dtype=None, shape=None):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def adaln_fwd_bwd_host(x, dy, shift, scale, seg_id, eps, out, scratch, chunk_rows=0,
                       stream=None):
    """Forward + backward on host tensors (pinned for overlap), pipelined in row
    chunks.  `out` is a dict of preallocated host tensors y, mean, rstd, dx,
    dshift, dscale; `scratch` a uint8 CUDA tensor of at least
    adaln_fwd_bwd_host_scratch_size bytes.  Asynchronous on `stream`."""
    T, D = x.shape
    nseg = shift.shape[0]
    dt = x.dtype
    _host(x, "x", dt)
    _host(dy, "dy", dt, (T, D))
    _host(shift, "shift", dt, (nseg, D))
    _host(scale, "scale", dt, (nseg, D))
    _host(seg_id, "seg_id", torch.int32, (T,))
    _host(out["y"], "y", dt, (T, D))
    _host(out["dx"], "dx", dt, (T, D))
    for k in ("mean", "rstd"):
        _host(out[k], k, torch.float32, (T,))
    for k in ("dshift", "dscale"):
        _host(out[k], k, torch.float32, (nseg, D))
    _dev(scratch, "scratch")
    rc = raw.adaln_fwd_bwd_host(_ptr(x), _ptr(dy), _ptr(shift), _ptr(scale), _ptr(seg_id), T, D,
                                nseg, dtype_code(dt), float(eps), _ptr(out["y"]),
                                _ptr(out["mean"]), _ptr(out["rstd"]), _ptr(out["dx"]),
                                _ptr(out["dshift"]), _ptr(out["dscale"]), int(chunk_rows),
                                _ptr(scratch), scratch.numel() * scratch.element_size(),
                                _stream_ptr(stream, scratch.device))
    _check(rc, "adaln_fwd_bwd_host")


def adaln_get_status(stream=None, device=None):
    """Synchronise the stream, read and clear the device status word.
    Returns (code, bits)."""
    bits = ctypes.c_uint32(0)
    dev = device if device is not None else torch.cuda.current_device()
    rc = raw.adaln_get_status(ctypes.byref(bits), _stream_ptr(stream, dev))
    return rc, bits.value


def adaln_status_bind(word):
    """Bind a caller-owned device status word (an int32 CUDA tensor of one
    element, zeroed) for the calls this host thread makes; None unbinds."""
    if word is not None:
        _dev(word, "status word", torch.int32, (1,))
    _check(raw.adaln_status_bind(_ptr(word)), "adaln_status_bind")


def adaln_strerror(code):
    return strerror(code)


def adaln_trace_begin(capacity):
    _check(raw.adaln_trace_begin(int(capacity)), "adaln_trace_begin")


def adaln_trace_end():
    _check(raw.adaln_trace_end(), "adaln_trace_end")


def adaln_trace_get(kernel_id):
    """(launches, total_ms) recorded for a kernel id in the last trace."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(raw.adaln_trace_get(int(kernel_id), ctypes.byref(n), ctypes.byref(ms)),
           "adaln_trace_get")
    return n.value, ms.value


def adaln_selftest_wait_timeout(limit_us, stream=None):
    """Launch the bounded-wait self-test (see include/adaln.h)."""
    dev = torch.cuda.current_device()
    _check(raw.adaln_selftest_wait_timeout(int(limit_us), _stream_ptr(stream, dev)),
           "adaln_selftest_wait_timeout")


def adaln_launch_shape(which, T, D, nseg, dtype):
    """dict(grid, threads, stages, smem) for ADALN_KERNEL_FWD / _BWD_ROWS."""
    vals = [ctypes.c_int32(0) for _ in range(4)]
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    _check(raw.adaln_launch_shape(int(which), int(T), int(D), int(nseg), code,
                                  *[ctypes.byref(v) for v in vals]), "adaln_launch_shape")
    return dict(zip(("grid", "threads", "stages", "smem"), (v.value for v in vals)))
