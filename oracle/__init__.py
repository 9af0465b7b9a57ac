"""CPU oracle for the fused AdaLN LayerNorm-Modulate operator.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
use it.  It is a plain fp64 statement of the operator of AdaptiveLoad's
"Technical summary", section 2.B (fused LayerNorm-Modulate kernels), written
as separate loops in C++ (adaln_oracle.cpp) and called through ctypes.  It
shares no code with the CUDA library.

Inputs are numpy arrays: float32, float64, or uint16 holding bf16 bits (widened
exactly).  Outputs are float64.

Pins: tests/test_oracle_pins.py (closed forms, invariants, finite differences,
torch CPU fp64 layer_norm, exact integer sums) and tests/test_oracle_mutants.py
(planted mistakes that the pins must catch).  No function here is unpinned.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F64 = 0, 1, 2
OK, ERR_ARG, ERR_SEG = 0, 1, 2

_lib = None


def _dtype_code(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle: unsupported input dtype {a.dtype}")


def _bind(lib):
    vp, i64, i32, ci, dbl = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                             ctypes.c_int, ctypes.c_double)
    lib.oracle_hw_threads.restype = ci
    lib.oracle_hw_threads.argtypes = []
    lib.oracle_row_stats.restype = ci
    lib.oracle_row_stats.argtypes = [vp, i64, i32, ci, dbl, vp, vp, ci]
    lib.oracle_adaln_fwd.restype = ci
    lib.oracle_adaln_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, ci, dbl,
                                     vp, i64, vp, vp, vp, ci]
    lib.oracle_adaln_bwd.restype = ci
    lib.oracle_adaln_bwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, ci, dbl,
                                     vp, vp, vp, i64, vp, vp, vp, ci]
    return lib


def load(path=None):
    """Load (building first if needed) the oracle library; cached."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dt is None else a.astype(dt, copy=False))
    return a


def hw_threads(lib=None):
    return (lib or load()).oracle_hw_threads()


def _check(rc, what):
    if rc == ERR_SEG:
        raise ValueError(f"{what}: seg_id outside [0, nseg)")
    if rc != OK:
        raise ValueError(f"{what}: bad arguments (code {rc})")


def row_stats(x, eps, nthreads=None, lib=None):
    """(mean, rstd) fp64 [T] of x [T, D]."""
    lib = lib or load()
    x = _c(x)
    T, D = x.shape
    mean = np.empty(T, np.float64)
    rstd = np.empty(T, np.float64)
    rc = lib.oracle_row_stats(_ptr(x), T, D, _dtype_code(x), float(eps),
                              _ptr(mean), _ptr(rstd), nthreads or hw_threads(lib))
    _check(rc, "row_stats")
    return mean, rstd


def adaln_fwd(x, shift, scale, seg_id, eps, rows=None, nthreads=None, lib=None):
    """Forward.  Returns (y [n, D], mean [n], rstd [n]) fp64 for `rows`
    (all rows when None)."""
    lib = lib or load()
    x, shift, scale = _c(x), _c(shift), _c(scale)
    seg_id = _c(seg_id, np.int32)
    T, D = x.shape
    nseg = shift.shape[0]
    assert shift.dtype == x.dtype == scale.dtype
    assert shift.shape == scale.shape == (nseg, D) and seg_id.shape == (T,)
    rows = _c(rows, np.int64)
    n = T if rows is None else rows.shape[0]
    y = np.empty((n, D), np.float64)
    mean = np.empty(n, np.float64)
    rstd = np.empty(n, np.float64)
    rc = lib.oracle_adaln_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(seg_id),
                              T, D, nseg, _dtype_code(x), float(eps),
                              _ptr(rows), n, _ptr(y), _ptr(mean), _ptr(rstd),
                              nthreads or hw_threads(lib))
    _check(rc, "adaln_fwd")
    return y, mean, rstd


def adaln_bwd(dy, x, scale, seg_id, eps, mean=None, rstd=None, rows=None,
              want_dx=True, want_dmod=True, nthreads=None, lib=None):
    """Backward.  Returns (dx [n, D] or None, dshift [nseg, D] or None,
    dscale [nseg, D] or None), fp64.  mean/rstd (fp32 [T]) select the saved
    statistics mode; otherwise the oracle recomputes them in fp64."""
    lib = lib or load()
    dy, x, scale = _c(dy), _c(x), _c(scale)
    seg_id = _c(seg_id, np.int32)
    T, D = x.shape
    nseg = scale.shape[0]
    assert dy.dtype == x.dtype == scale.dtype and dy.shape == x.shape
    if (mean is None) != (rstd is None):
        raise ValueError("give both mean and rstd, or neither")
    mean = _c(mean, np.float32)
    rstd = _c(rstd, np.float32)
    rows = _c(rows, np.int64)
    n = T if rows is None else rows.shape[0]
    dx = np.empty((n, D), np.float64) if want_dx else None
    dshift = np.empty((nseg, D), np.float64) if want_dmod else None
    dscale = np.empty((nseg, D), np.float64) if want_dmod else None
    rc = lib.oracle_adaln_bwd(_ptr(dy), _ptr(x), _ptr(scale), _ptr(seg_id),
                              T, D, nseg, _dtype_code(x), float(eps),
                              _ptr(mean), _ptr(rstd), _ptr(rows), n, _ptr(dx),
                              _ptr(dshift), _ptr(dscale),
                              nthreads or hw_threads(lib))
    _check(rc, "adaln_bwd")
    return dx, dshift, dscale
