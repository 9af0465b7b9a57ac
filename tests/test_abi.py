"""The C-ABI library: it loads, exports every entry point declared in
include/*.h, and rejects bad arguments on the host before any CUDA call
(no GPU is touched by these tests)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from adaln_video_dit_gb300 import build
    build.build()
    from adaln_video_dit_gb300 import _lib
    return _lib


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"^ADALN_API\s+[\w\s\*]+?\b(adaln_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(lib.raw, n)
    # nothing else with the library prefix leaks out
    assert {e for e in exported if e.startswith("adaln_")} == set(names)
    assert set(lib.EXPORTS) == set(names)


def test_strerror_covers_codes(lib):
    msgs = {lib.strerror(c) for c in range(10)}
    assert len(msgs) == 10
    assert lib.strerror(12345) == "unknown status code"


P16 = ctypes.c_void_p(0x10000)       # 16-byte aligned fake addresses: never dereferenced
P16b = ctypes.c_void_p(0x20000)
P_ODD = ctypes.c_void_p(0x10008)     # 8-byte aligned only


def fwd(lib, **kw):
    a = dict(x=P16, shift=P16, scale=P16, seg=P16, T=10, D=64, nseg=1, dt=lib.ADALN_BF16,
             eps=1e-6, y=P16b, mean=P16b, rstd=P16b)
    a.update(kw)
    return lib.raw.adaln_fwd(a["x"], a["shift"], a["scale"], a["seg"], a["T"], a["D"],
                             a["nseg"], a["dt"], a["eps"], a["y"], a["mean"], a["rstd"], None)


def test_fwd_argument_checks(lib):
    assert fwd(lib, dt=7) == lib.ADALN_ERR_DTYPE
    assert fwd(lib, T=-1) == lib.ADALN_ERR_DIM
    assert fwd(lib, D=12) == lib.ADALN_ERR_DIM          # 24 bytes: not a 16-byte multiple
    assert fwd(lib, D=0) == lib.ADALN_ERR_DIM
    assert fwd(lib, D=8192 + 8) == lib.ADALN_ERR_DIM
    assert fwd(lib, D=4100, dt=lib.ADALN_F32) == lib.ADALN_ERR_DIM
    assert fwd(lib, D=6, dt=lib.ADALN_F32) == lib.ADALN_ERR_DIM
    assert fwd(lib, nseg=0) == lib.ADALN_ERR_DIM
    assert fwd(lib, x=None) == lib.ADALN_ERR_NULL
    assert fwd(lib, rstd=None) == lib.ADALN_ERR_NULL
    assert fwd(lib, x=P_ODD) == lib.ADALN_ERR_ALIGN
    assert fwd(lib, y=P_ODD) == lib.ADALN_ERR_ALIGN
    assert fwd(lib, seg=ctypes.c_void_p(0x10002)) == lib.ADALN_ERR_ALIGN
    assert fwd(lib, eps=-1.0) == lib.ADALN_ERR_ARG
    assert fwd(lib, eps=float("nan")) == lib.ADALN_ERR_ARG
    # T = 0 is a no-op that touches nothing
    assert fwd(lib, T=0, x=None, y=None) == lib.ADALN_OK


def bwd(lib, **kw):
    a = dict(dy=P16, x=P16, mean=P16, rstd=P16, scale=P16, seg=P16, T=10, D=64, nseg=2,
             dt=lib.ADALN_BF16, dx=P16b, dshift=P16b, dscale=P16b, ws=P16b, wsb=1 << 20)
    a.update(kw)
    return lib.raw.adaln_bwd(a["dy"], a["x"], a["mean"], a["rstd"], a["scale"], a["seg"],
                             a["T"], a["D"], a["nseg"], a["dt"], a["dx"], a["dshift"],
                             a["dscale"], a["ws"], a["wsb"], None)


def test_bwd_argument_checks(lib):
    assert bwd(lib, dt=3) == lib.ADALN_ERR_DTYPE
    assert bwd(lib, D=20) == lib.ADALN_ERR_DIM
    assert bwd(lib, nseg=-2) == lib.ADALN_ERR_DIM
    assert bwd(lib, ws=None) == lib.ADALN_ERR_NULL
    assert bwd(lib, dscale=None) == lib.ADALN_ERR_NULL
    assert bwd(lib, dy=None) == lib.ADALN_ERR_NULL
    assert bwd(lib, dx=P_ODD) == lib.ADALN_ERR_ALIGN
    assert bwd(lib, ws=P_ODD) == lib.ADALN_ERR_ALIGN
    assert bwd(lib, dshift=P_ODD) == lib.ADALN_ERR_ALIGN


def test_trace_argument_checks(lib):
    assert lib.raw.adaln_trace_get(5, None, None) == lib.ADALN_ERR_ARG
    assert lib.raw.adaln_trace_get(-1, None, None) == lib.ADALN_ERR_ARG
    assert lib.raw.adaln_trace_begin(0) == lib.ADALN_ERR_ARG
    n = ctypes.c_int64(-1)
    ms = ctypes.c_double(-1)
    assert lib.raw.adaln_trace_get(0, ctypes.byref(n), ctypes.byref(ms)) == lib.ADALN_OK
    assert n.value == 0 and ms.value == 0.0


def test_status_bind_checks_alignment_on_host(lib):
    assert lib.raw.adaln_status_bind(ctypes.c_void_p(0x1002)) == lib.ADALN_ERR_ALIGN
    assert lib.raw.adaln_status_bind(None) == lib.ADALN_OK  # unbinding needs no GPU


def test_selftest_limit_is_checked_on_host(lib):
    assert lib.raw.adaln_selftest_wait_timeout(0, None) == lib.ADALN_ERR_ARG
    assert lib.raw.adaln_selftest_wait_timeout(100001, None) == lib.ADALN_ERR_ARG


def test_binding_rejects_host_tensors(lib):
    import torch
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lib.adaln_fwd(x, x[:1], x[:1], torch.zeros(4, dtype=torch.int32), 1e-6)
    with pytest.raises(TypeError):
        lib.dtype_code(torch.float16)


def host_step(lib, **kw):
    a = dict(x=P16, dy=P16, shift=P16, scale=P16, seg=P16, T=10, D=64, nseg=2,
             dt=lib.ADALN_BF16, eps=1e-6, y=P16b, mean=P16b, rstd=P16b, dx=P16b, dshift=P16b,
             dscale=P16b, chunk=0, scratch=ctypes.c_void_p(0x100000), sb=1 << 30)
    a.update(kw)
    return lib.raw.adaln_fwd_bwd_host(a["x"], a["dy"], a["shift"], a["scale"], a["seg"], a["T"],
                                      a["D"], a["nseg"], a["dt"], a["eps"], a["y"], a["mean"],
                                      a["rstd"], a["dx"], a["dshift"], a["dscale"], a["chunk"],
                                      a["scratch"], a["sb"], None)


def test_host_step_argument_checks(lib):
    assert host_step(lib, dt=2) == lib.ADALN_ERR_DTYPE
    assert host_step(lib, D=12) == lib.ADALN_ERR_DIM
    assert host_step(lib, nseg=0) == lib.ADALN_ERR_DIM
    assert host_step(lib, scratch=None) == lib.ADALN_ERR_NULL
    assert host_step(lib, dshift=None) == lib.ADALN_ERR_NULL
    assert host_step(lib, dx=None) == lib.ADALN_ERR_NULL
    assert host_step(lib, scratch=P_ODD) == lib.ADALN_ERR_ALIGN  # 256-byte rule
    assert host_step(lib, scratch=ctypes.c_void_p(0x10010)) == lib.ADALN_ERR_ALIGN
    assert host_step(lib, eps=float("inf")) == lib.ADALN_ERR_ARG
    assert host_step(lib, chunk=-1) == lib.ADALN_ERR_ARG
    n = ctypes.c_size_t(0)
    assert lib.raw.adaln_fwd_bwd_host_scratch_size(10, 64, 2, lib.ADALN_BF16, -5,
                                                   ctypes.byref(n)) == lib.ADALN_ERR_ARG
    assert lib.raw.adaln_fwd_bwd_host_scratch_size(10, 64, 2, lib.ADALN_BF16, 0,
                                                   None) == lib.ADALN_ERR_NULL
