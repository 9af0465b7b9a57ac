"""adaln_bwd_noalloc: the backward for callers that cannot allocate device
memory (code running inside a host framework whose allocator owns all device
memory, or on a path where an allocation would synchronise the device).  Its
scratch is the library's fixed static device array.

Called through the C ABI on two calls in a row with different inputs, so the
second call runs on scratch that still holds the first call's partials.  Each
call's outputs sit inside guard bands and are compared with the CPU oracle
(within the tolerances of the other parity tests, from the oracle's own
statistics and from the GPU's saved ones) and with the existing adaln_bwd
entry point (caller-provided workspace), which must give the same bits.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, d, mean, rstd, dtype, T, D, nseg):
    g, out = {}, {}
    g["dx"], out["dx"] = H.guarded_empty((T, D), dtype)
    g["dshift"], out["dshift"] = H.guarded_empty((nseg, D), torch.float32)
    g["dscale"], out["dscale"] = H.guarded_empty((nseg, D), torch.float32)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.raw.adaln_bwd_noalloc(_p(d["dy"]), _p(d["x"]), _p(mean), _p(rstd), _p(d["scale"]),
                                 _p(d["seg_id"]), T, D, nseg, L.dtype_code(dtype),
                                 _p(out["dx"]), _p(out["dshift"]), _p(out["dscale"]), stream)
    assert rc == L.ADALN_OK, L.strerror(rc)
    H.check_guards(g)
    return out


def _check_oracle(c, d, out, mean, rstd):
    dt = c["dtype"]
    x, dy, seg, sc = c["x"], c["dy"], c["seg_id"], d["scale_np"]
    dx_ref, dsh_ref, dsc_ref = oracle.adaln_bwd(dy, x, sc, seg, c["eps"])
    H.check_rowwise("dx", dt, H.to_f64(out["dx"]), dx_ref)
    H.check_norm("dshift", dt, H.to_f64(out["dshift"]), dsh_ref)
    H.check_norm("dscale", dt, H.to_f64(out["dscale"]), dsc_ref)
    dx_s, _, dsc_s = oracle.adaln_bwd(dy, x, sc, seg, c["eps"], mean=mean.cpu().numpy(),
                                      rstd=rstd.cpu().numpy())
    H.check_rowwise("dx", dt, H.to_f64(out["dx"]), dx_s)
    H.check_norm("dscale", dt, H.to_f64(out["dscale"]), dsc_s)


def test_noalloc_matches_oracle_and_adaln_bwd_on_two_calls(adaln):
    L = adaln
    L.adaln_get_status()  # clear
    cases = [I.random_case(101, 5000, 3072, 40, dtype="bf16"),   # many segments
             I.random_case(102, 9001, 1536, 2, dtype="bf16", lengths=[4000, 5001])]
    for c in cases:
        d = H.device_inputs(c)
        T, D, nseg = c["T"], c["D"], c["nseg"]
        dtype = torch.bfloat16
        y, mean, rstd = L.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], c["eps"])
        new = _noalloc(L, d, mean, rstd, dtype, T, D, nseg)
        _check_oracle(c, d, new, mean, rstd)
        ref = L.adaln_bwd(d["dy"], d["x"], mean, rstd, d["scale"], d["seg_id"])
        torch.cuda.synchronize()
        for k, r in zip(("dx", "dshift", "dscale"), ref):
            assert torch.equal(new[k], r), k
    rc, bits = L.adaln_get_status()
    assert rc == L.ADALN_OK and bits == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(adaln):
    L = adaln
    T, D, nseg = 200000, 8192, 4000
    need = L.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16)
    assert need > L.NOALLOC_SCRATCH_BYTES
    # Rejected before any pointer is used or anything is launched.
    rc = L.raw.adaln_bwd_noalloc(None, None, None, None, None, None, T, D, nseg,
                                 L.ADALN_BF16, None, None, None, None)
    assert rc == L.ADALN_ERR_WORKSPACE
