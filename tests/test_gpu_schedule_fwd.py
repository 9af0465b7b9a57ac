"""Forward work distribution: the teams of a CTA share its rows, or all teams
share all rows through a device-wide counter slot.  Per-row results must not
depend on which team computes a row, counter slots must be reset and reused
across launches, and concurrent launches on several streams must not share
a slot."""
import os

import numpy as np
import pytest
import torch

import gpu_helpers as H
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _fwd(adaln, d, eps, stream=None, out=None):
    kw = {} if out is None else dict(y=out["y"], mean=out["mean"], rstd=out["rstd"])
    return adaln.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], eps, stream=stream, **kw)


@pytest.fixture
def sched(monkeypatch):
    def set_mode(mode):
        if mode is None:
            monkeypatch.delenv("ADALN_FWD_SCHED", raising=False)
        else:
            monkeypatch.setenv("ADALN_FWD_SCHED", mode)
    yield set_mode
    monkeypatch.delenv("ADALN_FWD_SCHED", raising=False)


@pytest.mark.parametrize("T,D,nseg,dtype", [(20000, 5120, 1, "bf16"), (9000, 1536, 3, "bf16"),
                                            (7001, 3072, 40, "bf16"), (5003, 1024, 2, "f32")])
def test_modes_give_identical_rows(adaln, sched, T, D, nseg, dtype):
    c = I.random_case(T + D, T, D, nseg, dtype=dtype)
    d = H.device_inputs(c)
    outs = {}
    for mode in ("cta", "device", None):
        sched(mode)
        outs[mode] = [t.clone() for t in _fwd(adaln, d, c["eps"])]
        torch.cuda.synchronize()
    H.status_ok()
    for mode in ("device", None):
        for a, b in zip(outs[mode], outs["cta"]):
            assert torch.equal(a, b), mode
    rows = H.sample_rows(T, 152, n_random=64)
    y_ref, m_ref, r_ref = H.oracle.adaln_fwd(c["x"], d["shift_np"], d["scale_np"], c["seg_id"],
                                             c["eps"], rows=rows)
    idx = torch.from_numpy(rows).cuda()
    H.check_rowwise("y", dtype, H.to_f64(outs["device"][0][idx]), y_ref)


def test_counter_slots_are_reused(adaln, sched):
    """More launches than counter slots, alternating sizes: every launch must
    see its slot zeroed by the previous user."""
    sched("device")
    c = I.random_case(5, 6000, 2048, 1, dtype="bf16")
    d = H.device_inputs(c)
    ref = [t.clone() for t in _fwd(adaln, d, c["eps"])]
    small = {k: (v[:2500] if k in ("x", "seg_id") else v) for k, v in d.items()}
    ref_small = [t.clone() for t in _fwd(adaln, small, c["eps"])]
    out = {k: torch.empty_like(v) for k, v in zip(("y", "mean", "rstd"), ref)}
    out_s = {k: torch.empty_like(v) for k, v in zip(("y", "mean", "rstd"), ref_small)}
    for i in range(600):
        _fwd(adaln, d, c["eps"], out=out)
        _fwd(adaln, small, c["eps"], out=out_s)
        if i % 150 == 149:
            torch.cuda.synchronize()
            assert torch.equal(out["y"], ref[0]) and torch.equal(out_s["y"], ref_small[0])
    torch.cuda.synchronize()
    H.status_ok()


def test_concurrent_streams(adaln, sched):
    """Launches in flight at once on four streams, each with its own inputs
    and outputs, give the results of sequential launches."""
    sched("device")
    cases = [I.random_case(40 + i, 8000 + 1000 * i, 4096, 1, dtype="bf16") for i in range(4)]
    ds = [H.device_inputs(c) for c in cases]
    refs = [[t.clone() for t in _fwd(adaln, d, c["eps"])] for c, d in zip(cases, ds)]
    outs = [{k: torch.empty_like(v) for k, v in zip(("y", "mean", "rstd"), r)} for r in refs]
    streams = [torch.cuda.Stream() for _ in ds]
    torch.cuda.synchronize()
    for rep in range(20):
        for c, d, o, s in zip(cases, ds, outs, streams):
            _fwd(adaln, d, c["eps"], stream=s, out=o)
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o["y"], r[0]) and torch.equal(o["mean"], r[1])
    H.status_ok()


def test_graph_capture_uses_cta_local_units(adaln, sched):
    """A long-segment forward (device-wide units when launched eagerly) captured
    into a CUDA graph runs with CTA-local units and gives the same bits."""
    sched(None)
    c = I.random_case(77, 24000, 5120, 1, dtype="bf16")
    d = H.device_inputs(c)
    ref = [t.clone() for t in _fwd(adaln, d, c["eps"])]
    out = {k: torch.empty_like(v) for k, v in zip(("y", "mean", "rstd"), ref)}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fwd(adaln, d, c["eps"], stream=s, out=out)
        g = torch.cuda.CUDAGraph()
        g.capture_begin()
        _fwd(adaln, d, c["eps"], stream=s, out=out)
        g.capture_end()
    torch.cuda.current_stream().wait_stream(s)
    for k in out:
        out[k].zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out["y"], ref[0]) and torch.equal(out["rstd"], ref[2])
    H.status_ok()
