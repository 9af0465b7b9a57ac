"""Pipelined forward + backward on host-resident tensors (adaln_fwd_bwd_host)
against the device path: per-row outputs bit for bit, the chunk-summed
modulation gradients within the oracle tolerance."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _host_tensors(c):
    def h(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) \
            if a.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory()
    return {k: h(c[k]) for k in ("x", "dy", "shift", "scale", "seg_id")}


CASES = [
    # (T, D, nseg, dtype, lengths, chunk_rows)
    (5000, 1024, 7, "bf16", None, 1024),     # ramped chunk plan; chunks split segments
    (100, 256, 40, "bf16", None, 8),         # ramp of 1, 2, 4 rows; many short segments
    (300, 1536, 2, "bf16", [120, 180], 1000),  # one chunk, T below the chunk size
    (2049, 512, 3, "f32", [0, 2049, 0], 256),  # fp32, empty first/last segments
    (0, 256, 2, "bf16", [0, 0], 64),           # no rows: gradients are zero
    (6000, 3072, 2, "bf16", None, 1000),     # the forward's shape follows the batch's
                                             # rows per segment, not a chunk's
]


@pytest.mark.parametrize("T,D,nseg,dtype,lengths,chunk", CASES,
                         ids=[f"T{c[0]}_D{c[1]}_{c[3]}_c{c[5]}" for c in CASES])
def test_host_pipeline_matches_device_path(adaln, T, D, nseg, dtype, lengths, chunk):
    c = I.random_case(T + D + chunk, T, D, nseg, dtype=dtype, lengths=lengths, dy_std=1.0)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    h = _host_tensors(c)
    out = dict(y=torch.empty(T, D, dtype=tdt).pin_memory(),
               dx=torch.empty(T, D, dtype=tdt).pin_memory(),
               mean=torch.empty(T).pin_memory(), rstd=torch.empty(T).pin_memory(),
               dshift=torch.full((nseg, D), float("nan")).pin_memory(),
               dscale=torch.full((nseg, D), float("nan")).pin_memory())
    scratch = torch.empty(adaln.adaln_fwd_bwd_host_scratch_size(T, D, nseg, tdt, chunk),
                          device="cuda", dtype=torch.uint8)
    for _ in range(2):  # a second call on the same scratch
        adaln.adaln_fwd_bwd_host(h["x"], h["dy"], h["shift"], h["scale"], h["seg_id"], c["eps"],
                                 out, scratch, chunk_rows=chunk)
        torch.cuda.synchronize()
    H.status_ok()
    if T == 0:
        assert torch.all(out["dshift"] == 0) and torch.all(out["dscale"] == 0)
        return
    d = H.device_inputs(c)
    ref = H.run_gpu(d, c["eps"])
    for k in ("y", "dx", "mean", "rstd"):
        assert torch.equal(out[k], ref[k].cpu()), k
    for k in ("dshift", "dscale"):
        a, b = H.to_f64(out[k]), H.to_f64(ref[k])
        assert H.normwise(a, b) < 1e-5, k
    _, dsh_ref, dsc_ref = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"],
                                           want_dx=False)
    H.check_norm("dshift", dtype, H.to_f64(out["dshift"]), dsh_ref)
    H.check_norm("dscale", dtype, H.to_f64(out["dscale"]), dsc_ref)


def test_host_pipeline_from_two_threads(adaln):
    """Two host threads run the pipelined step at once, each with its own
    buffers and scratch: the calls are serialised on the device's internal
    streams and both give the device path's results."""
    import threading
    cases = [I.random_case(900 + i, 3000 + 500 * i, 2048, 3, dtype="bf16", dy_std=1.0)
             for i in range(2)]
    refs, jobs = [], []
    for c in cases:
        T, D, nseg = c["T"], c["D"], c["nseg"]
        refs.append(H.run_gpu(H.device_inputs(c), c["eps"]))
        h = _host_tensors(c)
        out = dict(y=torch.empty(T, D, dtype=torch.bfloat16).pin_memory(),
                   dx=torch.empty(T, D, dtype=torch.bfloat16).pin_memory(),
                   mean=torch.empty(T).pin_memory(), rstd=torch.empty(T).pin_memory(),
                   dshift=torch.empty(nseg, D).pin_memory(),
                   dscale=torch.empty(nseg, D).pin_memory())
        scratch = torch.empty(adaln.adaln_fwd_bwd_host_scratch_size(T, D, nseg, torch.bfloat16, 512),
                              device="cuda", dtype=torch.uint8)
        jobs.append((c, h, out, scratch))
    torch.cuda.synchronize()
    errors = []

    def work(c, h, out, scratch):
        try:
            s = torch.cuda.Stream()
            for _ in range(5):
                adaln.adaln_fwd_bwd_host(h["x"], h["dy"], h["shift"], h["scale"], h["seg_id"],
                                         c["eps"], out, scratch, chunk_rows=512, stream=s)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=j) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (c, h, out, scratch), ref in zip(jobs, refs):
        for k in ("y", "dx", "mean", "rstd"):
            assert torch.equal(out[k], ref[k].cpu()), k
        assert H.normwise(H.to_f64(out["dshift"]), H.to_f64(ref["dshift"])) < 1e-5
    H.status_ok()
