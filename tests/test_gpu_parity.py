"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Workloads 1-2 are compared on every element; workloads 3-5 (full size, in the
launch configuration the benchmark uses) on rows sampled at every CTA range
boundary plus random rows, and on all of dscale/dshift.  Edge cases: empty
input, single rows, T below the grid size, ragged tails, minimum and maximum
D, every vectors-per-thread variant, empty and one-row segments, many
segments.  Segment indexing is checked bit-exactly.
"""
import numpy as np
import pytest
import torch

import gpu_helpers as H
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(adaln):
    adaln.adaln_get_status()  # clear
    yield
    H.status_ok()


@pytest.mark.parametrize("config", [1, 2])
def test_workload_full_parity(adaln, config):
    c = I.make(config)
    d = H.device_inputs(c)
    out = H.run_gpu(d, c["eps"])
    H.check_against_oracle(c, d, out)


@pytest.mark.parametrize("config", [3, 4])
def test_workload_full_size_sampled_parity(adaln, config):
    c = I.make(config)
    d = H.device_inputs(c)
    out = H.run_gpu(d, c["eps"])
    rows = np.union1d(*[H.sample_rows(c["T"], adaln.adaln_launch_shape(
        k, c["T"], c["D"], c["nseg"], adaln.ADALN_BF16)["grid"])
        for k in (adaln.ADALN_KERNEL_BWD_ROWS, adaln.ADALN_KERNEL_FWD)])
    H.check_against_oracle(c, d, out, rows=rows)


def test_mmdit_joint_sites(adaln):
    c = I.make(5, sites=3)
    x, dy, seg = H.to_dev(c["x"]), H.to_dev(c["dy"]), H.to_dev(c["seg_id"])
    rows = H.sample_rows(c["T"], 152, n_random=256)
    for site in (0, 2):
        d = dict(x=x, dy=dy, seg_id=seg, shift=H.to_dev(c["shift"][site]),
                 scale=H.to_dev(c["scale"][site]), shift_np=c["shift"][site],
                 scale_np=c["scale"][site])
        out = H.run_gpu(d, c["eps"])
        H.check_against_oracle(c, d, out, rows=rows)


EDGE = [
    # (T, D, nseg, dtype, lengths); nvec = 16-byte vectors per row
    (1, 64, 1, "bf16", None),
    (3, 5120, 2, "bf16", [1, 2]),   # fewer rows than backward teams on the GPU
    (1, 4, 1, "f32", None),
    (7, 8, 3, "bf16", [0, 7, 0]),          # T below the grid; empty first/last segment
    (1001, 136, 5, "bf16", None),          # ragged: odd T, nvec = 17
    (999, 24, 4, "f32", [1, 1, 1, 996]),   # one-row segments, nvec = 6
    (300, 1536, 2, "bf16", None),          # nvec 192: variants 5/6 (VPT 2), 3 warps
    (300, 1528, 2, "bf16", None),          # nvec 191: variants 5/6, ragged last vector
    (300, 1544, 2, "bf16", None),          # nvec 193: variant 4 (VPT 4), 2 warps, ragged
    (600, 512, 3, "bf16", None),           # nvec 64: 1-warp teams, 8 forward / 6 backward
    (600, 1024, 3, "bf16", None),          # nvec 128: 2-warp teams, 5 forward / 4 backward
    (600, 2048, 3, "bf16", None),          # nvec 256: variant 4, 2-warp teams, 4 per CTA
    (300, 3064, 3, "bf16", None),          # nvec 383: variant 4, 3 warps, ragged
    (300, 3072, 3, "bf16", None),          # nvec 384: variant 1 forward, 6 warps
    (300, 3080, 3, "bf16", None),          # nvec 385: variant 2 (VPT 4), 4 warps, ragged
    (260, 5120, 3, "bf16", None),          # nvec 640: variant 2, 5 warps
    (260, 5128, 3, "bf16", None),          # nvec 641: variant 3 (VPT 4), 6 warps, ragged
    (200, 8192, 2, "bf16", None),          # nvec 1024: largest bf16 row, 8 warps
    (200, 4096, 2, "f32", None),           # largest fp32 row
    (200, 1540, 2, "f32", None),           # fp32 nvec 385: variant 2, ragged
    (2048, 1536, 2048, "bf16", [1] * 2048),  # every row its own segment
    (3000, 256, 700, "bf16", None),        # many segments, many empty
    (4099, 512, 1, "bf16", None),          # one segment across every CTA
]


@pytest.mark.parametrize("T,D,nseg,dtype,lengths", EDGE,
                         ids=[f"T{e[0]}_D{e[1]}_n{e[2]}_{e[3]}" for e in EDGE])
def test_edge_shapes(adaln, T, D, nseg, dtype, lengths):
    c = I.random_case(T * 31 + D, T, D, nseg, dtype=dtype, lengths=lengths, dy_std=1.0)
    d = H.device_inputs(c)
    out = H.run_gpu(d, c["eps"])
    H.check_against_oracle(c, d, out)


def test_empty_input_zeroes_modulation_grads(adaln):
    dev = "cuda"
    x = torch.empty(0, 64, device=dev, dtype=torch.bfloat16)
    sh = torch.zeros(3, 64, device=dev, dtype=torch.bfloat16)
    seg = torch.empty(0, device=dev, dtype=torch.int32)
    y, m, r = adaln.adaln_fwd(x, sh, sh, seg, 1e-6)
    assert y.shape == (0, 64)
    dsh = torch.full((3, 64), float("nan"), device=dev)
    dsc = torch.full((3, 64), float("nan"), device=dev)
    adaln.adaln_bwd(x, x, m, r, sh, seg, dshift=dsh, dscale=dsc)
    torch.cuda.synchronize()
    assert torch.all(dsh == 0) and torch.all(dsc == 0)


def test_segment_indexing_bit_exact(adaln):
    """Constant rows give xhat = 0 exactly, so y = shift[seg_id] bit for bit;
    with dy = 1, dshift[b] is exactly the segment length."""
    lengths = [5, 0, 130, 1, 64, 0, 300, 12]
    nseg, T, D = len(lengths), sum(lengths), 64
    seg = I.seg_ids_from_lengths(lengths)
    dev = "cuda"
    for tdt in (torch.bfloat16, torch.float32):
        x = torch.full((T, D), 0.5, device=dev, dtype=tdt)
        scale = torch.zeros(nseg, D, device=dev, dtype=tdt)
        shift = (torch.arange(nseg, device=dev, dtype=torch.float32) + 1)[:, None].expand(nseg, D)
        shift = shift.contiguous().to(tdt)
        segd = torch.from_numpy(seg).to(dev)
        y, m, r = adaln.adaln_fwd(x, shift, scale, segd, 1e-6)
        want = torch.from_numpy(seg.astype(np.float32) + 1).to(dev)[:, None].expand(T, D).to(tdt)
        assert torch.equal(y, want)
        dy = torch.ones(T, D, device=dev, dtype=tdt)
        dx, dsh, dsc = adaln.adaln_bwd(dy, x, m, r, scale, segd)
        want_sh = torch.tensor(lengths, device=dev, dtype=torch.float32)[:, None].expand(nseg, D)
        assert torch.equal(dsh, want_sh)
        assert torch.equal(dsc, torch.zeros_like(dsc))


def _guarded(shape, dtype, fill, dev="cuda", pad=4096):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, device=dev, dtype=dtype)
    return buf, buf[pad:pad + n].view(*shape), pad


def test_guard_bands_untouched(adaln):
    """Outputs and workspace sit inside canary-filled buffers; nothing outside
    the stated extents is written."""
    c = I.random_case(77, 777, 1040, 9, dtype="bf16")
    d = H.device_inputs(c)
    T, D, nseg = c["T"], c["D"], c["nseg"]
    bufs = {}
    bufs["y"] = _guarded((T, D), torch.bfloat16, 7.0)
    bufs["dx"] = _guarded((T, D), torch.bfloat16, 7.0)
    bufs["mean"] = _guarded((T,), torch.float32, 7.0)
    bufs["rstd"] = _guarded((T,), torch.float32, 7.0)
    bufs["dshift"] = _guarded((nseg, D), torch.float32, 7.0)
    bufs["dscale"] = _guarded((nseg, D), torch.float32, 7.0)
    ws_bytes = adaln.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16)
    bufs["ws"] = _guarded((ws_bytes,), torch.uint8, 0xA5)
    adaln.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], c["eps"],
                    y=bufs["y"][1], mean=bufs["mean"][1], rstd=bufs["rstd"][1])
    adaln.adaln_bwd(d["dy"], d["x"], bufs["mean"][1], bufs["rstd"][1], d["scale"], d["seg_id"],
                    dx=bufs["dx"][1], dshift=bufs["dshift"][1], dscale=bufs["dscale"][1],
                    workspace=bufs["ws"][1])
    torch.cuda.synchronize()
    for k, (buf, _, pad) in bufs.items():
        fill = 0xA5 if k == "ws" else 7.0
        assert torch.all(buf[:pad] == fill), k
        assert torch.all(buf[-pad:] == fill), k
    out = {k: bufs[k][1] for k in ("y", "dx", "mean", "rstd", "dshift", "dscale")}
    H.check_against_oracle(c, d, out)


def test_backward_is_bitwise_deterministic(adaln):
    c = I.make(2)
    d = H.device_inputs(c)
    a = H.run_gpu(d, c["eps"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        junk = torch.randn(1 << 24, device="cuda")  # shift the stream position
        b = H.run_gpu(d, c["eps"], stream=s)
        del junk
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_bad_segment_ids_set_status_and_stay_in_bounds(adaln):
    dev = "cuda"
    T, D, nseg = 600, 256, 4
    x = torch.randn(T, D, device=dev).to(torch.bfloat16)
    sh = torch.randn(nseg, D, device=dev).to(torch.bfloat16)
    for bad, bit in ((np.r_[np.zeros(300), np.ones(300) * 9], adaln.ADALN_DEV_SEG_RANGE),
                     (np.r_[np.ones(300) * 2, np.zeros(300)], adaln.ADALN_DEV_SEG_ORDER),
                     (np.r_[np.zeros(300), -np.ones(300)], adaln.ADALN_DEV_SEG_RANGE)):
        seg = torch.from_numpy(bad.astype(np.int32)).to(dev)
        y_buf, y, _ = _guarded((T, D), torch.bfloat16, 3.0)
        y, m, r = adaln.adaln_fwd(x, sh, sh, seg, 1e-6, y=y)
        rc, bits = adaln.adaln_get_status()
        assert rc == adaln.ADALN_ERR_SEG and bits & bit, (rc, bits)
        ws_bytes = adaln.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16)
        ws_buf, ws, _ = _guarded((ws_bytes,), torch.uint8, 0x5A)
        dsh_buf, dsh, _ = _guarded((nseg, D), torch.float32, 3.0)
        adaln.adaln_bwd(x, x, m, r, sh, seg, dshift=dsh, workspace=ws)
        rc, bits = adaln.adaln_get_status()
        assert rc == adaln.ADALN_ERR_SEG and bits & bit, (rc, bits)
        for buf, f in ((y_buf, 3.0), (ws_buf, 0x5A), (dsh_buf, 3.0)):
            assert torch.all(buf[:4096] == f) and torch.all(buf[-4096:] == f)


def test_workspace_and_alignment_errors(adaln):
    dev = "cuda"
    T, D, nseg = 64, 64, 1
    x = torch.randn(T, D, device=dev).to(torch.bfloat16)
    sh = torch.zeros(nseg, D, device=dev, dtype=torch.bfloat16)
    seg = torch.zeros(T, device=dev, dtype=torch.int32)
    y, m, r = adaln.adaln_fwd(x, sh, sh, seg, 1e-6)
    need = adaln.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16)
    small = torch.empty(need - 256, device=dev, dtype=torch.uint8)  # sizes round up by < 256
    with pytest.raises(adaln.AdalnError) as e:
        adaln.adaln_bwd(x, x, m, r, sh, seg, workspace=small)
    assert e.value.code == adaln.ADALN_ERR_WORKSPACE
    flat = torch.empty(T * D + 8, device=dev, dtype=torch.bfloat16)
    mis = flat[1:1 + T * D].view(T, D)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(adaln.AdalnError) as e:
        adaln.adaln_fwd(mis, sh, sh, seg, 1e-6)
    assert e.value.code == adaln.ADALN_ERR_ALIGN


def test_trace_counts_launches(adaln):
    c = I.random_case(5, 500, 512, 2, dtype="bf16")
    d = H.device_inputs(c)
    adaln.adaln_trace_begin(16)
    for _ in range(3):
        H.run_gpu(d, c["eps"])
    adaln.adaln_trace_end()
    for k in range(3):
        n, ms = adaln.adaln_trace_get(k)
        assert n == 3 and ms > 0.0, (k, n, ms)


def test_launch_shape_matches_the_rules(adaln):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # D = 5120 bf16: 640 vectors, 4 per thread -> teams of 5 consumer warps +
    # 1 producer, two teams per CTA, one CTA per SM.
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_BWD_ROWS, 32760, 5120, 1, torch.bfloat16)
    assert s["threads"] == 2 * 6 * 32 and s["grid"] == sms and s["stages"] >= 2
    # Every backward team owns rows: fewer CTAs, then one team, for tiny T.
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_BWD_ROWS, 7, 5120, 1, torch.bfloat16)
    assert s["grid"] == 3 and s["threads"] == 2 * 6 * 32
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_BWD_ROWS, 1, 5120, 1, torch.bfloat16)
    assert s["grid"] == 1 and s["threads"] == 6 * 32
    # D = 1536 bf16: 192 vectors, 2 per thread -> 3 consumer warps; the
    # forward runs one CTA per SM with four teams of 3 + 1 warps.
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_FWD, 8192, 1536, 2, torch.bfloat16)
    assert s["threads"] == 4 * 4 * 32 and s["grid"] == sms
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_FWD, 5, 5120, 1, torch.bfloat16)
    assert s["grid"] == 5
    # Rows that need fewer warps run more teams in the variant's thread
    # budget: D = 1024 bf16 (128 vectors, 2 warps a team) gets five forward
    # teams of 2 + 1 warps and four backward ones; D = 2048 bf16 (256
    # vectors, 4 per thread) four teams of 2 + 1 warps both ways.
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_FWD, 32768, 1024, 4, torch.bfloat16)
    assert s["threads"] == 5 * 3 * 32
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_BWD_ROWS, 32768, 1024, 4, torch.bfloat16)
    assert s["threads"] == 4 * 3 * 32
    for which in (adaln.ADALN_KERNEL_FWD, adaln.ADALN_KERNEL_BWD_ROWS):
        s = adaln.adaln_launch_shape(which, 32768, 2048, 4, torch.bfloat16)
        assert s["threads"] == 4 * 3 * 32 and s["grid"] == sms
    # D = 3072 bf16 (384 vectors): the forward runs three teams of 3 + 1 warps
    # when segments are long, two of 6 + 1 when they are short.
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_FWD, 36864, 3072, 16, torch.bfloat16)
    assert s["threads"] == 3 * 4 * 32
    s = adaln.adaln_launch_shape(adaln.ADALN_KERNEL_FWD, 36864, 3072, 64, torch.bfloat16)
    assert s["threads"] == 2 * 7 * 32


def test_cuda_graph_capture_matches_eager(adaln):
    """fwd + bwd (three launches, the finalize a programmatic dependent)
    captured into a CUDA graph and replayed give bitwise the eager results."""
    c = I.random_case(31, 3000, 2048, 5, dtype="bf16")
    d = H.device_inputs(c)
    ref = H.run_gpu(d, c["eps"])
    T, D, nseg = c["T"], c["D"], c["nseg"]
    out = {k: torch.empty_like(v) for k, v in ref.items()}
    ws = torch.empty(adaln.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16), device="cuda",
                     dtype=torch.uint8)

    def step(stream):
        adaln.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], c["eps"], y=out["y"],
                        mean=out["mean"], rstd=out["rstd"], stream=stream)
        adaln.adaln_bwd(d["dy"], d["x"], out["mean"], out["rstd"], d["scale"], d["seg_id"],
                        dx=out["dx"], dshift=out["dshift"], dscale=out["dscale"], workspace=ws,
                        stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)  # warm the launch-shape cache outside capture
        g = torch.cuda.CUDAGraph()
        g.capture_begin()
        step(s)
        g.capture_end()
    torch.cuda.current_stream().wait_stream(s)
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(out[k], ref[k]), k



@pytest.mark.parametrize("T,D,nseg", [(20000, 3072, 3), (300, 1024, 5)])
def test_inputs_written_by_the_previous_kernel_are_read_after_it(adaln, T, D, nseg):
    """The row kernels are launched as programmatic dependents of the
    stream's previous kernel: inputs that a torch kernel writes just before
    each call (no synchronisation in between) must be read only after it
    has completed, seg_id included (the finalize reads it before waiting for
    the row pass; with few rows it has SMs to itself early).  The buffers
    hold other, valid data until those kernels run."""
    c = I.random_case(77 + T, T, D, nseg, dtype="bf16")
    d = H.device_inputs(c)
    x = torch.full_like(d["x"], 7.0)
    dy = torch.full_like(d["dy"], -3.0)
    seg = torch.zeros_like(d["seg_id"])  # every row in segment 0
    y = torch.empty_like(x)
    mean = torch.empty(T, device="cuda")
    rstd = torch.empty(T, device="cuda")
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6))  # keep the GPU busy so the launches queue up
    x.copy_(d["x"])              # the previous kernel writes x ...
    adaln.adaln_fwd(x, d["shift"], d["scale"], d["seg_id"], c["eps"], y=y, mean=mean, rstd=rstd)
    dy.copy_(d["dy"])            # ... dy
    seg.copy_(d["seg_id"])       # ... and seg_id
    dx, dsh, dsc = adaln.adaln_bwd(dy, x, mean, rstd, d["scale"], seg)
    torch.cuda.synchronize()
    H.check_against_oracle(c, d, dict(y=y, mean=mean, rstd=rstd, dx=dx, dshift=dsh, dscale=dsc))


def test_bound_status_words_keep_callers_apart(adaln):
    """Two host threads, each with its own bound status word: the thread
    whose call has a decreasing seg_id sees the order bit, the other thread
    and the device's shared word see nothing."""
    import threading
    dev = "cuda"
    T, D, nseg = 600, 256, 4
    x = torch.randn(T, D, device=dev).to(torch.bfloat16)
    sh = torch.randn(nseg, D, device=dev).to(torch.bfloat16)
    good = torch.from_numpy(np.repeat(np.arange(nseg), T // nseg).astype(np.int32)).to(dev)
    bad = torch.from_numpy(np.r_[np.ones(300) * 2, np.zeros(300)].astype(np.int32)).to(dev)
    words = {k: torch.zeros(1, device=dev, dtype=torch.int32) for k in ("good", "bad")}
    results = {}

    def worker(name, seg):
        s = torch.cuda.Stream()
        adaln.adaln_status_bind(words[name])
        try:
            with torch.cuda.stream(s):
                y, m, r = adaln.adaln_fwd(x, sh, sh, seg, 1e-6, stream=s)
                adaln.adaln_bwd(x, x, m, r, sh, seg, stream=s)
            results[name] = adaln.adaln_get_status(stream=s)
        finally:
            adaln.adaln_status_bind(None)

    threads = [threading.Thread(target=worker, args=(n, sg)) for n, sg in (("good", good),
                                                                          ("bad", bad))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert results["good"] == (adaln.ADALN_OK, 0)
    rc, bits = results["bad"]
    assert rc == adaln.ADALN_ERR_SEG and bits & adaln.ADALN_DEV_SEG_ORDER
    assert adaln.adaln_get_status() == (adaln.ADALN_OK, 0)  # the shared word stayed clean
    assert int(words["good"].item()) == 0 and int(words["bad"].item()) == 0  # read and cleared
