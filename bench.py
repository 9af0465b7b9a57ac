"""Benchmark of the fused AdaLN forward + backward on GB300.

A step is one pass of the whole hot path over one batch: adaln_fwd (row
statistics + modulation) then adaln_bwd (dx, and the sequence reductions
dscale/dshift with their finalize), through the C ABI of libadaln.so.  The
default workload is the long-video bucket: T = 32760 tokens (21 x 30 x 52
latent patches), D = 5120, bf16, one modulation segment.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (plain
fp64 C++) on the host cores instead, on a bounded sample of the same workload.
With N > 1 (torchrun) every rank runs an independent replica on its own GPU:
the operator has no exchange step, so there is no collective on the data path.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("fused AdaLN fwd+bwd tokens/s and achieved HBM GB/s (% of peak) "
          "at D=5120 bf16")
WORKLOADS = {"tiny_fp32": 1, "wan13b": 2, "long_video": 3, "mixed_varlen": 4,
             "mmdit_joint": 5}
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="long_video", choices=sorted(WORKLOADS))
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--e2e-chunk", type=int, default=0,
                   help="rows per pipelined chunk of the e2e leg (0: the library default)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--rows", type=int, default=0,
                   help="only the first ROWS tokens of the workload (a smaller case of the "
                        "same structure, for profiler captures); 0 = all")
    p.add_argument("--sites", type=int, default=1,
                   help="modulation sites per step (mmdit_joint steady state: 60 = 2 per "
                        "block x 30 blocks), each its own shift/scale, back to back")
    p.add_argument("--graph", action="store_true",
                   help="with --sites: replay each step as one captured CUDA graph")
    p.add_argument("--report", choices=["unfused", "shapes", "fixed-cost", "widths"],
                   default=None,
                   help="instead of the benchmark line: compare with torch's unfused "
                        "chain (time and saved activation bytes), shape-benchmark the "
                        "operator and fit the step-time cost model, split a call's "
                        "fixed cost into host and GPU time, or time the forward and "
                        "backward over a grid of row widths of both dtypes")
    return p.parse_args()


# ---------------------------------------------------------------------------
# Algorithmic bytes (what the operator must move; partial-sum workspace and
# any re-reads excluded).  s = element size, per token and per segment.
# ---------------------------------------------------------------------------
def alg_bytes(T, D, nseg, esize):
    fwd = T * (2 * D * esize + 4 + 8) + 2 * nseg * D * esize
    bwd_rows = T * (3 * D * esize + 4 + 8) + nseg * D * esize
    bwd = bwd_rows + 2 * nseg * D * 4
    return dict(fwd=fwd, bwd=bwd, bwd_rows=bwd_rows, fwd_bwd=fwd + bwd)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Clock record.  A thread samples the SM clock, the clock-event (throttle)
# reasons and the power draw every ~1 ms through NVML (read-only queries,
# libnvidia-ml via ctypes), or every 100 ms through nvidia-smi when NVML is
# not loadable.  The main thread marks host-time windows (the timed loop, the
# trace pass, the e2e leg); samples inside them are "under load".
# ---------------------------------------------------------------------------
REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
SMI_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class _Nvml:
    """Minimal read-only NVML binding (clock, max clock, event reasons, power)."""

    def __init__(self, pci_bus_id=None, uuid=None, index=None):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
        if rc != 0 and uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        if rc != 0 and index is not None:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(int(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        mhz, mx, mw = ct.c_uint(0), ct.c_uint(0), ct.c_uint(0)
        bits = ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.reasons_fn(self.h, ct.byref(bits))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        names = [n for b, n in REASON_BITS.items() if bits.value & b]
        return float(mhz.value), float(mx.value), names, mw.value / 1000.0

    def close(self):
        self.lib.nvmlShutdown()


def parse_smi_line(line):
    """(sm_mhz, sm_max_mhz, reasons, power_w) from one nvidia-smi CSV line, or None."""
    f = [x.strip() for x in line.split(",")]
    if len(f) < 9:
        return None
    try:
        sm, smax = float(f[1]), float(f[2])
    except ValueError:
        return None
    try:
        pw = float(f[3])
    except ValueError:
        pw = None
    return sm, smax, [n for n, v in zip(SMI_REASONS, f[5:9]) if v.lower() == "active"], pw


class ClockRecord:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_ids=None, period_s=0.001):
        self.ids = dev_ids or {}
        self.period = period_s
        self.samples = []   # (host time, sm_mhz, sm_max_mhz, reasons, power_w)
        self.windows = []   # (name, t0, t1)
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    # -- sampling ------------------------------------------------------------
    def start(self):
        try:
            nv = _Nvml(self.ids.get("pci_bus_id"), self.ids.get("uuid"), self.ids.get("index"))
        except (OSError, AttributeError):
            nv = None
        if nv is not None:
            self.source = "nvml"
            self._thread = threading.Thread(target=self._nvml_loop, args=(nv,), daemon=True)
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.ids.get("smi", 0)), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                return self
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._smi_loop, daemon=True)
        self._thread.start()
        return self

    def _nvml_loop(self, nv):
        try:
            while not self._stop.is_set():
                v = nv.sample()
                if v is not None:
                    self.samples.append((time.perf_counter(),) + v)
                time.sleep(self.period)
        finally:
            nv.close()

    def _smi_loop(self):
        for line in self._proc.stdout:
            v = parse_smi_line(line)
            if v is not None:
                self.samples.append((time.perf_counter(),) + v)

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    # -- windows ------------------------------------------------------------
    def window(self, name):
        rec = self

        class _W:
            def __enter__(self_):
                self_.t0 = time.perf_counter()

            def __exit__(self_, *exc):
                rec.windows.append((name, self_.t0, time.perf_counter()))
        return _W()

    def summary(self):
        def inside(t, names=None):
            return any(a <= t <= b for n, a, b in self.windows if names is None or n in names)
        load = [s_ for s_ in self.samples if inside(s_[0])]
        out = {"source": self.source, "samples": len(self.samples),
               "samples_under_load": len(load),
               "samples_by_window": {n: sum(1 for s_ in self.samples if inside(s_[0], (n,)))
                                     for n in dict.fromkeys(w[0] for w in self.windows)}}
        use = load or self.samples
        if not use:
            out.update(sm_mhz=None, sm_max_mhz=None, reasons=[], power_w_max=None)
            return out
        reasons = sorted({r for s_ in use for r in s_[3]})
        pw = [s_[4] for s_ in use if s_[4] is not None]
        out.update(sm_mhz=statistics.median(s_[1] for s_ in use),
                   sm_mhz_min=min(s_[1] for s_ in use),
                   sm_max_mhz=max(s_[2] for s_ in use), reasons=reasons,
                   power_w_max=max(pw) if pw else None)
        return out


def device_ids(dev, local):
    """Identifiers NVML can find the torch device by (PCI bus id, UUID, index)."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    ids = {"smi": gpu_smi_id(local)}
    try:
        ids["pci_bus_id"] = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        pass
    u = str(getattr(p, "uuid", "") or "")
    if u:
        ids["uuid"] = u if u.startswith("GPU-") else "GPU-" + u
    if ids["smi"].isdigit():
        ids["index"] = int(ids["smi"])
    return ids


# ---------------------------------------------------------------------------
# Process group (one rank per GPU under torchrun; replicas, no data exchange).
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend, rank=rank, world_size=world)
        pg = dist
    return rank, local, world, pg


def barrier(pg, dev):
    if pg is not None:
        if pg.get_backend() == "nccl":
            pg.barrier(device_ids=[dev.index])
        else:
            pg.barrier()


def max_over_ranks(pg, value, dev):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=dev if pg.get_backend() == "nccl" else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# Inputs.
# ---------------------------------------------------------------------------
def host_inputs(name, rows=0):
    """The workload's seeded inputs (one modulation site); with rows > 0 only
    its first `rows` tokens and the segments they touch (a smaller case of
    the same structure, e.g. for profiler captures)."""
    from adaln_video_dit_gb300 import inputs as I
    c = I.make(WORKLOADS[name])
    if isinstance(c["shift"], list):
        c["shift"], c["scale"] = c["shift"][0], c["scale"][0]
    if 0 < rows < c["T"]:
        nseg = int(c["seg_id"][rows - 1]) + 1
        c.update(x=c["x"][:rows], dy=c["dy"][:rows], seg_id=c["seg_id"][:rows],
                 shift=c["shift"][:nseg], scale=c["scale"][:nseg], T=rows, nseg=nseg,
                 name=f"{c['name']}[:{rows}]")
    return c


def torch_view(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


# ---------------------------------------------------------------------------
# Native arm: device-resident timing, per-kernel trace, end-to-end timing.
# ---------------------------------------------------------------------------
def run_native(args, c, rank, local, world, pg):
    import torch
    from adaln_video_dit_gb300 import _lib as L

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    T, D, nseg = c["T"], c["D"], c["nseg"]
    tdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    esize = 2 if tdt == torch.bfloat16 else 4

    h = {k: torch_view(c[k]) for k in ("x", "dy", "shift", "scale", "seg_id")}
    d = {k: v.to(dev) for k, v in h.items()}
    y = torch.empty(T, D, device=dev, dtype=tdt)
    dx = torch.empty_like(y)
    mean = torch.empty(T, device=dev, dtype=torch.float32)
    rstd = torch.empty_like(mean)
    dshift = torch.empty(nseg, D, device=dev, dtype=torch.float32)
    dscale = torch.empty_like(dshift)
    ws = torch.empty(max(16, L.adaln_bwd_workspace_size(T, D, nseg, tdt)), device=dev,
                     dtype=torch.uint8)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, device=dev, dtype=torch.float32)
    flush_out = torch.empty((), device=dev, dtype=torch.float32)

    def evict_l2():
        # Read 2x L2 of unrelated data: evicts the operator's lines without
        # leaving dirty lines whose write-back would land on the next kernel.
        torch.sum(flush, dim=0, out=flush_out)

    def fwd():
        L.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], c["eps"], y=y, mean=mean,
                    rstd=rstd, stream=stream)

    def bwd():
        L.adaln_bwd(d["dy"], d["x"], mean, rstd, d["scale"], d["seg_id"], dx=dx,
                    dshift=dshift, dscale=dscale, workspace=ws, stream=stream)

    clocks = ClockRecord(device_ids(dev, local)).start()
    for _ in range(args.warmup):
        evict_l2()
        fwd()
        evict_l2()
        bwd()
    rc, bits = L.adaln_get_status()
    if rc != L.ADALN_OK:
        clocks.stop()
        raise RuntimeError(f"device status after warm-up: {L.strerror(rc)} ({bits})")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    with clocks.window("timed"):
        for i in range(K):
            # L2 flushed before each call (not timed): inputs come from HBM.
            evict_l2()
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            evict_l2()
            ev[i][2].record(stream)
            bwd()
            ev[i][3].record(stream)
        torch.cuda.synchronize(dev)
    barrier(pg, dev)

    # Per-kernel durations: the library's event trace (a pair of CUDA events
    # on the launch stream around every kernel), in a second pass of the same
    # steps, so that the trace's events do not sit between the kernels of the
    # timed steps above.
    KT = min(K, 500)
    L.adaln_trace_begin(3 * KT + 8)
    with clocks.window("trace"):
        for i in range(KT):
            evict_l2()
            fwd()
            evict_l2()
            bwd()
        torch.cuda.synchronize(dev)
    L.adaln_trace_end()
    rc, bits = L.adaln_get_status()
    if rc != L.ADALN_OK:
        raise RuntimeError(f"device status after timing: {L.strerror(rc)} ({bits})")

    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in ev]
    step_ms_local = (sum(fwd_ms) + sum(bwd_ms)) / K
    step_ms = max_over_ranks(pg, step_ms_local, dev)
    kern = {}
    for kid, name in L.KERNEL_NAMES.items():
        n, ms = L.adaln_trace_get(kid)
        kern[name] = dict(launches=n, avg_us=1000.0 * ms / n if n else None)
    launches = sum(n for n, _ in (L.adaln_trace_get(k) for k in L.KERNEL_NAMES)) * K // KT

    e2e = run_e2e(args, c, h, dev, stream, L, tdt, pg, clocks)
    clocks.stop()
    fb_ms = [f + b for f, b in zip(fwd_ms, bwd_ms)]
    return dict(step_ms=step_ms, fwd_ms=statistics.mean(fwd_ms), bwd_ms=statistics.mean(bwd_ms),
                per_call={k: (statistics.median(v), min(v))
                          for k, v in (("fwd", fwd_ms), ("bwd", bwd_ms), ("fwd_bwd", fb_ms))},
                kernels=kern, launches=launches, clocks=clocks.summary(), e2e=e2e,
                shape_fwd=L.adaln_launch_shape(L.ADALN_KERNEL_FWD, T, D, nseg, tdt),
                shape_bwd=L.adaln_launch_shape(L.ADALN_KERNEL_BWD_ROWS, T, D, nseg, tdt),
                esize=esize)


def run_e2e(args, c, h, dev, stream, L, tdt, pg, clocks):
    """Same step through the public host-buffer entry point
    (adaln_fwd_bwd_host): every step copies its inputs from pinned host memory
    to the device, runs fwd + bwd, and copies every result back, all inside
    the timed region.  The library pipelines the copies and kernels in row
    chunks over its own streams."""
    import torch
    T, D, nseg = c["T"], c["D"], c["nseg"]
    if args.e2e_steps <= 0:
        return None
    hin = {k: v.pin_memory() for k, v in h.items()}
    hout = dict(y=torch.empty(T, D, dtype=tdt).pin_memory(),
                dx=torch.empty(T, D, dtype=tdt).pin_memory(),
                mean=torch.empty(T, dtype=torch.float32).pin_memory(),
                rstd=torch.empty(T, dtype=torch.float32).pin_memory(),
                dshift=torch.empty(nseg, D, dtype=torch.float32).pin_memory(),
                dscale=torch.empty(nseg, D, dtype=torch.float32).pin_memory())
    scratch = torch.empty(L.adaln_fwd_bwd_host_scratch_size(T, D, nseg, tdt, args.e2e_chunk),
                          device=dev, dtype=torch.uint8)

    def step():
        L.adaln_fwd_bwd_host(hin["x"], hin["dy"], hin["shift"], hin["scale"], hin["seg_id"],
                             c["eps"], hout, scratch, chunk_rows=args.e2e_chunk, stream=stream)

    for _ in range(3):
        step()
    # The host link bounds this leg: its copy rate on this machine, each way alone
    # (pinned memory, one copy of x), for reading the e2e number.
    probe = torch.empty_like(hin["x"], device=dev)
    link = {}
    for name, dst, src in (("h2d_gbs", probe, hin["x"]), ("d2h_gbs", hout["y"], probe)):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dst.copy_(src, non_blocking=True)
        a_.record(stream)
        dst.copy_(src, non_blocking=True)
        b_.record(stream)
        torch.cuda.synchronize(dev)
        link[name] = src.numel() * src.element_size() / (a_.elapsed_time(b_) * 1e-3) / 1e9
    del probe
    K = args.e2e_steps
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    with clocks.window("e2e"):
        ev[0].record(stream)
        for i in range(K):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    ms = max_over_ranks(pg, ev[0].elapsed_time(ev[K]) / K, dev)
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    bi = sum(v.numel() * v.element_size() for v in hin.values())
    bo = sum(v.numel() * v.element_size() for v in hout.values())
    return dict(ms_per_step=ms, h2d=bi, d2h=bo, steps=K, link=link,
                step_ms={"median": statistics.median(per_step), "min": min(per_step),
                         "max": max(per_step)})


# ---------------------------------------------------------------------------
# CPU oracle timing (bounded sample of the same workload): the forward, and the
# backward from the forward's saved statistics, timed separately.
# ---------------------------------------------------------------------------
def oracle_sample(c, rows):
    """The first `rows` tokens of the workload with the segments they touch."""
    sl = slice(0, rows)
    x, dy, seg = c["x"][sl], c["dy"][sl], c["seg_id"][sl]
    nseg = int(seg.max()) + 1 if rows else 1
    return x, dy, seg, c["shift"][:nseg], c["scale"][:nseg]


def oracle_fwd_bwd_seconds(c, rows, nthreads):
    """Seconds of one oracle forward and of one backward (from the forward's
    mean/rstd, stored as fp32 like the library's) on the first `rows` tokens."""
    import oracle
    x, dy, seg, sh, sc = oracle_sample(c, rows)
    t0 = time.perf_counter()
    _, mean, rstd = oracle.adaln_fwd(x, sh, sc, seg, c["eps"], nthreads=nthreads)
    t1 = time.perf_counter()
    oracle.adaln_bwd(dy, x, sc, seg, c["eps"], mean=mean.astype(np.float32),
                     rstd=rstd.astype(np.float32), nthreads=nthreads)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def time_oracle(c, seconds, nthreads):
    """Time the oracle's forward and backward on the first `rows` tokens of
    the workload, `rows` grown until one fwd + bwd takes about `seconds`;
    when the whole workload takes less, whole-workload calls are repeated
    until about `seconds` have passed.  Returns dict(rows, calls, fwd_s,
    bwd_s) (seconds summed over the calls)."""
    rows = min(64, c["T"])
    while True:
        tf, tb = oracle_fwd_bwd_seconds(c, rows, nthreads)
        if tf + tb >= seconds:
            return dict(rows=rows, calls=1, fwd_s=tf, bwd_s=tb)
        if rows >= c["T"]:
            calls = 1
            while tf + tb < seconds:
                f, b = oracle_fwd_bwd_seconds(c, rows, nthreads)
                tf, tb, calls = tf + f, tb + b, calls + 1
            return dict(rows=rows, calls=calls, fwd_s=tf, bwd_s=tb)
        grow = max(2.0, min(8.0, 1.2 * seconds / max(tf + tb, 1e-3)))
        rows = min(c["T"], int(rows * grow))


def oracle_rates(r):
    """Tokens/s of the forward, the backward and the fwd+bwd step."""
    n = r["rows"] * r["calls"]
    return {"fwd": n / r["fwd_s"], "bwd": n / r["bwd_s"], "fwd_bwd": n / (r["fwd_s"] + r["bwd_s"])}


def cpu_baseline(c, seconds):
    """The oracle on the host cores, all threads and one thread, for the
    forward, the backward and the fwd+bwd step."""
    import oracle
    cores = oracle.hw_threads()
    mt = time_oracle(c, seconds, cores)
    st = time_oracle(c, max(1.0, seconds / 4), 1)
    rm, rs = oracle_rates(mt), oracle_rates(st)

    def sample(r, n):
        return (f"fp64 C++ oracle on the first {r['rows']} of {c['T']} tokens, {r['calls']} "
                f"call(s) of fwd then bwd ({r['fwd_s'] + r['bwd_s']:.1f} s, {n} thread(s))")
    return {"value": rm["fwd_bwd"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample(mt, cores),
            "modes": {k: {"threads": cores, "tokens_per_s": rm[k],
                          "single_thread_tokens_per_s": rs[k]} for k in ("fwd", "bwd", "fwd_bwd")},
            "single_thread": {"value": rs["fwd_bwd"], "unit": "tokens/s", "cores": 1,
                              "sample": sample(st, 1)}}


def gpu_smi_id(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle, as it stands, on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    c = host_inputs(args.workload, args.rows)
    cores = oracle.hw_threads()
    # Size one step so that warm-up + timed steps take about two minutes.
    budget = 120.0 / max(1, args.steps + args.warmup)
    n0 = min(64, c["T"])
    tf, tb = oracle_fwd_bwd_seconds(c, n0, cores)
    rows = int(max(1, min(c["T"], budget / max((tf + tb) / n0, 1e-9))))
    for _ in range(args.warmup):
        oracle_fwd_bwd_seconds(c, rows, cores)
    sf = sb = 0.0
    for _ in range(args.steps):
        f, b = oracle_fwd_bwd_seconds(c, rows, cores)
        sf, sb = sf + f, sb + b
    dt = sf + sb
    value = rows * args.steps / dt
    sample = (f"fp64 C++ oracle fwd then bwd on the first {rows} of {c['T']} tokens per step, "
              f"{cores} threads")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": c["dtype"], "data": "synthetic",
           "config": bench_config(c, world),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                            "kind": "oracle", "sample": sample,
                            "modes": {"fwd": {"threads": cores,
                                              "tokens_per_s": rows * args.steps / sf},
                                      "bwd": {"threads": cores,
                                              "tokens_per_s": rows * args.steps / sb}},
                            "tokens_per_step": rows},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def bench_config(c, world):
    """The workload description both arms print (identical keys and values)."""
    es = 2 if c["dtype"] == "bf16" else 4
    return {"workload": c["name"], "T": c["T"], "D": c["D"], "nseg": c["nseg"],
            "io_dtype": c["dtype"], "accumulate": "f32",
            "l2": "inputs larger than L2 (x, dy %d MiB each); L2 also evicted before every "
                  "call by an untimed read of 2x L2" % (c["T"] * c["D"] * es >> 20),
            "parallelism": f"replicas x{world} (no data-path collective)"}


def load_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.txt), if it was taken on this workload and on the
    current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if line.startswith("#") or not line.strip():
                    continue
                k, v = line.split()
                vals[k] = v
        from adaln_video_dit_gb300 import build as B
        if vals.get("workload") != workload:
            return None, "no ncu capture of this workload"
        if vals.get("source_hash") != B.source_hash():
            return None, "stale: kernels changed since the ncu capture"
        return int(vals[kernel]), "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch"
    except (OSError, KeyError, ValueError):
        return None, "no ncu capture"


# ---------------------------------------------------------------------------
# Steady state over many modulation sites (the MMDiT joint-stream recipe: the
# operator runs at 2 sites per block x 30 blocks, each site with its own
# shift/scale).  A step = every site's forward + backward, back to back, with
# no L2 eviction between sites; L2 is evicted between steps.
# ---------------------------------------------------------------------------
def run_sites(args, rank, local, world, pg):
    import torch
    from adaln_video_dit_gb300 import _lib as L
    from adaln_video_dit_gb300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    c = I.make(WORKLOADS[args.workload], sites=args.sites) if WORKLOADS[args.workload] == 5 \
        else I.make(WORKLOADS[args.workload])
    T, D, nseg = c["T"], c["D"], c["nseg"]
    shifts = c["shift"] if isinstance(c["shift"], list) else [c["shift"]] * args.sites
    scales = c["scale"] if isinstance(c["scale"], list) else [c["scale"]] * args.sites
    tdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    x, dy, seg = (torch_view(c[k]).to(dev) for k in ("x", "dy", "seg_id"))
    sh = [torch_view(a).to(dev) for a in shifts]
    sc = [torch_view(a).to(dev) for a in scales]
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    mean = torch.empty(T, device=dev)
    rstd = torch.empty(T, device=dev)
    dsh = torch.empty(args.sites, nseg, D, device=dev)
    dsc = torch.empty(args.sites, nseg, D, device=dev)
    ws = torch.empty(L.adaln_bwd_workspace_size(T, D, nseg, tdt), device=dev, dtype=torch.uint8)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, device=dev)
    flush_out = torch.empty((), device=dev)

    def step(stream):
        for i in range(args.sites):
            L.adaln_fwd(x, sh[i], sc[i], seg, c["eps"], y=y, mean=mean, rstd=rstd, stream=stream)
            L.adaln_bwd(dy, x, mean, rstd, sc[i], seg, dx=dx, dshift=dsh[i], dscale=dsc[i],
                        workspace=ws, stream=stream)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        step(stream)
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            graph.capture_begin()
            step(cap)
            graph.capture_end()
        stream.wait_stream(cap)
        graph.replay()
    torch.cuda.synchronize(dev)
    rc, bits = L.adaln_get_status()
    if rc != L.ADALN_OK:
        raise RuntimeError(f"device status: {L.strerror(rc)} ({bits})")
    K = args.steps
    ms = []
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    clocks = ClockRecord(device_ids(dev, local)).start()
    with clocks.window("timed"):
        for _ in range(K):
            torch.sum(flush, dim=0, out=flush_out)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                step(stream)
            e1.record(stream)
            ms.append((e0, e1))
        torch.cuda.synchronize(dev)
    clocks.stop()
    barrier(pg, dev)
    step_ms = max_over_ranks(pg, statistics.mean(a.elapsed_time(b) for a, b in ms), dev)
    if rank == 0:
        ab = alg_bytes(T, D, nseg, 2 if tdt == torch.bfloat16 else 4)
        peak, kind = peaks()
        gbs = args.sites * ab["fwd_bwd"] / (step_ms * 1e-3) / 1e9
        out = {"report": "sites_steady_state", "metric": METRIC,
               "value": world * args.sites * T / (step_ms * 1e-3), "unit": "tokens/s",
               "n_gpus": world, "steps": K, "ms_per_step": step_ms, "dtype": c["dtype"],
               "config": {"workload": c["name"], "T": T, "D": D, "nseg": nseg,
                          "sites": args.sites, "cuda_graph": bool(args.graph),
                          "launches_per_step": 3 * args.sites},
               "gbs": gbs, "frac_of_" + kind: gbs / peak, "clocks": clocks.summary()}
        print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# Context report: torch's unfused chain (layer_norm, gather, multiply, add and
# their autograd backward) against the fused operator on the same inputs.
# ---------------------------------------------------------------------------
def report_shapes(args):
    """Shape benchmarking (AdaptiveLoad, Technical summary section 2.A) of the
    fused operator itself: fwd + bwd time over a grid of (B samples, S tokens)
    at D = 5120 bf16, the fit t ~ a + b*B*S**p, and the compute bound M_comp
    and bucket sizes B_shape(S) it implies for a target step time."""
    import torch
    from adaln_video_dit_gb300 import schedule as Sch

    torch.cuda.set_device(0)
    shapes = [(B, S) for S in (1024, 4096, 16384, 32760) for B in (1, 2, 4, 8)]
    res = Sch.shape_benchmark(shapes, D=5120, steps=20, warmup=3)
    Bs, Ss, ts = zip(*res)
    a, b, p = Sch.fit_cost_model(Bs, Ss, ts)
    tau = 1.0  # ms
    m_comp = Sch.m_comp_for_step_time(a, b, tau)
    buckets = Sch.bucket_plan([256, 1024, 4096, 16384, 32760], 65536, m_comp, p)
    rel = [abs(float(Sch.cost_model(B_, S_, a, b, p)) - t_) / t_ for B_, S_, t_ in res]
    print(json.dumps({
        "report": "shape_benchmark", "device": torch.cuda.get_device_name(0),
        "D": 5120, "dtype": "bf16", "step": "adaln_fwd + adaln_bwd, one segment per sample",
        "points_B_S_ms": [[int(B_), int(S_), round(t_, 5)] for B_, S_, t_ in res],
        "fit": {"a_ms": a, "b_ms_per_token_p": b, "p": p,
                "max_rel_residual": max(rel)},
        "target_step_ms": tau, "m_comp": m_comp, "m_mem": 65536,
        "b_shape": {str(k): v for k, v in buckets.items()}}))


def report_widths(args):
    """Forward and backward per call over a grid of row widths D (bf16 and
    fp32, T = 32768 rows in 4 segments, seeded synthetic inputs): median of 30
    calls, L2 evicted before every call, algorithmic GB/s as a fraction of the
    measured copy peak, and the launch shape each width gets."""
    import statistics
    import torch
    from adaln_video_dit_gb300 import _lib as L

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, device=dev)
    fo = torch.empty((), device=dev)
    peak, peak_kind = peaks()
    T, nseg = 32768, 4
    gen = torch.Generator(device=dev)
    gen.manual_seed(17)
    rows = []
    for dt, widths in ((torch.bfloat16, (512, 1024, 1536, 2048, 3072, 4096, 5120, 6144, 8192)),
                       (torch.float32, (512, 1024, 1536, 2048, 3072, 4096))):
        es = 2 if dt == torch.bfloat16 else 4
        for D in widths:
            x = torch.randn(T, D, device=dev, generator=gen).to(dt)
            dy = (torch.randn(T, D, device=dev, generator=gen) * 1e-2).to(dt)
            sh = (torch.randn(nseg, D, device=dev, generator=gen) * 0.5).to(dt)
            sc = (torch.randn(nseg, D, device=dev, generator=gen) * 0.5).to(dt)
            seg = (torch.arange(T, device=dev) * nseg // T).to(torch.int32)
            y, dx = torch.empty_like(x), torch.empty_like(x)
            mean, rstd = torch.empty(T, device=dev), torch.empty(T, device=dev)
            dsh, dsc = torch.empty(nseg, D, device=dev), torch.empty(nseg, D, device=dev)
            ws = torch.empty(L.adaln_bwd_workspace_size(T, D, nseg, dt), device=dev,
                             dtype=torch.uint8)

            def fwd():
                L.adaln_fwd(x, sh, sc, seg, 1e-6, y=y, mean=mean, rstd=rstd)

            def bwd():
                L.adaln_bwd(dy, x, mean, rstd, sc, seg, dx=dx, dshift=dsh, dscale=dsc,
                            workspace=ws)

            for _ in range(3):
                fwd()
                bwd()
            tf, tb = [], []
            for _ in range(30):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                torch.sum(flush, dim=0, out=fo)
                ev[0].record()
                fwd()
                ev[1].record()
                torch.sum(flush, dim=0, out=fo)
                ev[2].record()
                bwd()
                ev[3].record()
                torch.cuda.synchronize()
                tf.append(ev[0].elapsed_time(ev[1]) * 1e3)
                tb.append(ev[2].elapsed_time(ev[3]) * 1e3)
            rc, bits = L.adaln_get_status()
            if rc != L.ADALN_OK:
                raise RuntimeError(f"device status: {L.strerror(rc)} ({bits})")
            ab = alg_bytes(T, D, nseg, es)
            mf, mb = statistics.median(tf), statistics.median(tb)
            rows.append({
                "dtype": "bf16" if es == 2 else "f32", "D": D,
                "fwd_us": round(mf, 1), "fwd_frac": round(ab["fwd"] / (mf * 1e3) / peak, 3),
                "bwd_us": round(mb, 1), "bwd_frac": round(ab["bwd"] / (mb * 1e3) / peak, 3),
                "fwd_shape": L.adaln_launch_shape(L.ADALN_KERNEL_FWD, T, D, nseg, dt),
                "bwd_shape": L.adaln_launch_shape(L.ADALN_KERNEL_BWD_ROWS, T, D, nseg, dt)})
            del x, dy, y, dx, ws
    print(json.dumps({"report": "widths", "device": torch.cuda.get_device_name(0), "T": T,
                      "nseg": nseg, "peak_gbs": peak, "peak_kind": peak_kind,
                      "l2": "evicted before every call", "rows": rows}))


def report_fixed_cost(args):
    """Where a call's time goes, host or GPU, per workload: host time of one
    call through the C ABI (the raw ctypes call and the Python binding with
    outputs given), GPU time between CUDA events per call with the host kept
    ahead of the GPU (a device-side delay first, so no launch waits for the
    host), the library's per-kernel trace, and the floor of any call timed
    this way (a one-element fill between the same events).  L2 evicted
    before every call."""
    import ctypes
    import torch
    from adaln_video_dit_gb300 import _lib as L

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, device=dev)
    fo = torch.empty((), device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    S = ctypes.c_void_p(st.cuda_stream)
    K = 40

    def gpu_us(f, b):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        torch.cuda.synchronize(dev)
        torch.cuda._sleep(int(1e8))  # the host queues every call meanwhile
        for e in ev:
            torch.sum(flush, dim=0, out=fo)
            e[0].record(st)
            f()
            e[1].record(st)
            torch.sum(flush, dim=0, out=fo)
            e[2].record(st)
            b()
            e[3].record(st)
        torch.cuda.synchronize(dev)
        return (statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in ev),
                statistics.median(e[2].elapsed_time(e[3]) * 1e3 for e in ev))

    def host_us(fn, n=200):
        torch.cuda._sleep(int(4e8))
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        dt = (time.perf_counter() - t0) / n * 1e6
        torch.cuda.synchronize(dev)
        return dt

    tiny = torch.empty(1, device=dev)
    floor = gpu_us(lambda: tiny.fill_(0), lambda: tiny.fill_(1))
    out = {"report": "fixed_cost", "device": torch.cuda.get_device_name(dev),
           "l2": "evicted before every call", "floor_us": min(floor),
           "ctypes_call_us": host_us(lambda: L.raw.adaln_strerror(0)), "cases": []}
    from adaln_video_dit_gb300 import inputs as I
    for name in ("wan13b", "mmdit_joint", "long_video", "shape_1x1024x5120"):
        if name.startswith("shape"):
            c = I.random_case(11, 1024, 5120, 1, dtype="bf16")
            c["name"] = name
        else:
            c = host_inputs(name)
        T, D, nseg = c["T"], c["D"], c["nseg"]
        d = {k: torch_view(c[k]).to(dev) for k in ("x", "dy", "shift", "scale", "seg_id")}
        y, dx = torch.empty_like(d["x"]), torch.empty_like(d["x"])
        mean, rstd = torch.empty(T, device=dev), torch.empty(T, device=dev)
        dsh, dsc = torch.empty(nseg, D, device=dev), torch.empty(nseg, D, device=dev)
        nws = L.adaln_bwd_workspace_size(T, D, nseg, torch.bfloat16)
        ws = torch.empty(nws, device=dev, dtype=torch.uint8)
        fa = (P(d["x"]), P(d["shift"]), P(d["scale"]), P(d["seg_id"]), T, D, nseg, L.ADALN_BF16,
              ctypes.c_float(1e-6), P(y), P(mean), P(rstd), S)
        ba = (P(d["dy"]), P(d["x"]), P(mean), P(rstd), P(d["scale"]), P(d["seg_id"]), T, D, nseg,
              L.ADALN_BF16, P(dx), P(dsh), P(dsc), P(ws), ctypes.c_size_t(nws), S)

        def fwd_py():
            L.adaln_fwd(d["x"], d["shift"], d["scale"], d["seg_id"], 1e-6, y=y, mean=mean,
                        rstd=rstd, stream=st)

        def bwd_py():
            L.adaln_bwd(d["dy"], d["x"], mean, rstd, d["scale"], d["seg_id"], dx=dx, dshift=dsh,
                        dscale=dsc, workspace=ws, stream=st)

        fwd_raw = lambda: L.raw.adaln_fwd(*fa)  # noqa: E731
        bwd_raw = lambda: L.raw.adaln_bwd(*ba)  # noqa: E731
        for _ in range(3):
            fwd_raw()
            bwd_raw()
        torch.cuda.synchronize(dev)
        g_f, g_b = gpu_us(fwd_raw, bwd_raw)
        L.adaln_trace_begin(3 * K + 8)
        gpu_us(fwd_raw, bwd_raw)
        L.adaln_trace_end()
        trace = {nm: 1e3 * L.adaln_trace_get(k)[1] / max(1, L.adaln_trace_get(k)[0])
                 for k, nm in L.KERNEL_NAMES.items()}
        ab = alg_bytes(T, D, nseg, 2)
        peak, kind = peaks()
        out["cases"].append({
            "workload": c["name"], "T": T, "D": D, "nseg": nseg,
            "host_us": {"fwd_raw": host_us(fwd_raw), "bwd_raw": host_us(bwd_raw),
                        "fwd_binding": host_us(fwd_py), "bwd_binding": host_us(bwd_py)},
            "gpu_us": {"fwd": g_f, "bwd": g_b},
            "trace_us": trace,
            "at_peak_us": {"fwd": ab["fwd"] / (peak * 1e3), "bwd": ab["bwd"] / (peak * 1e3)},
            "peak_gbs": peak, "peak_kind": kind})
        rc, bits = L.adaln_get_status()
        if rc != L.ADALN_OK:
            raise RuntimeError(f"device status: {L.strerror(rc)} ({bits})")
        del d, y, dx, ws
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)


def report_unfused(args):
    import torch
    import torch.nn.functional as F
    from adaln_video_dit_gb300 import _lib as L
    from adaln_video_dit_gb300 import autograd as A

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, device=dev, dtype=torch.float32)
    flush_out = torch.empty((), device=dev, dtype=torch.float32)

    def timed(fn, reps=30, warm=5):
        for _ in range(warm):
            fn()
        ms = []
        for _ in range(reps):
            torch.sum(flush, dim=0, out=flush_out)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    def saved_bytes(fn):
        seen = {}

        def pack(t):
            st = t.untyped_storage()
            seen[st.data_ptr()] = max(seen.get(st.data_ptr(), 0), st.nbytes())
            return t
        with torch.autograd.graph.saved_tensors_hooks(pack, lambda t: t):
            fn()
        return sum(seen.values())

    out = {"report": "unfused_torch_vs_fused", "device": torch.cuda.get_device_name(dev),
           "torch": torch.__version__, "dtype": "bf16", "l2": "evicted by a 2x L2 read before each rep",
           "cases": []}
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    for name, T, D in (("long_video", 32760, 5120), ("N=64000", 64000, 5120)):
        x = torch.randn(T, D, device=dev, generator=g).to(torch.bfloat16)
        dy = (torch.randn(T, D, device=dev, generator=g) * 1e-2).to(torch.bfloat16)
        shift = (torch.randn(1, D, device=dev, generator=g) * 0.5).to(torch.bfloat16)
        scale = (torch.randn(1, D, device=dev, generator=g) * 0.5).to(torch.bfloat16)
        seg = torch.zeros(T, device=dev, dtype=torch.int32)
        y, mean, rstd = L.adaln_fwd(x, shift, scale, seg, 1e-6)
        dx = torch.empty_like(x)
        dsh = torch.empty(1, D, device=dev)
        dsc = torch.empty(1, D, device=dev)
        ws = torch.empty(L.adaln_bwd_workspace_size(T, D, 1, torch.bfloat16), device=dev,
                         dtype=torch.uint8)

        def fused_fwd():
            L.adaln_fwd(x, shift, scale, seg, 1e-6, y=y, mean=mean, rstd=rstd)

        def fused_fwd_bwd():
            fused_fwd()
            L.adaln_bwd(dy, x, mean, rstd, scale, seg, dx=dx, dshift=dsh, dscale=dsc, workspace=ws)

        # The usual DiT form of the unfused chain: per-sample modulation
        # broadcast over the sample's tokens ([B, N, D] with [B, 1, D]; B = 1).
        def unfused_fwd():
            with torch.no_grad():
                xb = x.view(1, T, D)
                F.layer_norm(xb, (D,), eps=1e-6) * (1 + scale.view(1, 1, D)) + shift.view(1, 1, D)

        xg = x.detach().requires_grad_(True)
        shg = shift.detach().requires_grad_(True)
        scg = scale.detach().requires_grad_(True)

        def unfused_chain():
            xb = xg.view(1, T, D)
            return (F.layer_norm(xb, (D,), eps=1e-6) * (1 + scg.view(1, 1, D))
                    + shg.view(1, 1, D))

        def unfused_fwd_bwd():
            unfused_chain().backward(dy.view(1, T, D))

        t_ff, t_ffb = timed(fused_fwd), timed(fused_fwd_bwd)
        t_uf, t_ufb = timed(unfused_fwd), timed(unfused_fwd_bwd)
        fused_saved = saved_bytes(lambda: A.adaln_modulate(xg, shg, scg, seg))
        chain_saved = saved_bytes(unfused_chain)
        out["cases"].append({
            "workload": name, "T": T, "D": D,
            "fused_fwd_ms": t_ff, "fused_fwd_bwd_ms": t_ffb,
            "unfused_fwd_ms": t_uf, "unfused_fwd_bwd_ms": t_ufb,
            "speedup_fwd": t_uf / t_ff, "speedup_bwd": (t_ufb - t_uf) / (t_ffb - t_ff),
            "speedup_fwd_bwd": t_ufb / t_ffb,
            "saved_bytes_fused": fused_saved, "saved_bytes_unfused": chain_saved,
            "activation_memory_saving": 1.0 - fused_saved / chain_saved})
        del x, dy, y, dx, xg, ws
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.report == "unfused":
        report_unfused(args)
        return
    if args.report == "shapes":
        report_shapes(args)
        return
    if args.report == "fixed-cost":
        report_fixed_cost(args)
        return
    if args.report == "widths":
        report_widths(args)
        return
    rank, local, world, pg = dist_setup(args.gpus)
    if args.sites > 1 and args.impl == "native":
        run_sites(args, rank, local, world, pg)
        if pg is not None:
            pg.destroy_process_group()
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        if pg is not None:
            pg.destroy_process_group()
        return
    c = host_inputs(args.workload, args.rows)
    r = run_native(args, c, rank, local, world, pg)
    if rank == 0:
        T, D, nseg, es = c["T"], c["D"], c["nseg"], r["esize"]
        ab = alg_bytes(T, D, nseg, es)
        peak, peak_kind = peaks()
        step_s = r["step_ms"] / 1000.0
        value = world * T / step_s
        dom = "adaln_bwd_rows_kernel"
        dom_us = r["kernels"][dom]["avg_us"]
        achieved = ab["bwd_rows"] / (dom_us * 1e-6) / 1e9
        traffic, traffic_note = load_traffic(
            dom, args.workload if not args.rows else f"{args.workload}:{args.rows}")
        breakdown = {}
        for k, ms in (("fwd", r["fwd_ms"]), ("bwd", r["bwd_ms"]),
                      ("fwd_bwd", r["fwd_ms"] + r["bwd_ms"])):
            gbs = ab[k] / (ms * 1e-3) / 1e9
            med, best = r["per_call"][k]
            breakdown[k] = {"ms": ms, "ms_median": med, "ms_best": best,
                            "tokens_per_s": T / (ms * 1e-3), "alg_bytes": ab[k],
                            "gbs": gbs, "frac_of_" + peak_kind: gbs / peak,
                            "frac_of_8000_spec": gbs / 8000.0}
        e2e = r["e2e"]
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["step_ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": c["dtype"], "data": "synthetic",
            "config": bench_config(c, world),
            "launch": {"fwd": r["shape_fwd"], "bwd_rows": r["shape_bwd"]},
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "traffic_note": traffic_note,
                         "alg_bytes_per_launch": ab["bwd_rows"], "avg_us": dom_us},
            "breakdown": breakdown,
            "kernels": r["kernels"],
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
            "e2e": None if e2e is None else {
                "value": world * T / (e2e["ms_per_step"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e["ms_per_step"], "steps": e2e["steps"],
                "api": "adaln_fwd_bwd_host",
                "host_link_gbs": e2e["link"],
                "step_ms_spread": e2e["step_ms"],
                "link_bound_ms": 1e3 * max(e2e["h2d"] / (e2e["link"]["h2d_gbs"] * 1e9),
                                           e2e["d2h"] / (e2e["link"]["d2h_gbs"] * 1e9))},
        }
        if r["clocks"].get("sm_mhz"):
            # Clock-normalised cost of a step: its time in SM clock cycles.
            out["clocks"]["step_mcycles"] = r["step_ms"] * 1e-3 * r["clocks"]["sm_mhz"]
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(c, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
