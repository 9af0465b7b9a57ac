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
    p.add_argument("--sites", type=int, default=1,
                   help="modulation sites per step (mmdit_joint steady state: 60 = 2 per "
                        "block x 30 blocks), each its own shift/scale, back to back")
    p.add_argument("--graph", action="store_true",
                   help="with --sites: replay each step as one captured CUDA graph")
    p.add_argument("--report", choices=["unfused", "shapes"], default=None,
                   help="instead of the benchmark line: compare with torch's unfused "
                        "chain (time and saved activation bytes), or shape-benchmark "
                        "the operator and fit the step-time cost model")
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
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


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
def host_inputs(name):
    from adaln_video_dit_gb300 import inputs as I
    c = I.make(WORKLOADS[name])
    if isinstance(c["shift"], list):
        c["shift"], c["scale"] = c["shift"][0], c["scale"][0]
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

    for _ in range(args.warmup):
        evict_l2()
        fwd()
        evict_l2()
        bwd()
    rc, bits = L.adaln_get_status()
    if rc != L.ADALN_OK:
        raise RuntimeError(f"device status after warm-up: {L.strerror(rc)} ({bits})")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_smi_id(local)) as clocks:
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
    launches = 3 * K  # fwd, bwd row pass and finalize per timed step

    e2e = run_e2e(args, c, h, dev, stream, L, tdt, pg)
    return dict(step_ms=step_ms, fwd_ms=statistics.mean(fwd_ms), bwd_ms=statistics.mean(bwd_ms),
                fwd_ms_median=statistics.median(fwd_ms), bwd_ms_median=statistics.median(bwd_ms),
                kernels=kern, launches=launches, clocks=clocks.summary(), e2e=e2e,
                shape_fwd=L.adaln_launch_shape(L.ADALN_KERNEL_FWD, T, D, nseg, tdt),
                shape_bwd=L.adaln_launch_shape(L.ADALN_KERNEL_BWD_ROWS, T, D, nseg, tdt),
                esize=esize)


def run_e2e(args, c, h, dev, stream, L, tdt, pg):
    """Same step through the public host-buffer entry point
    (adaln_fwd_bwd_host): every step copies its inputs from pinned host memory
    to the device, runs fwd + bwd, and copies every result back, all inside
    the timed region.  The library pipelines the copies and kernels in row
    chunks over its own streams."""
    import torch
    T, D, nseg = c["T"], c["D"], c["nseg"]
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
    K = args.e2e_steps
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / K, dev)
    bi = sum(v.numel() * v.element_size() for v in hin.values())
    bo = sum(v.numel() * v.element_size() for v in hout.values())
    return dict(ms_per_step=ms, h2d=bi, d2h=bo, steps=K)


# ---------------------------------------------------------------------------
# CPU oracle timing (bounded sample of the same workload).
# ---------------------------------------------------------------------------
def oracle_step_fn(c, rows):
    import oracle
    sl = slice(0, rows)
    x, dy, seg = c["x"][sl], c["dy"][sl], c["seg_id"][sl]
    nseg = int(seg.max()) + 1 if rows else 1
    sh, sc = c["shift"][:nseg], c["scale"][:nseg]

    def step(nthreads):
        oracle.adaln_fwd(x, sh, sc, seg, c["eps"], nthreads=nthreads)
        oracle.adaln_bwd(dy, x, sc, seg, c["eps"], nthreads=nthreads)
    return step


def time_oracle(c, seconds, nthreads):
    """Tokens/s of the oracle's fwd+bwd on the first `rows` tokens of the
    workload, `rows` grown until one call takes about `seconds`; when the
    whole workload takes less, whole-workload calls are repeated until about
    `seconds` have passed.  Returns (tokens/s, rows per call, seconds, calls)."""
    rows = min(64, c["T"])
    while True:
        step = oracle_step_fn(c, rows)
        t0 = time.perf_counter()
        step(nthreads)
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return rows / dt, rows, dt, 1
        if rows >= c["T"]:
            calls = 1
            while dt < seconds:
                step(nthreads)
                calls += 1
                dt = time.perf_counter() - t0
            return rows * calls / dt, rows, dt, calls
        grow = max(2.0, min(8.0, 1.2 * seconds / max(dt, 1e-3)))
        rows = min(c["T"], int(rows * grow))


def cpu_baseline(c, seconds):
    import oracle
    cores = oracle.hw_threads()
    tps_mt, rows_mt, dt_mt, n_mt = time_oracle(c, seconds, cores)
    tps_st, rows_st, dt_st, n_st = time_oracle(c, max(1.0, seconds / 4), 1)
    return {"value": tps_mt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"fp64 C++ oracle fwd+bwd on the first {rows_mt} tokens of the "
                       f"workload, {n_mt} call(s) ({dt_mt:.1f} s, {cores} threads)"),
            "single_thread": {"value": tps_st, "unit": "tokens/s", "cores": 1,
                              "sample": f"first {rows_st} tokens, {n_st} call(s) ({dt_st:.1f} s)"}}


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
    c = host_inputs(args.workload)
    cores = oracle.hw_threads()
    # Size one step so that warm-up + timed steps take about two minutes.
    budget = 120.0 / max(1, args.steps + args.warmup)
    probe = oracle_step_fn(c, min(64, c["T"]))
    t0 = time.perf_counter()
    probe(cores)
    per_row = (time.perf_counter() - t0) / min(64, c["T"])
    rows = int(max(1, min(c["T"], budget / max(per_row, 1e-9))))
    step = oracle_step_fn(c, rows)
    for _ in range(args.warmup):
        step(cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(cores)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    sample = (f"fp64 C++ oracle fwd+bwd on the first {rows} of {c['T']} tokens per step, "
              f"{cores} threads")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": c["dtype"], "data": "synthetic",
           "config": {"workload": c["name"], "T": c["T"], "D": c["D"], "nseg": c["nseg"],
                      "tokens_per_step": rows},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def load_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.txt), if it was taken on the current kernel sources."""
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
    with ClockSampler(gpu_smi_id(local)) as clocks:
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
    c = host_inputs(args.workload)
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
        traffic, traffic_note = load_traffic(dom)
        breakdown = {}
        for k, ms in (("fwd", r["fwd_ms"]), ("bwd", r["bwd_ms"]),
                      ("fwd_bwd", r["fwd_ms"] + r["bwd_ms"])):
            gbs = ab[k] / (ms * 1e-3) / 1e9
            breakdown[k] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "alg_bytes": ab[k],
                            "gbs": gbs, "frac_of_" + peak_kind: gbs / peak,
                            "frac_of_8000_spec": gbs / 8000.0}
        e2e = r["e2e"]
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["step_ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": c["dtype"], "data": "synthetic",
            "config": {"workload": c["name"], "T": T, "D": D, "nseg": nseg,
                       "io_dtype": c["dtype"], "accumulate": "f32",
                       "l2": "inputs larger than L2 (x, dy %d MiB each); L2 also evicted "
                             "before every call by an untimed read of 2x L2" % (T * D * es >> 20),
                       "parallelism": f"replicas x{world} (no data-path collective)",
                       "launch_fwd": r["shape_fwd"], "launch_bwd_rows": r["shape_bwd"]},
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "traffic_note": traffic_note,
                         "alg_bytes_per_launch": ab["bwd_rows"], "avg_us": dom_us},
            "breakdown": breakdown,
            "kernels": r["kernels"],
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
            "e2e": {"value": world * T / (e2e["ms_per_step"] * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": e2e["ms_per_step"], "steps": e2e["steps"],
                    "api": "adaln_fwd_bwd_host"},
        }
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(c, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
