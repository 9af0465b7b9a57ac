"""Host-side logic of bench.py (no GPU): algorithmic byte counts, the clock
record's parsing, the ncu traffic lookup and its staleness rule, the CPU
baseline sampling, and the kernel source hash that ties them together."""
import os

import pytest

import bench
from adaln_video_dit_gb300 import build as B


def test_algorithmic_bytes_long_video():
    # bf16, D = 5120: 20,492 B/token forward, 30,732 B/token backward row pass.
    T, D, nseg, s = 32760, 5120, 1, 2
    b = bench.alg_bytes(T, D, nseg, s)
    assert b["fwd"] == T * 20492 + 2 * nseg * D * s == 671338400
    assert b["bwd_rows"] == T * 30732 + nseg * D * s == 1006790560
    assert b["bwd"] == b["bwd_rows"] + 2 * nseg * D * 4
    assert b["fwd_bwd"] == b["fwd"] + b["bwd"]


def test_clock_record_summary_counts_samples_under_load():
    c = bench.ClockRecord({})
    c.windows = [("timed", 10.0, 11.0), ("e2e", 20.0, 21.0)]
    c.samples = [(9.5, 1400.0, 2070.0, [], 300.0),
                 (10.1, 2070.0, 2070.0, [], 900.0),
                 (10.5, 2050.0, 2070.0, ["sw_power_cap"], 1300.0),
                 (10.9, 1990.0, 2070.0, ["sw_power_cap"], 1390.0),
                 (11.5, 1000.0, 2070.0, ["hw_slowdown"], 200.0),
                 (20.5, 2070.0, 2070.0, [], 700.0)]
    s = c.summary()
    assert s["samples"] == 6 and s["samples_under_load"] == 4
    assert s["samples_by_window"] == {"timed": 3, "e2e": 1}
    # statistics over the samples under load only
    assert s["sm_mhz"] == 2060 and s["sm_mhz_min"] == 1990 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0
    empty = bench.ClockRecord({}).summary()
    assert empty["samples"] == 0 and empty["sm_mhz"] is None and empty["reasons"] == []


def test_smi_line_parsing():
    v = bench.parse_smi_line("0, 2050, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active")
    assert v == (2050.0, 2070.0, ["sw_power_cap"], 1300.0)
    v = bench.parse_smi_line("0, 1500, 2070, [N/A], 0x8, Active, Not Active, Not Active, Not Active")
    assert v == (1500.0, 2070.0, ["hw_slowdown"], None)
    assert bench.parse_smi_line("garbage line") is None
    assert bench.parse_smi_line("0, [N/A], 2070, 1.0, 0x0, a, b, c, d") is None


class _FakeNvml:
    """Getters only: a call to any NVML setter would raise AttributeError."""

    def __init__(self):
        self.shutdown = False

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, h):
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        assert kind == 1  # NVML_CLOCK_SM
        out._obj.value = 1980
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = 0x1 | 0x4  # idle + software power cap
        return 0

    def nvmlDeviceGetPowerUsage(self, h, out):
        out._obj.value = 1234000
        return 0

    def nvmlShutdown(self):
        self.shutdown = True
        return 0


def test_nvml_sampler_reads_clocks_in_windows(monkeypatch):
    import ctypes
    import time
    fake = _FakeNvml()
    monkeypatch.setattr(ctypes, "CDLL", lambda name: fake)
    c = bench.ClockRecord({"pci_bus_id": "00000000:01:00.0"}, period_s=0.001).start()
    with c.window("timed"):
        time.sleep(0.1)
    c.stop()
    s = c.summary()
    assert s["source"] == "nvml" and fake.shutdown
    assert s["samples_under_load"] >= 20
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1234.0


def test_traffic_lookup_follows_the_workload_and_source_hash(tmp_path, monkeypatch):
    os.makedirs(tmp_path / "profiles")
    p = tmp_path / "profiles" / "traffic.txt"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p.write_text(f"# comment\nworkload long_video\nsource_hash {B.source_hash()}\n"
                 "adaln_bwd_rows_kernel 123\n")
    assert bench.load_traffic("adaln_bwd_rows_kernel", "long_video")[0] == 123
    assert bench.load_traffic("adaln_fwd_kernel", "long_video")[0] is None  # not captured
    v, note = bench.load_traffic("adaln_bwd_rows_kernel", "wan13b")  # another workload
    assert v is None and note == "no ncu capture of this workload"
    assert bench.load_traffic("adaln_bwd_rows_kernel", "long_video:4096")[0] is None  # truncated
    p.write_text("workload long_video\nsource_hash 0000000000000000\nadaln_bwd_rows_kernel 123\n")
    v, note = bench.load_traffic("adaln_bwd_rows_kernel", "long_video")
    assert v is None and note.startswith("stale")
    p.unlink()
    assert bench.load_traffic("adaln_bwd_rows_kernel", "long_video") == (None, "no ncu capture")


def test_source_hash_ignores_comments_only():
    code = 'int f(int a) { // add one\n  return a + 1; /* "x" */ }\nconst char* s = "a // b";\n'
    same = 'int f(int a) {\n  return a + 1;   }\nconst char* s = "a // b";  // c\n'
    other = 'int f(int a) { return a + 2; }\nconst char* s = "a // b";\n'
    assert B._strip_comments(code) == B._strip_comments(same)
    assert B._strip_comments(code) != B._strip_comments(other)
    # a comment marker inside a string literal is code
    assert "a // b" in B._strip_comments(code)


@pytest.mark.timeout(300)
def test_cpu_baseline_sample_reaches_the_target_time():
    c = bench.host_inputs("tiny_fp32")
    r = bench.time_oracle(c, 0.3, 1)
    assert r["rows"] == c["T"] and r["calls"] > 1 and r["fwd_s"] + r["bwd_s"] >= 0.3
    rates = bench.oracle_rates(r)
    n = r["rows"] * r["calls"]
    assert rates["fwd"] == pytest.approx(n / r["fwd_s"])
    assert rates["bwd"] == pytest.approx(n / r["bwd_s"])
    assert rates["fwd_bwd"] == pytest.approx(n / (r["fwd_s"] + r["bwd_s"]))


def test_truncated_workload_keeps_its_structure():
    full = bench.host_inputs("mmdit_joint")
    c = bench.host_inputs("mmdit_joint", rows=5000)
    assert c["T"] == 5000 and c["x"].shape == (5000, full["D"])
    # 512 text + 4096 video tokens per sample: row 4999 is sample 1's text
    assert c["nseg"] == 3 and c["shift"].shape == (3, full["D"])
    assert (c["seg_id"] == full["seg_id"][:5000]).all()


@pytest.mark.timeout(300)
def test_reference_arm_prints_the_native_config(capsys):
    import argparse
    import json
    args = argparse.Namespace(workload="tiny_fp32", steps=2, warmup=1, rows=0)
    bench.run_reference(args, 0, 1)
    out = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert out["impl"] == "reference"
    assert out["config"] == bench.bench_config(bench.host_inputs("tiny_fp32"), 1)
    assert set(out["cpu_baseline"]["modes"]) == {"fwd", "bwd"}
    assert out["e2e"]["value"] == out["value"]
