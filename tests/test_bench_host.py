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


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2050, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1990, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2050 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    c.lines = ["0, 1500, 2070, 1000, 0x8, Active, Not Active, Not Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown"]
    assert bench.ClockSampler(0).summary() == {"sm_mhz": None, "sm_max_mhz": None,
                                              "reasons": [], "samples": 0}


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    os.makedirs(tmp_path / "profiles")
    p = tmp_path / "profiles" / "traffic.txt"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p.write_text(f"# comment\nsource_hash {B.source_hash()}\nadaln_bwd_rows_kernel 123\n")
    assert bench.load_traffic("adaln_bwd_rows_kernel")[0] == 123
    assert bench.load_traffic("adaln_fwd_kernel")[0] is None  # not captured
    p.write_text("source_hash 0000000000000000\nadaln_bwd_rows_kernel 123\n")
    v, note = bench.load_traffic("adaln_bwd_rows_kernel")
    assert v is None and note.startswith("stale")
    p.unlink()
    assert bench.load_traffic("adaln_bwd_rows_kernel") == (None, "no ncu capture")


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
    tps, rows, dt, calls = bench.time_oracle(c, 0.3, 1)
    assert rows == c["T"] and calls > 1 and dt >= 0.3
    assert tps == pytest.approx(rows * calls / dt)
