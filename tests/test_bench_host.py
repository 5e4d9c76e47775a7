"""Host logic of bench.py that decides what a result line reports, checked on
the CPU: the clock summary (only samples inside the timed region count;
throttle reasons are collected), the source key of the committed DRAM-traffic
record (comment edits keep it, code edits drop it, so traffic turns null once
the kernel changes), and the weight bytes the HBM roofline counts."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_scaled_mx_gb300 import workload as W  # noqa: E402


def _line(sm, reasons=()):
    flags = ["Active" if n in reasons else "Not Active"
             for n in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    return ", ".join(["0", str(sm), "2070", "900.5", "0x0"] + flags)


def test_clock_summary_counts_only_the_timed_region():
    c = bench.ClockSampler(0)
    c.lines = [(0.0, _line(1000, ["hw_slowdown"])),    # before the timed region
               (1.00, _line(2070)), (1.02, _line(2055, ["sw_power_cap"])), (1.04, _line(2070)),
               (5.0, _line(300, ["sw_thermal_slowdown"]))]   # long after it
    c.mark(0.99, 1.05)
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_short_region_takes_the_neighbouring_samples():
    """A sample reports the period before it arrived, so one arriving up to 1.5
    periods after the region still counts; with none there, the nearest ones do."""
    c = bench.ClockSampler(0)
    c.lines = [(1.000, _line(2070)), (1.020, _line(2040)), (9.0, _line(100))]
    c.mark(1.0101, 1.0102)                # shorter than one sampling period
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2040
    c.lines = [(1.000, _line(2070)), (1.100, _line(2040))]
    s = c.summary()                       # nothing within 1.5 periods after: the sample before
    assert s["samples"] == 1 and s["sm_mhz"] == 2070


def test_clock_summary_without_samples_says_so():
    c = bench.ClockSampler(0)
    c.lines = [(1.0, "garbage"), (1.01, "0, [N/A], 2070")]
    assert c.summary()["reasons"] == ["unsampled"]


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and profiles that bench.py reads."""
    src = os.path.join(ROOT, "block_scaled_mx_gb300", "csrc")
    shutil.copytree(src, tmp_path / "block_scaled_mx_gb300" / "csrc")
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_record_follows_the_kernel_code(tree):
    key = bench.source_hash()
    rec = {"source_hash": key, "dram_bytes_per_launch": 123456789.0}
    (tree / "profiles" / "ncu_gemm1_decode_mxfp8.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("gemm1", "decode_mxfp8") == 123456789.0
    assert bench.ncu_traffic("gemm1", "prefill_mxfp8") is None       # no record for that workload
    gemm = tree / "block_scaled_mx_gb300" / "csrc" / "gemm.cu"
    text = gemm.read_text()
    gemm.write_text("// a new comment line\n" + text.replace("\n", "\n\n", 3) + "\n/* and a block comment */\n")
    assert bench.source_hash() == key                                 # comments and blank lines only
    assert bench.ncu_traffic("gemm1", "decode_mxfp8") == 123456789.0
    gemm.write_text(text + "\nstatic int added_code = 1;\n")
    assert bench.source_hash() != key                                 # the code changed
    assert bench.ncu_traffic("gemm1", "decode_mxfp8") is None


def test_weight_bytes_per_expert_include_the_scales():
    wl = W.WORKLOADS["decode_mxfp8"]
    w1, w2 = bench.weight_bytes_per_expert(wl)
    assert w1 + w2 == 3 * wl.H * wl.I * (1 + 1 / 32) == 19_464_192     # MXFP8: 1.03125 B per element
    wl4 = W.WORKLOADS["decode_mxfp4"]
    w1, w2 = bench.weight_bytes_per_expert(wl4)
    assert w1 + w2 == 3 * wl4.H * wl4.I * (0.5 + 1 / 32) == 10_027_008  # MXFP4: 0.53125 B per element
