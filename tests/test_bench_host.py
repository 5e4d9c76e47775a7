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


def test_gateup_algorithmic_bytes():
    """Touched experts' W1 (codes + scales), each activation row once, h once."""
    wl = W.WORKLOADS["decode_mxfp8"]
    w1, _ = bench.weight_bytes_per_expert(wl)
    got = bench.gateup_algorithmic_bytes(wl, 113)
    assert got == 113 * w1 + 32 * 4096 * 1.03125 + 32 * 9 * 1536 * 1.03125


def test_both_arms_describe_the_workload_alike():
    for name, wl in W.WORKLOADS.items():
        a, b = bench.config_of(wl, 1), bench.config_of(W.WORKLOADS[name], 1)
        assert a == b and a["workload"] == name and a["T"] == wl.T
    assert bench.config_of(W.WORKLOADS["prefill_mxfp8"], 1)["router_bias"] != "none"


class _Runner:
    def __init__(self, wl, ids):
        self.wl, self.ids = wl, ids


def test_reference_plan_keeps_the_whole_batch_when_it_fits():
    import numpy as np

    wl = W.WORKLOADS["decode_mxfp8"]
    rng = np.random.default_rng(0)
    ids = np.stack([rng.choice(wl.E, wl.k, replace=False) for _ in range(wl.T)])
    r = _Runner(wl, ids)
    assert bench.reference_plan(1.0, wl.T, r, steps=20, budget_s=180) == wl.T
    n = bench.reference_plan(11.0, wl.T, r, steps=100, budget_s=180)
    assert 1 <= n < wl.T
    touched = len(set(ids[:n].ravel().tolist()) | {wl.E})
    touched_full = len(set(ids.ravel().tolist()) | {wl.E})
    assert 100 * 11.0 * touched / touched_full <= 180 or n == 1


def test_reference_arm_line(tmp_path):
    """The reference arm on the tiny workload: same config as the GPU arm, every
    step one whole-batch oracle call, ms_per_step x steps = oracle time spent."""
    import subprocess

    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "3",
                        "--warmup", "2"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][-1])
    assert line["config"] == bench.config_of(W.WORKLOADS["tiny"], 1)
    assert line["tokens_per_step"] == 16 and line["steps"] == 3
    spent = float(line["cpu_baseline"]["sample"].split(" s of oracle time")[0].split()[-1])
    assert abs(line["ms_per_step"] * 3 / 1e3 - spent) <= 0.05 + 0.01 * spent
    assert abs(line["value"] - 3 * 16 / (line["ms_per_step"] * 3 / 1e3)) <= 1e-6 * line["value"]
