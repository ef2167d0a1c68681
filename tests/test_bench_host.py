"""bench.py's host-side bookkeeping on CPU: the DRAM traffic it reports
from a committed ncu summary (only while that summary was captured on the
current kernel sources), and the clock record it keeps beside each number."""
import os
import tempfile

import pytest

import bench


def _fake_tree(root, source=b"__global__ void k() {}\n"):
    csrc = os.path.join(root, "task_graph_interpreter_gb300", "csrc")
    os.makedirs(csrc, exist_ok=True)
    with open(os.path.join(csrc, "k.cu"), "wb") as f:
        f.write(source)
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)


def _write_profile(root, config, fields):
    with open(os.path.join(root, "profiles", f"dram_traffic_{config}.md"), "w") as f:
        f.write("# DRAM traffic per launch\n\n")
        for k, v in fields.items():
            f.write(f"{k}: {v}\n")
        f.write("\n| metric | value |\n|---|---|\n| traffic | 1 GB |\n")


def test_traffic_scales_the_capture_by_algorithmic_bytes(tmp_path, monkeypatch):
    root = str(tmp_path)
    _fake_tree(root)
    monkeypatch.setattr(bench, "ROOT", root)
    _write_profile(root, "x", {"kernel_source_hash": bench.kernel_source_hash(),
                               "dram_bytes_per_launch": "2010000000", "captured_algorithmic_bytes": "2000000000",
                               "captured_case": "two layers"})
    got, note = bench.profiled_traffic("x", 16e9)
    assert got == pytest.approx(2.01e9 * 8.0)  # traffic grows with the bytes the launch streams
    assert "two layers" in note and "x8.000" in note


def test_traffic_is_null_once_the_kernel_sources_change(tmp_path, monkeypatch):
    root = str(tmp_path)
    _fake_tree(root)
    monkeypatch.setattr(bench, "ROOT", root)
    _write_profile(root, "x", {"kernel_source_hash": bench.kernel_source_hash(),
                               "dram_bytes_per_launch": "1e9", "captured_algorithmic_bytes": "1e9"})
    assert bench.profiled_traffic("x", 1e9)[0] == pytest.approx(1e9)
    _fake_tree(root, source=b"__global__ void k() { /* changed */ }\n")
    assert bench.profiled_traffic("x", 1e9) == (None, None)


def test_traffic_is_null_without_a_usable_summary(tmp_path, monkeypatch):
    root = str(tmp_path)
    _fake_tree(root)
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.profiled_traffic("absent", 1e9) == (None, None)
    _write_profile(root, "broken", {"kernel_source_hash": bench.kernel_source_hash(),
                                    "dram_bytes_per_launch": "not a number", "captured_algorithmic_bytes": "1e9"})
    assert bench.profiled_traffic("broken", 1e9) == (None, None)
    _write_profile(root, "partial", {"kernel_source_hash": bench.kernel_source_hash()})
    assert bench.profiled_traffic("partial", 1e9) == (None, None)


def _summary_of(lines):
    s = bench.ClockSampler(0)
    s.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.f.write("".join(line + "\n" for line in lines))
    return s.summary()


def test_clock_summary_takes_the_median_and_names_throttle_reasons():
    idle = "Not Active"
    rows = [f"0, {mhz}, 2070, 900.5, 0x0, {idle}, {idle}, {idle}, {cap}"
            for mhz, cap in ((2070, idle), (2055, "Active"), (1980, idle))]
    got = _summary_of(rows)
    assert got["sm_mhz"] == 2055 and got["sm_max_mhz"] == 2070 and got["samples"] == 3
    assert got["reasons"] == ["sw_power_cap"]
    hot = _summary_of([f"0, 1500, 2070, 1200, 0x48, Not Active, Active, {idle}, {idle}"])
    assert hot["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples_says_so():
    got = _summary_of(["garbage line"])
    assert got["sm_mhz"] is None and got["reasons"] == ["unavailable"]
