"""Host-side pieces of the benchmark that need no GPU: the clock summary and the traffic lookup."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _row(sm, smax=2070, reasons=("Not Active",) * 4):
    return ", ".join(["0", str(sm), str(smax), "900.0", "0x0", *reasons])


def test_clock_summary_takes_the_busy_samples_and_flags_throttling():
    idle = [_row(345)] * 3
    busy = [_row(2070), _row(2055), _row(2070), _row(1980, reasons=("Not Active", "Not Active", "Not Active", "Active"))]
    out = bench.parse_clock_samples(idle + busy + ["garbage line", "0, [N/A], 2070, 1, 0, a, b, c, d"])
    assert out["samples"] == 7
    assert out["sm_mhz"] == 2062.5            # median of the four busy samples, idle ones left out
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    hot = bench.parse_clock_samples([_row(1500, reasons=("Active", "Not Active", "Active", "Not Active"))])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples([])["samples"] == 0


def test_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// a kernel\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel_key dram_bytes_per_launch source_sha256_16 source_file\n"
        f"bwd_main 12345 {bench.source_sha(str(src))} kernel.cu\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("bwd_main", str(src)) == 12345.0
    assert bench.measured_traffic("fwd", str(src)) is None
    # a changed source (the counters no longer describe it) gets no traffic figure
    src.write_text("// a kernel, changed\n")
    assert bench.measured_traffic("bwd_main", str(src)) is None
