"""Host logic of bench.py that the JSON line depends on, on the CPU: the
clock-sample summary (median SM clock, throttle reasons) and the traffic
record lookup, which must drop a record once its kernel source changes."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler_with_rows(tmp_path, rows):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.index = "0"
    s.proc = _FakeProc()
    f = open(tmp_path / "clocks.csv", "w+")
    f.write("\n".join(rows) + "\n")
    s.file = f
    return s


def test_clock_summary_takes_median_and_active_reasons(tmp_path):
    rows = [
        "1965, 2070, 850.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2070, 2070, 1210.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2040, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = _sampler_with_rows(tmp_path, rows).stop()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2040.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_thermal_and_hw_slowdown(tmp_path):
    rows = ["1500, 2070, 1390.0, 0x68, Active, Not Active, Active, Not Active",
            "1490, 2070, 1395.0, 0x68, Not Active, Active, Not Active, Not Active"]
    out = _sampler_with_rows(tmp_path, rows).stop()
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1495.0


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    out = s.stop()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_record_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "kern.cu"
    src.write_text("// kernel v1\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k": {"source": "kern.cu", "source_sha256": h, "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k") == 1234
    assert bench.kernel_traffic("missing") is None
    src.write_text("// kernel v2\n")
    assert bench.kernel_traffic("k") is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    for name, r in records.items():
        assert os.path.exists(os.path.join(ROOT, r["source"])), name
        assert len(r["source_sha256"]) == 64, name
        assert os.path.exists(os.path.join(ROOT, r["profile"])), name
