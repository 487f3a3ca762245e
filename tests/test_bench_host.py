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
        for dep in r.get("deps", {}):
            assert os.path.exists(os.path.join(ROOT, dep)), (name, dep)
        assert len(r["source_sha256"]) == 64, name
        assert os.path.exists(os.path.join(ROOT, r["profile"])), name


def test_traffic_record_scaled_and_summed(tmp_path, monkeypatch):
    src = tmp_path / "kern.cu"
    src.write_text("// two kernels\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k": {"source": "kern.cu", "source_sha256": h, "n_tokens": 512,
               "dram_bytes_per_launch": {"a": 100, "b": 300}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k") == 400
    assert bench.kernel_traffic("k", 4096) == 3200


def test_prefill_flop_counts():
    from serving_gdn_decode_gb300.workloads import WORKLOADS
    w = WORKLOADS["long_prefill"]
    # two-pass: 64 chunks x 4 seqs x (48 value heads x 8 x 2^20 + 16 key heads x 2 x 2^20)
    mib = 1 << 20
    assert bench.chunked_mma_flops(w, True) == 64 * 4 * (48 * 8 * mib + 16 * 2 * mib)
    # one-pass: per (value head, chunk) 2 + 1 + 2 + 1 + 2 + 1 + 2 = 11 x 2^20
    assert bench.chunked_mma_flops(w, False) == 64 * 4 * 48 * 11 * mib
    # a ragged last chunk still runs whole products
    assert bench.chunked_mma_flops(w.with_(n_tokens=4095), True) == bench.chunked_mma_flops(w, True)
    # split-bf16 operands: three bf16 products for every one
    for two in (False, True):
        assert bench.chunked_mma_flops(w, two, split=True) == 3 * bench.chunked_mma_flops(w, two)
    # bf16 activations, one pass: per (value head, chunk) 2 + 2 + 4 + 3 + 4 + 3 + 6 = 24 x 2^20
    assert bench.chunked_mma_flops(w, False, split=True, bf16_in=True) == 64 * 4 * 48 * 24 * mib
    # ... two passes: per (value head, chunk) 8 + 3 + 3 + 4 = 18, per (key head, chunk) 2 x 2^20
    assert bench.chunked_mma_flops(w, True, split=True, bf16_in=True) == 64 * 4 * (48 * 18 + 16 * 2) * mib
    assert bench.scan_executed_flops(w) == 6 * 128 * 128 * 48 * 4 * 4096


def test_prefill_roofline_fields():
    from serving_gdn_decode_gb300.workloads import WORKLOADS
    w = WORKLOADS["long_prefill"]
    peaks = {"hbm_gbs": 6700.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}
    r = bench.prefill_roofline("chunked_two_pass_tf32", w, 1e-3, peaks, "measured", {"sm_mhz": 2000.0})
    assert r["bound"] == "tensor" and r["peak"] == 950.0          # TF32: bf16 x 1/2
    assert abs(r["frac"] - r["achieved"] / 950.0) < 2e-3
    assert r["flops_per_call"] == bench.chunked_mma_flops(w, True)
    b = bench.prefill_roofline("chunked_two_pass", w, 1e-3, peaks, "measured", {"sm_mhz": 2000.0})
    assert b["peak"] == 1900.0 and "bf16" in b["flops_counted"]   # split operands: bf16 MMAs
    assert b["flops_per_call"] == 3 * r["flops_per_call"]
    o = bench.prefill_roofline("chunked", w, 1e-3, peaks, "measured", None)
    assert o["flops_per_call"] == bench.chunked_mma_flops(w, False, split=True)
    assert r["hbm_frac"] == round(w.algorithmic_bytes() / 1e-3 / 1e9 / 6700.0, 3)
    s = bench.prefill_roofline("scan", w, 1e-3, peaks, "measured", {"sm_mhz": 2000.0})
    assert s["bound"] == "alu"
    assert abs(s["peak"] - 152 * 128 * 2 * 2000e6 / 1e12) < 0.1
    # no clock samples: the maximum clock, and the record says so
    s2 = bench.prefill_roofline("scan", w, 1e-3, peaks, "measured", None)
    assert abs(s2["peak"] - 152 * 128 * 2 * 2070e6 / 1e12) < 0.1 and "maximum" in s2["peak_kind"]


def test_traffic_record_follows_its_headers(tmp_path, monkeypatch):
    src, dep = tmp_path / "kern.cu", tmp_path / "common.cuh"
    src.write_text("// kernel\n")
    dep.write_text("// shared helpers v1\n")
    h = lambda p: hashlib.sha256(p.read_bytes()).hexdigest()  # noqa: E731
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"k": {"source": "kern.cu", "source_sha256": h(src), "deps": {"common.cuh": h(dep)},
               "dram_bytes_per_launch": 77}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k") == 77
    dep.write_text("// shared helpers v2\n")
    assert bench.kernel_traffic("k") is None
