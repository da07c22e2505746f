"""Host-side parts of bench.py that need no GPU: the reference arm's JSON line
(the oracle timed on the host cores) and the clock sampler's parsing of
nvidia-smi lines into a median clock and the set of throttle reasons seen."""
import json
import os
import subprocess
import sys

import bench
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert line["steps"] == 1 and line["warmup"] >= 3          # at least three warm-up steps
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["dtype"] == "f64"
    assert "workload" in line["config"] and "model" not in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


class _FakeProc:
    def __init__(self, lines):
        self.stdout = iter(lines)


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    s._first = type("E", (), {"set": lambda self: None})()
    s._proc = _FakeProc([
        "2032, 2032, Not Active, Not Active, Not Active, Not Active\n",
        "1965, 2032, Not Active, Not Active, Not Active, Active\n",
        "garbage line\n",
        "[N/A], 2032, Not Active, Not Active, Not Active, Not Active\n",
        "1890, 2032, Active, Not Active, Not Active, Active\n",
    ])
    s._smi_read()
    out = s.summary()
    assert out["samples"] == 3 and out["sm_max_mhz"] == 2032.0
    assert out["sm_mhz"] == 1965.0
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_sampler_without_samples_reports_none():
    out = bench.ClockSampler(0).summary()
    assert out["sm_mhz"] is None and out["reasons"] == [] and out["samples"] == 0


def test_traffic_record_is_used_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """Recorded DRAM counters count for the headline only while the kernel file
    and the library headers are unchanged; a changed source gives null."""
    rel = "global_attention_sinks_swa_b300/csrc/prefill_swa.cu"
    assert bench.source_sha(rel) == bench.source_sha(rel)
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    entry = rec["prefill_swa_stream_kernel"]
    assert bench.ncu_traffic(rel, "prefill_swa_stream_kernel") == (
        float(entry["dram_bytes_per_launch"]) if entry["source_sha"] == bench.source_sha(rel)
        else None)
    # a copy of the tree whose kernel file differs by one byte: the record is stale
    root = tmp_path / "tree"
    csrc = root / "global_attention_sinks_swa_b300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "profiles").mkdir()
    src_dir = os.path.join(ROOT, "global_attention_sinks_swa_b300", "csrc")
    for f in os.listdir(src_dir):
        data = open(os.path.join(src_dir, f), "rb").read()
        if f == "prefill_swa.cu":
            data += b"\n"
        (csrc / f).write_bytes(data)
    (root / "profiles" / "traffic.json").write_text(json.dumps(
        {"prefill_swa_stream_kernel": dict(entry, source_sha=bench.source_sha(rel))}))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.ncu_traffic(rel, "prefill_swa_stream_kernel") is None


class _FakeNvmlLib:
    """The NVML C entry points the ctypes reader calls, answering like a GPU at
    1965 of 2032 MHz under a power cap."""

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, index, handle_ref):
        handle_ref._obj.value = 1234
        return 0

    def nvmlDeviceGetClockInfo(self, handle, kind, out_ref):
        out_ref._obj.value = 1965
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, kind, out_ref):
        out_ref._obj.value = 2032
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle, out_ref):
        out_ref._obj.value = 0x4 | 0x1   # sw power cap + idle
        return 0


def test_clock_sampler_reads_nvml_through_ctypes():
    nvml = bench.CtypesNvml(lib=_FakeNvmlLib())
    s = bench.ClockSampler(0)
    s._start_nvml(nvml, "nvml-ctypes")
    s._stop.set()
    s._thread.join(timeout=2)
    s._nvml_once()
    out = s.summary()
    assert out["source"] == "nvml-ctypes" and out["sm_max_mhz"] == 2032.0
    assert out["sm_mhz"] == 1965.0 and out["reasons"] == ["sw_power_cap"]


def test_ctypes_nvml_raises_on_an_error_code():
    class Bad(_FakeNvmlLib):
        def nvmlInit_v2(self):
            return 9   # NVML_ERROR_DRIVER_NOT_LOADED
    with pytest.raises(RuntimeError):
        bench.CtypesNvml(lib=Bad()).nvmlInit()
