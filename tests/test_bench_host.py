"""Host-side logic of the benchmark, on the CPU: the clock sampler's parsing and
filtering (against a stand-in for nvidia-smi that prints the same CSV fields), and the
launch flags each workload runs with by default."""

import os
import stat
import time

import bench


def _fake_smi(tmp_path, power_cap: str) -> str:
    d = tmp_path / "bin"
    d.mkdir()
    script = d / "nvidia-smi"
    script.write_text(
        "#!/bin/bash\n"
        "while true; do\n"
        "  echo \"$(date '+%Y/%m/%d %H:%M:%S.%3N'), 0, 1980, 2070, 900.5, 0x0, Not Active, "
        f"Not Active, Not Active, {power_cap}\"\n"
        "  sleep 0.02\n"
        "done\n")
    script.chmod(script.stat().st_mode | stat.S_IXUSR)
    return str(d)


def test_clock_sampler_reads_samples_of_the_timed_region(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, "Not Active") + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.3)
    r = c.stop()
    assert r is not None and r["within_region"]
    assert r["samples"] >= 3
    assert r["sm_mhz"] == 1980.0 and r["sm_max_mhz"] == 2070.0 and r["reasons"] == []


def test_clock_sampler_reports_active_throttle_reasons(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, "Active") + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.2)
    r = c.stop()
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))            # no nvidia-smi anywhere
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() is None


def test_default_launch_flags():
    assert bench.LAUNCH_FLAGS[bench.default_launch_flags("llama13b")] == 1 | 2 | 4 | 16
    assert bench.LAUNCH_FLAGS[bench.default_launch_flags("decode7b")] == 1 | 2 | 4 | 16
    assert bench.LAUNCH_FLAGS[bench.default_launch_flags("parallel")] == 1 | 2 | 4 | 16
