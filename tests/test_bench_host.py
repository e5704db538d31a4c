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


def test_traffic_record_only_for_the_measured_kernel_sources(tmp_path, monkeypatch):
    """A stored ncu traffic figure is reported only while the kernel sources hash to the
    version it was measured on."""
    import shutil
    src = tmp_path / "paged_kv_cache_169_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in bench.KERNEL_SRCS:
        shutil.copy(os.path.join(bench.ROOT, "paged_kv_cache_169_gb300", "csrc", f), src / f)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_sources_hash()
    assert len(h) == 16
    (tmp_path / "profiles" / "traffic_w.txt").write_text(
        f"# test\nsource_sha256_16: {h}\ndram_bytes_per_launch: 1234\n")
    assert bench.traffic_record("w") == 1234.0
    assert bench.traffic_record("other") is None
    with open(src / bench.KERNEL_SRCS[0], "a") as f:
        f.write("// changed\n")
    assert bench.traffic_record("w") is None
