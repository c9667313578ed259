"""The bench's host records (CPU only): the summary of nvidia-smi samples that
decides whether a timed run saw throttling, and the CPU model beside the
oracle's time."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(lines):
    c = bench.Clocks(0)
    c.proc = object()          # stands for the sampling process
    with open(c.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s = c.summary()
    assert not os.path.exists(c.path)   # the sample file is removed
    return s


def test_power_cap_is_reported_and_clocks_summarised():
    s = _summary([
        "0, 2070, 2070, 900.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 1300.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1380.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_thermal_and_hw_slowdown_are_reported():
    s = _summary([
        "0, 1500, 2070, 700.0, 0x0000000000000048, Active, Not Active, Active, Not Active",
        "0, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",
    ])
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1500.0 and s["sm_max_mhz"] == 2070.0   # the row without numbers is skipped


def test_no_sampler_and_no_samples():
    c = bench.Clocks(0)
    assert c.summary()["reasons"] == ["nvidia-smi unavailable"]
    assert _summary(["garbage"])["reasons"] == ["no samples"]


def test_cpu_model_never_raises(monkeypatch):
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()

    def boom(*a, **k):
        raise OSError("no lscpu")

    monkeypatch.setattr(bench.subprocess, "run", boom)
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()   # /proc/cpuinfo or the machine type
