"""Host-side pieces of bench.py that need no GPU: the clock sampler's parsing of nvidia-smi's
CSV output (run against a stand-in nvidia-smi script on PATH) and the throttle reasons it reports."""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _fake_smi(tmp_path, lines):
    d = tmp_path / "bin"
    d.mkdir()
    exe = d / "nvidia-smi"
    body = "\n".join(f"echo '{ln}'" for ln in lines)
    exe.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    return str(d)


TS = "2026/12/02 10:00:00.000"


@pytest.mark.parametrize("lines,want", [
    ([f"{TS}, 0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"] * 3,
     {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}),
    ([f"{TS}, 0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
      f"{TS}, 0, 1950, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active"],
     {"sm_mhz": 1925.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}),
    ([f"{TS}, 0, 1200, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active"],
     {"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"]}),
])
def test_clock_sampler_parses_nvidia_smi_csv(tmp_path, monkeypatch, lines, want):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    monkeypatch.setenv("EA_CLOCKS_DIR", str(tmp_path))
    with bench.ClockSampler(0) as cs:
        time.sleep(0.5)
    got = cs.summary()
    assert cs.path.startswith(str(tmp_path))
    assert {k: got[k] for k in want} == want
    assert got["samples"] == len(lines)


def test_clock_sampler_keeps_only_the_window(tmp_path, monkeypatch):
    # samples before and after the marked window (idle clocks) are left out of the summary
    lines = ["2026/12/02 10:00:00.000, 0, 345, 2070, 90.0, 0x1, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:01.000, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:01.500, 0, 2040, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:02.000, 0, 2070, 2070, 920.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:03.000, 0, 600, 2070, 100.0, 0x8, Active, Not Active, Not Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    monkeypatch.setenv("EA_CLOCKS_DIR", str(tmp_path))
    with bench.ClockSampler(0) as cs:
        time.sleep(0.5)
    t0 = bench.ClockSampler._when("2026/12/02 10:00:00.900")
    t1 = bench.ClockSampler._when("2026/12/02 10:00:02.100")
    got = cs.summary(t0, t1)
    assert got["samples"] == 3 and got["sm_mhz"] == 2070.0 and got["reasons"] == []
    assert got["window_s"] == 1.2


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi anywhere
    monkeypatch.setenv("EA_CLOCKS_DIR", str(tmp_path))
    with bench.ClockSampler(0) as cs:
        pass
    assert cs.summary()["reasons"] == ["unavailable"]
