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


@pytest.mark.parametrize("lines,want", [
    (["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"] * 3,
     {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}),
    (["0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
      "0, 1950, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active"],
     {"sm_mhz": 1925.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}),
    (["0, 1200, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active"],
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


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi anywhere
    monkeypatch.setenv("EA_CLOCKS_DIR", str(tmp_path))
    with bench.ClockSampler(0) as cs:
        pass
    assert cs.summary()["reasons"] == ["unavailable"]
