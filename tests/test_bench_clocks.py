"""bench.py's clock sampler, against a stand-in for nvidia-smi that prints the
same CSV rows (timestamp first) at the requested interval: only the samples
taken inside the timed region count, and every sampler process ends."""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

FAKE = r'''#!/usr/bin/env python3
import datetime, sys, time
ms = int(sys.argv[sys.argv.index("-lms") + 1])
slow_until = time.time() + float(sys.argv[0].rsplit("_", 1)[1])   # idle clocks first
while True:
    now = datetime.datetime.now()
    sm = 1005 if time.time() < slow_until else 2070
    cap = "Active" if sm == 2070 else "Not Active"
    print(f"{now:%Y/%m/%d %H:%M:%S}.{now.microsecond // 1000:03d}, {sm}, 2070, 905.50, 0x0000000000000004, "
          f"Not Active, Not Active, Not Active, {cap}", flush=True)
    time.sleep(ms / 1000.0)
'''


def _fake(tmp_path, slow_s):
    p = tmp_path / f"fake_smi_{slow_s}"
    p.write_text(FAKE)
    p.chmod(p.stat().st_mode | stat.S_IEXEC)
    return str(p)


def test_only_samples_inside_the_timed_region_count(tmp_path):
    import bench
    clk = bench.ClockSampler(0, interval_ms=20, exe=_fake(tmp_path, 0.4)).start()
    assert clk.proc is not None
    time.sleep(0.6)                 # the idle (1005 MHz) samples come before the region
    clk.mark(True)
    time.sleep(0.4)
    clk.mark(False)
    clk.stop()
    assert clk.proc.poll() is not None
    s = clk.summary()
    assert s["window"] == "timed region"
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert 8 <= s["samples"] <= 40, s
    assert not os.path.exists(clk.path)


def test_missing_tool_reports_unavailable(tmp_path):
    import bench
    clk = bench.ClockSampler(0, exe=str(tmp_path / "no_such_tool")).start()
    clk.mark(True)
    clk.mark(False)
    clk.stop()
    assert clk.summary()["reasons"] == ["unavailable"]
