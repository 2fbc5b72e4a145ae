"""Host-side helpers of bench.py: the default timed-step count and the clock
sample parsing / timed-window filter (no GPU, no nvidia-smi)."""
from __future__ import annotations

import datetime
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_default_steps_fill_the_timed_region():
    b = _bench()
    assert b.resolve_steps(0.2) == 7500           # 1.5 s of 0.2 ms steps
    assert b.resolve_steps(4.0) == 400            # 375 rounded to a hundred
    assert b.resolve_steps(50.0) == 200           # at least 200
    assert b.resolve_steps(0.01) == 10000         # at most 10000
    assert b.resolve_steps(0.0) == 10000          # a zero timing cannot divide by zero


def _line(t: datetime.datetime, sm=2070, mx=2070, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return ", ".join([t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], str(sm), str(mx), "900.0", "0x0"] + flags)


def test_clock_summary_keeps_the_timed_window():
    b = _bench()
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(base + datetime.timedelta(milliseconds=200 * i), sm=(1000 if i in (0, 9) else 2070),
                   reasons=(("sw_power_cap",) if i == 5 else ())) for i in range(10)]
    lines.append("garbage line")
    clk = b.ClockSampler(0)
    clk.lines = lines
    assert len(b.ClockSampler.parse(lines)) == 10
    t0 = (base + datetime.timedelta(milliseconds=100)).timestamp()
    t1 = (base + datetime.timedelta(milliseconds=1700)).timestamp()
    s = clk.summary(t0, t1)
    # samples 1..8 are inside; the idle samples 0 and 9 (1000 MHz) are not
    assert s["in_timed_region"] == 8 and s["samples"] == 8
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    # no sample inside the window: all samples, flagged by in_timed_region = 0
    late = (base + datetime.timedelta(hours=1)).timestamp()
    s2 = clk.summary(late, late + 1)
    assert s2["in_timed_region"] == 0 and s2["samples"] == 10
    assert clk.summary()["samples"] == 10
    empty = b.ClockSampler(0)
    assert empty.summary(t0, t1) is None
    # a timestamp in another format keeps the sample, outside any window
    odd = b.ClockSampler(0)
    odd.lines = ["Tue Jan  1 12:00:00 2026, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s3 = odd.summary(t0, t1)
    assert s3["samples"] == 1 and s3["in_timed_region"] == 0 and s3["sm_mhz"] == 2070


def test_clock_sampler_names_the_physical_gpu():
    """nvidia-smi numbers GPUs physically: device 0 of a process that sees
    CUDA_VISIBLE_DEVICES=5,2 is physical GPU 5, and a UUID list maps to the
    UUID."""
    b = _bench()
    assert b.smi_device(0, "5,2") == "5"
    assert b.smi_device(1, "5, 2") == "2"
    assert b.smi_device(0, "GPU-1234abcd-0000-1111-2222-333344445555") == "GPU-1234abcd-0000-1111-2222-333344445555"
    assert b.smi_device(3, None if False else "") == "3"
    assert b.smi_device(1, "7") == "1"          # more devices than listed: leave the index alone
