"""Host logic of the benchmark's clock record: nvidia-smi samples are parsed with their
timestamps and only those taken inside the timed region are summarised (no GPU needed)."""
import datetime
import importlib.util
import os
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _line(t, sm, reasons=()):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if n in reasons else "Not Active"
             for n in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    return ", ".join([ts, "0", str(sm), "2070", "1100.00", "0x0"] + flags)


def test_only_samples_inside_the_timed_region_count():
    b = _bench()
    c = b.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now, now + 1.0
    c.lines = [_line(now - 2.0, 900, ("hw_slowdown",)),          # before the region: ignored
               _line(now + 0.1, 2070, ("sw_power_cap",)),
               _line(now + 0.6, 2010),
               _line(now + 0.9, 2040),
               _line(now + 3.0, 1000, ("hw_thermal_slowdown",)),  # after it: ignored
               "not a sample"]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2040.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["window"] == "timed region"


def test_short_region_falls_back_to_all_samples():
    b = _bench()
    c = b.ClockSampler(0)
    now = time.time()
    c.t0, c.t1 = now + 10.0, now + 10.01
    c.lines = [_line(now, 1980), _line(now + 0.05, 2000, ("hw_slowdown",))]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1990.0
    assert s["reasons"] == ["hw_slowdown"]
    assert s["window"].startswith("whole sampler run")


def test_no_samples_reads_unsampled():
    b = _bench()
    c = b.ClockSampler(0)
    c.t0, c.t1 = time.time(), time.time() + 1.0
    c.lines = ["garbage", ""]
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
