"""Host logic of bench.py that needs no GPU: the clock sampler keeps only the nvidia-smi
samples taken inside the timed region and reports the throttle reasons seen there."""
import datetime
import os
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _write_log(path, t0, rows):
    with open(path, "w") as f:
        for dt, mhz, power_cap in rows:
            ts = datetime.datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            cap = "Active" if power_cap else "Not Active"
            f.write(f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}\n")


def test_clock_summary_keeps_the_timed_region():
    import bench
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp()
    os.close(fd)
    t0 = time.time()
    # Outside the region (idle, 2070 MHz) and inside it (1900 MHz, one power-cap sample).
    _write_log(c.path, t0, [(-0.5, 2070, False), (0.01, 1900, False), (0.05, 1900, True),
                            (0.09, 1900, False), (0.6, 2070, False)])
    c.proc = object()
    c.t0, c.t1 = t0, t0 + 0.1
    s = c.summary()
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(c.path)


def test_clock_summary_without_samples_in_region_uses_all():
    import bench
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp()
    os.close(fd)
    t0 = time.time()
    _write_log(c.path, t0, [(-0.5, 2070, False), (0.6, 2070, False)])
    c.proc = object()
    c.t0, c.t1 = t0, t0 + 0.01
    s = c.summary()
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 2
    assert s["sm_mhz"] == 2070.0 and s["reasons"] == []


def test_clock_summary_without_nvidia_smi():
    import bench
    c = bench.ClockSampler(0)
    assert c.summary()["reasons"] == ["nvidia-smi unavailable"]
