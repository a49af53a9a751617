"""Host-side logic of bench.py that needs no GPU: the clock record keeps the
nvidia-smi samples taken inside the timed region and reports their median
and throttle reasons (all samples when none fell inside)."""
import datetime
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines, t0, t1):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(c.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    c.f = open(c.path, "a")
    c.proc = _Proc()
    c.t0, c.t1 = t0, t1
    return c


def _line(ts, mhz, cap="Not Active", thermal="Not Active"):
    return (f"{ts.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {mhz}, 2032, 900.0, 0x0, "
            f"Not Active, Not Active, {thermal}, {cap}")


def test_clock_record_uses_the_timed_region():
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(base, 900), _line(base + 50 * ms, 1900, cap="Active"),
             _line(base + 100 * ms, 1880, cap="Active"), _line(base + 150 * ms, 1870),
             _line(base + 400 * ms, 600, thermal="Active")]
    r = _sampler(lines, base + 40 * ms, base + 160 * ms).stop()
    assert r["samples"] == 5 and r["samples_in_timed_region"] == 3
    assert r["sm_mhz"] == 1880 and r["sm_max_mhz"] == 2032
    assert r["reasons"] == ["sw_power_cap"]  # the thermal sample lies outside the region


def test_clock_record_falls_back_to_all_samples():
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(base, 1000), _line(base + 50 * ms, 2000)]
    r = _sampler(lines, base + 10 * ms, base + 20 * ms).stop()
    assert r["samples_in_timed_region"] == 0 and r["sm_mhz"] == 1500
