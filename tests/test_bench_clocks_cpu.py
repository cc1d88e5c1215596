"""The benchmark's clock record (CPU): nvidia-smi samples inside the timed
window give the median SM clock, the maximum clock and the active throttle
reasons; samples outside the window and malformed lines are ignored."""
import datetime
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _line(ts, sm, mx, hw="Not Active", cap="Not Active"):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    # timestamp, index, clocks.sm, clocks.max.sm, power, active, hw, hw_thermal, sw_thermal, sw_power_cap
    return f"{stamp}, 0, {sm}, {mx}, 900.00, 0x0, {hw}, Not Active, Not Active, {cap}"


def _sampler(lines):
    s = bench.ClockSampler(0)
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    f.write("\n".join(lines) + "\n")
    f.flush()
    s.file, s.proc = f, _DoneProc()
    return s


def test_median_clock_and_no_reason_inside_the_window():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1 * i, 2070 if i % 3 else 2055, 2070) for i in range(10)]
    lines.append(_line(t0 + 50.0, 900, 2070, hw="Active"))  # long after the window: ignored
    lines.append("garbage line")
    rec = _sampler(lines).stop(t0, t0 + 1.0)
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == [] and rec["samples"] == 10


def test_throttle_reasons_inside_the_window_are_reported():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1 * i, 1900, 2070, hw="Active" if i == 4 else "Not Active",
                   cap="Active" if i == 6 else "Not Active") for i in range(8)]
    rec = _sampler(lines).stop(t0, t0 + 1.0)
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == 1900.0


def test_no_sampler_process_is_reported():
    s = bench.ClockSampler(0)
    s.proc = None
    rec = s.stop(0.0, 1.0)
    assert rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]
