"""bench.py's clock record: nvidia-smi samples are summarised over the timed window only (host-side
logic, checked on the CPU with a recorded sample file instead of a running nvidia-smi)."""
import datetime
import os
import tempfile

import bench


class _DoneProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _stamp(t):
    return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]


def _sampler_with(lines, window):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = _DoneProcess()
    s.mark(*window)
    return s


def _line(t, mhz, watts, hw="Not Active", power_cap="Not Active"):
    # timestamp, sm, max sm, instantaneous power, active mask, hw, hw thermal, sw thermal, sw power cap
    return f"{_stamp(t)}, {mhz}, 2070, {watts}, 0x0, {hw}, Not Active, Not Active, {power_cap}"


def test_only_samples_inside_the_timed_window_count():
    t0 = 1_800_000_000.0
    lines = [
        _line(t0 - 0.20, 2070, 185.0),                                  # idle, before the window
        _line(t0 + 0.05, 1900, 1410.0, power_cap="Active"),
        _line(t0 + 0.10, 1800, 1420.0, power_cap="Active"),
        _line(t0 + 0.15, 2000, 1390.0),
        _line(t0 + 0.90, 2070, 190.0, hw="Active"),                     # after the window
        "garbage line",
    ]
    s = _sampler_with(lines, (t0, t0 + 0.5))
    rec = s.stop()
    assert not os.path.exists(s.path)
    assert rec["samples"] == 3 and rec["samples_in_window"]
    assert rec["sm_mhz"] == 1900 and rec["sm_mhz_min"] == 1800 and rec["sm_max_mhz"] == 2070
    assert rec["power_w_median"] == 1410.0
    assert rec["reasons"] == ["sw_power_cap"]          # the hw_slowdown sample lies outside


def test_a_window_shorter_than_the_sampling_period_falls_back_to_all_samples():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.04, 2070, 300.0), _line(t0 + 0.06, 2055, 900.0)]
    rec = _sampler_with(lines, (t0, t0 + 0.02)).stop()
    assert rec["samples"] == 2 and not rec["samples_in_window"]
    assert rec["sm_mhz"] == (2070 + 2055) / 2
    assert rec["reasons"] == []


def test_no_nvidia_smi_is_reported_not_invented():
    rec = bench.ClockSampler(0).stop()
    assert rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]
