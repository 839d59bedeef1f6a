"""The benchmark's clock record from nvidia-smi's CSV samples, on the host: the median SM clock of the
samples inside the timed window, the maximum clock, the throttle reasons that were active and the peak
power draw."""
import os
import tempfile
import time

import bench


def _sampler(rows):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(prefix="tpmlp_clocks_test_", suffix=".csv")
    os.close(fd)
    with open(s.path, "w") as fh:
        for r in rows:
            fh.write(", ".join(r) + "\n")
    s.proc = object()  # a sampler that ran
    return s


def _stamp(t):
    return time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int((t % 1) * 1000)


def _row(t, sm, power, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    return [_stamp(t), str(sm), "2070", str(power), "0x0", hw, hw_th, sw_th, cap]


def test_median_clock_and_reasons_inside_the_window():
    t0 = time.time()
    rows = [_row(t0 - 5, 2070, 100)]                                   # before the window
    rows += [_row(t0 + 0.2 * i, mhz, 900 + i, cap="Active" if i == 2 else "Not Active")
             for i, mhz in enumerate([1500, 1550, 1600, 1650, 1700])]
    rows += [_row(t0 + 10, 990, 50, hw="Active")]                      # after the window
    out = _sampler(rows).summary(t0, t0 + 1.0)
    assert out["sm_mhz"] == 1600
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 5
    assert out["power_w_max"] == 904


def test_window_without_samples_uses_the_last_ones():
    t0 = time.time()
    rows = [_row(t0 - 30 + i, 1800 + 10 * i, 500, hw="Active" if i == 4 else "Not Active") for i in range(5)]
    out = _sampler(rows).summary(t0, t0 + 1.0)
    assert out["samples"] == 3 and out["sm_mhz"] == 1830
    assert out["reasons"] == ["hw_slowdown"]


def test_no_sampler_is_reported():
    s = bench.ClockSampler(0)
    assert s.summary()["reasons"] == ["nvidia-smi unavailable"]
