"""The bench's clock record (CPU only): nvidia-smi lines are kept with their arrival time, and
the summary covers only the samples inside the load window it is given."""

import bench


def line(mhz, power_cap="Not Active", thermal="Not Active"):
    return f"{mhz}, 2070, 900.5, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_summary_keeps_the_window_only():
    c = bench.ClockSampler(0)
    c.lines = [(0.0, line(345)), (1.0, line(2070)), (1.1, line(2055, power_cap="Active")),
               (1.2, line(2070)), (5.0, line(300, thermal="Active"))]
    s = c.summary(0.5, 2.0)
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    every = c.summary()
    assert every["samples"] == 5 and "sw_thermal_slowdown" in every["reasons"]


def test_no_sample_in_the_window_is_said():
    c = bench.ClockSampler(0)
    c.lines = [(0.0, line(2070)), (9.0, "garbled")]
    s = c.summary(1.0, 2.0)
    assert s["samples"] == 0 and s["sm_mhz"] is None
