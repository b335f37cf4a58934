"""The benchmark's clock record: nvidia-smi samples taken during the timed region become the
line's `clocks`, and a record with a hardware or thermal slowdown, or with SM clocks well
below their maximum and no reason given, sends the region to be measured once more."""
import bench


def summary_of(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s.summary()


def sample(sm, mx=2070, hw="Not Active", hw_th="Not Active", sw_th="Not Active",
           cap="Not Active"):
    return f"{sm}, {mx}, 950.12, 0x0000000000000000, {hw}, {hw_th}, {sw_th}, {cap}"


def test_steady_clocks_stand():
    s = summary_of([sample(2070)] * 6 + ["garbage line"])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 6}
    assert bench.clocks_rejected(s) is None


def test_idle_samples_do_not_pull_the_median_down():
    s = summary_of([sample(345)] * 2 + [sample(2070)] * 5)
    assert s["sm_mhz"] == 2070.0 and bench.clocks_rejected(s) is None


def test_power_cap_is_kept_and_reported():
    s = summary_of([sample(1800, cap="Active")] * 4)
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.clocks_rejected(s) is None


def test_slowdowns_are_rejected():
    for kw, name in ((dict(hw="Active"), "hw_slowdown"),
                     (dict(hw_th="Active"), "hw_thermal_slowdown"),
                     (dict(sw_th="Active"), "sw_thermal_slowdown")):
        s = summary_of([sample(2070)] * 3 + [sample(1500, **kw)])
        assert bench.clocks_rejected(s) == name


def test_clocks_held_low_without_a_reason_are_rejected():
    s = summary_of([sample(1400)] * 5)
    assert "no reason" in bench.clocks_rejected(s)


def test_no_samples_leave_the_number_standing():
    s = summary_of([])
    assert s["sm_mhz"] is None and bench.clocks_rejected(s) is None
