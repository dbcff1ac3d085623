"""The bench's clock record: nvidia-smi samples reduced to the SM clock under
load and the throttle reasons active during the timed region, with the verdict
that rejects a throttled or clock-locked run. Fed hand-written nvidia-smi rows
(no GPU)."""
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

T0 = time.mktime(time.strptime("2026/12/02 22:00:00", "%Y/%m/%d %H:%M:%S"))


def row(sec, sm, smax=2070, hw="Not Active", hwt="Not Active", swt="Not Active",
        swp="Not Active", power="900.5"):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(T0 + int(sec)))
    frac = f"{sec - int(sec):.3f}"[1:]
    return (f"{stamp}{frac}, 0, {sm}, {smax}, {power}, 0x0000000000000000, {hw}, {hwt}, "
            f"{swt}, {swp}")


def summary(rows, windows=((T0 + 1.0, T0 + 2.0),)):
    return bench.summarise_clocks("\n".join(rows) + "\n", list(windows))


def test_clean_run_at_max_clock():
    s = summary([row(1.1, 2070), row(1.5, 2070), row(1.9, 2055)])
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == [] and s["verdict"] == "ok"
    assert s["samples"] == s["samples_in_timed_region"] == 3


def test_only_samples_inside_the_timed_windows_count():
    """Idle samples well outside the window (low clocks, a slowdown) are left out."""
    rows = [row(0.2, 345, hw="Active"), row(1.2, 2070), row(1.6, 2070), row(3.5, 400)]
    s = summary(rows)
    assert s["samples_in_timed_region"] == 2 and s["sm_mhz"] == 2070
    assert s["verdict"] == "ok"


def test_hardware_and_thermal_slowdowns_reject_the_run():
    s = summary([row(1.2, 1800, hw="Active"), row(1.4, 2070)])
    assert "hw_slowdown" in s["reasons"] and s["verdict"].startswith("rejected")
    s = summary([row(1.2, 1900, hwt="Active")])
    assert s["verdict"] == "rejected: hw_thermal_slowdown"
    s = summary([row(1.2, 1900, swt="Active")])
    assert s["verdict"] == "rejected: sw_thermal_slowdown"


def test_power_cap_is_kept_and_noted():
    s = summary([row(1.2, 1460, swp="Active"), row(1.5, 1470, swp="Active")])
    assert s["reasons"] == ["sw_power_cap"] and s["verdict"] == "ok"
    assert s["sm_mhz"] == 1465


def test_low_clock_with_no_reason_reads_as_a_lock():
    s = summary([row(1.2, 1200), row(1.5, 1200), row(1.8, 1215)])
    assert s["reasons"] == [] and s["verdict"].startswith("rejected")


def test_no_samples_or_garbage():
    assert summary([])["reasons"] == ["no samples"]
    assert summary(["not, a, row"])["reasons"] == ["no samples"]
    s = summary([row(5.0, 2070)])          # nothing in the window: every sample is used
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 1
