"""The clocks summary a bench line carries, from synthetic nvidia-smi rows (CPU)."""
import bench

NA = "Not Active"


def row(sm, mx=2070, reasons=(NA, NA, NA, NA)):
    return ", ".join(["0", str(sm), str(mx), "812.50", "0x0000000000000000", *reasons])


def test_steady_clock_no_reason():
    s = bench.summarize_clock_samples([row(2070)] * 6)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 6}


def test_idle_samples_are_left_out_of_the_median():
    s = bench.summarize_clock_samples([row(345), row(2055), row(2070), row(2070), row(600)])
    assert s["sm_mhz"] == 2070.0 and s["samples"] == 5 and "note" not in s


def test_reasons_are_collected():
    rows = [row(1980, reasons=(NA, NA, NA, "Active")), row(2070),
            row(1500, reasons=("Active", NA, "Active", NA))]
    s = bench.summarize_clock_samples(rows)
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_low_clock_without_reason_is_flagged():
    s = bench.summarize_clock_samples([row(1200)] * 5)
    assert s["reasons"] == [] and "note" in s


def test_no_usable_rows():
    assert bench.summarize_clock_samples(["", "garbage", "0, N/A, N/A, 1, 2, 3, 4, 5, 6"])["reasons"] == ["no samples"]
