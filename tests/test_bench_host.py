"""Host-side pieces of bench.py: the parse of the clock samples taken during the timed region."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_samples_give_the_median_and_the_active_reasons():
    lines = [
        "0, 2070, 2070, 812.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 2055, 2070, 1391.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 1980, 2070, 1399.80, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, [N/A], 2070, 10.00, 0x0, Not Active, Not Active, Not Active, Not Active\n",  # skipped
        "short, line\n",
        "\n",
    ]
    got = bench.ClockSampler.parse(lines)
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "samples": 3,
                   "reasons": ["sw_power_cap"]}


def test_throttle_reasons_are_all_reported():
    lines = ["0, 1500, 2070, 1400, 0x68, Active, Active, Active, Not Active\n"]
    got = bench.ClockSampler.parse(lines)
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_no_usable_sample_gives_none():
    assert bench.ClockSampler.parse([]) is None
    assert bench.ClockSampler.parse(["0, N/A, N/A, N/A, N/A, N/A, N/A, N/A, N/A\n"]) is None
