"""The bench's rule for rejecting a timed region by its clock samples: a
hardware or thermal slowdown, or SM clocks well below their maximum with no
reason reported (a leftover clock lock); power capping alone is kept."""
import bench


def test_clean_and_power_capped_regions_are_kept():
    assert not bench.clocks_rejected({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []})
    assert not bench.clocks_rejected({"sm_mhz": 1492, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"]})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]})


def test_slowdowns_and_unexplained_low_clocks_are_rejected():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": [r]})
    assert bench.clocks_rejected({"sm_mhz": 1200, "sm_max_mhz": 2070, "reasons": []})
