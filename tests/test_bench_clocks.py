"""bench.py's record of the SM clock and throttle reasons during the timed region, parsed
from nvidia-smi's CSV samples (no GPU needed): the median clock under load, the maximum,
and every throttle reason that was active in any sample."""
import bench


def _sampler(lines):
    c = bench.ClockSampler()
    c.out = "\n".join(lines) + "\n"
    return c.summary()


def test_clean_samples():
    s = _sampler(["2070, 2070, 812.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
                  "2055, 2070, 820.10, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
                  "2070, 2070, 815.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == [] and s["samples"] == 3


def test_reasons_from_any_sample():
    s = _sampler(["1440, 2070, 1391.28, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
                  "1455, 2070, 1388.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
                  "1980, 2070, 1201.00, 0x0000000000000000, Not Active, Active, Not Active, Not Active"])
    assert s["sm_mhz"] == 1455.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_no_samples_is_reported_as_such():
    s = _sampler(["", "garbage"])
    assert s["sm_mhz"] is None and s["reasons"] == ["unsampled"]
