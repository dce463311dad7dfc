"""The benchmark's clock record, on the CPU against a fake NVML: the median
SM clock over the samples, the maximum clock, and every throttle reason seen
in any sample (a run that saw a thermal or hardware slowdown must say so)."""
import time

import bench


class FakeNVML:
    """Answers the two read-only queries the sampler makes, from a script of
    (SM MHz, reason bits) samples; the last one repeats."""

    def __init__(self, script):
        self.script = list(script)
        self.i = 0

    def nvmlDeviceGetClockInfo(self, handle, kind, p_mhz):
        p_mhz._obj.value = self.script[min(self.i, len(self.script) - 1)][0]

    def reasons(self, handle, p_bits):
        p_bits._obj.value = self.script[min(self.i, len(self.script) - 1)][1]
        self.i += 1


def sampler(script, max_mhz=2070):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    fake = FakeNVML(script)
    s.ok, s.samples, s.period = True, [], 0.001
    s.nv, s.h, s.max_mhz, s._reasons = fake, None, max_mhz, fake.reasons
    return s


def test_median_clock_and_no_reasons():
    s = sampler([(2070, 0), (2070, 0), (1980, 0), (2070, 0), (2055, 0)])
    for _ in range(5):
        s._sample()
    got = s.summary()
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == [] and got["samples"] == 5 and got["source"] == "nvml"


def test_every_reason_seen_in_any_sample_is_reported():
    s = sampler([(2070, 0), (1800, 0x4), (1500, 0x40 | 0x8), (2070, 0), (1900, 0x20)])
    for _ in range(5):
        s._sample()
    got = s.summary()
    assert got["reasons"] == sorted(["sw_power_cap", "hw_thermal_slowdown", "hw_slowdown",
                                     "sw_thermal_slowdown"])
    assert got["sm_mhz"] == 1900.0


def test_background_sampling_brackets_the_region():
    s = sampler([(2070, 0)])
    with s:
        time.sleep(0.03)
    got = s.summary()
    # one sample on entry, at least one in the loop, one on exit
    assert got["samples"] >= 3 and got["reasons"] == []


def test_no_nvml_means_no_clock_record():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.ok, s.samples = False, []
    with s:
        pass
    assert s.summary() is None
