"""The benchmark's clock record on CPU, with a stand-in for NVML: only samples
taken inside the timed region count, a region with no sample reports a
null clock instead of falling back to other samples, and the clock-event
reason bits map to the documented names.  No GPU and no NVML library are
involved."""
import ctypes

import pytest

import bench


class _FakeNvml:
    """Answers the three read-only queries the sampler makes, from a script
    of (sm MHz, reason bits, power mW) values."""

    def __init__(self, script):
        self.script = list(script)
        self.i = 0

    def _next(self):
        v = self.script[min(self.i, len(self.script) - 1)]
        return v

    def nvmlDeviceGetClockInfo(self, handle, which, out):
        out._obj.value = self._next()[0]
        return 0

    def reasons(self, handle, out):
        out._obj.value = self._next()[1]
        return 0

    def nvmlDeviceGetPowerUsage(self, handle, out):
        out._obj.value = self._next()[2]
        self.i += 1
        return 0


def _sampler(script):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = []
    s.t_start = s.t_stop = None
    s.error = None
    s.max_mhz = 2070.0
    s._thread = None
    import threading

    s._stop = threading.Event()
    s._lock = threading.Lock()
    s.ct = ctypes
    fake = _FakeNvml(script)
    s.nvml = fake
    s.handle = object()
    s._reasons_fn = fake.reasons
    return s


def test_only_samples_inside_the_timed_region_count(monkeypatch):
    clock = iter([1.0, 2.0, 3.0, 4.0, 5.0])
    monkeypatch.setattr(bench.time, "perf_counter", lambda: next(clock))
    s = _sampler([(1000, 0, 100000), (2070, 0x4, 900000), (2000, 0, 800000),
                  (500, 0x40, 50000)])
    s.sample()          # t = 1: before the region (idle, 1000 MHz)
    s.t_start = 1.5
    s.sample()          # t = 2: inside, power cap active
    s.sample()          # t = 3: inside
    s.t_stop = 3.5
    s.sample()          # t = 4: after (a thermal slowdown that must not count)
    out = s.summary()
    assert out["samples_in_timed_region"] == 2
    assert out["sm_mhz"] == pytest.approx(2035.0)
    assert out["sm_mhz_min"] == 2000.0 and out["sm_mhz_max"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == pytest.approx(900.0)


def test_no_sample_in_the_region_reports_a_null_clock(monkeypatch):
    clock = iter([1.0, 9.0])
    monkeypatch.setattr(bench.time, "perf_counter", lambda: next(clock))
    s = _sampler([(1500, 0x8, 100000)])
    s.sample()
    s.sample()
    s.t_start, s.t_stop = 2.0, 3.0
    out = s.summary()
    assert out["samples_in_timed_region"] == 0
    assert out["sm_mhz"] is None and out["reasons"] == []


def test_reason_bits_map_to_the_documented_names():
    assert bench.ClockSampler.REASONS == {
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


def test_sampler_without_nvml_reports_the_reason():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.handle = None
    s.error = "NVML unavailable: test"
    out = s.summary()
    assert out["sm_mhz"] is None and out["samples_in_timed_region"] == 0
    assert "NVML" in out["error"]
