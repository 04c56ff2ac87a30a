"""The bench's clock sampler, on the CPU: a fake NVML library and a fake nvidia-smi process
stand in for the driver.  Only samples taken inside the timed region may count, and the
clock-event reason bits map to the names the bench reports."""

import io
import time

import bench


class FakeNvml:
    """The few NVML calls the sampler makes; values are written through the byref args."""

    def __init__(self, sm=1965, mx=2070, bits=0x4):
        self.sm, self.mx, self.bits = sm, mx, bits
        self.calls = 0
        self.shut = False

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        assert kind == 1  # NVML_CLOCK_SM
        self.calls += 1
        out._obj.value = self.sm
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = self.mx
        return 0

    def reasons(self, h, out):
        out._obj.value = self.bits
        return 0

    def nvmlShutdown(self):
        self.shut = True
        return 0


def _with_fake_nvml(monkeypatch, lib):
    import ctypes

    def fake_open(self):
        self.nvml = (lib, ctypes.c_void_p(), lib.reasons, ctypes)
        return True

    monkeypatch.setattr(bench.ClockSampler, "_nvml_open", fake_open)


def test_nvml_samples_inside_the_region(monkeypatch):
    lib = FakeNvml(sm=1965, mx=2070, bits=0x4 | 0x40)
    _with_fake_nvml(monkeypatch, lib)
    c = bench.ClockSampler(0)
    with c:
        time.sleep(0.12)
    s = c.summary()
    assert s["source"].startswith("nvml")
    assert s["samples"] >= 3 and lib.calls >= s["samples"]
    assert s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert lib.shut


def test_samples_outside_the_region_do_not_count(monkeypatch):
    lib = FakeNvml(sm=2070, bits=0)
    _with_fake_nvml(monkeypatch, lib)
    c = bench.ClockSampler(0)
    with c:
        time.sleep(0.05)
    # a sample before the region and one after it, with other values
    c.samples.insert(0, (c.t0 - 1.0, 500.0, 2070.0, ["hw_slowdown"]))
    c.samples.append((c.t1 + 1.0, 600.0, 2070.0, ["sw_thermal_slowdown"]))
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["reasons"] == []


def test_nvidia_smi_fallback(monkeypatch):
    monkeypatch.setattr(bench.ClockSampler, "_nvml_open", lambda self: False)
    lines = ("0, 1800, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active\n"
             "0, 1750, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n")

    def slow_lines():  # one line every 10 ms, as nvidia-smi prints them over time
        for line in io.StringIO(lines):
            time.sleep(0.01)
            yield line

    class Proc:
        def __init__(self, *a, **k):
            self.stdout = slow_lines()

        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    monkeypatch.setattr(bench.subprocess, "Popen", Proc)
    c = bench.ClockSampler(0)
    with c:
        time.sleep(0.1)
    s = c.summary()
    assert s["source"].startswith("nvidia-smi")
    assert s["samples"] == 2 and s["sm_mhz"] == 1775 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_no_driver_reports_no_samples(monkeypatch):
    monkeypatch.setattr(bench.ClockSampler, "_nvml_open", lambda self: False)

    def no_smi(*a, **k):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    c = bench.ClockSampler(0)
    with c:
        pass
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["source"] is None
