"""Host-side pieces of bench.py that need no GPU: the clock-record summary
(median SM clock under load, throttle reasons), the NVML sampler's per-region
windows (driven by a stand-in for the NVML library, read-only queries only),
and the reference arm's JSON line (the fp64 oracle on a few rows)."""
import json
import time

import pytest


def test_summarize_clocks_median_under_load_and_reasons():
    import bench
    # (time, sm MHz, max MHz, power W, reasons): the idle samples (low power) are left out
    samples = [(0.0, 2070.0, 2070.0, 100.0, set()),
               (0.1, 1700.0, 2070.0, 1380.0, {"sw_power_cap"}),
               (0.2, 1750.0, 2070.0, 1390.0, set()),
               (0.3, 1800.0, 2070.0, 1385.0, {"sw_power_cap"})]
    c = bench.summarize_clocks(samples)
    assert c["sm_mhz"] == 1750.0
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 4 and c["power_w_max"] == 1390.0
    assert bench.summarize_clocks([])["reasons"] == ["no samples"]


class _FakeNvml:
    """Stands in for libnvidia-ml: a fixed device, clock 1800 MHz, 1200 W,
    the software power cap active."""

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, index, handle):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, kind, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, dev, kind, out):
        out._obj.value = 1800
        return 0

    def nvmlDeviceGetPowerUsage(self, dev, out):
        out._obj.value = 1200000
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, out):
        out._obj.value = 0x4
        return 0

    def nvmlShutdown(self):
        return 0


def test_nvml_sampler_windows(monkeypatch):
    import ctypes

    import bench
    monkeypatch.setattr(ctypes, "CDLL", lambda name: _FakeNvml())
    s = bench.NvmlClockSampler(0, period_s=0.001).start()
    time.sleep(0.02)
    t0 = s.mark()
    time.sleep(0.02)
    t1 = s.mark()
    win = s.window(t0, t1)
    assert win["sm_mhz"] == 1800.0 and win["sm_max_mhz"] == 2070.0
    assert win["reasons"] == ["sw_power_cap"] and win["samples"] >= 1
    # a region shorter than the polling period falls back to the first sample after it
    time.sleep(0.02)
    late = s.window(t1 + 1e-9, t1 + 2e-9)
    full = s.stop()
    assert full["samples"] >= win["samples"]
    assert "note" in late and late["samples"] == 1 and late["sm_mhz"] == 1800.0


def test_reference_arm_line(tmp_path):
    """bench.py --impl reference: the oracle on a few rows per step, one JSON
    line with the keys the driver reads."""
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    json.dumps(line)
