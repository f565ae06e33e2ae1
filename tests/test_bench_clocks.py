"""The bench's clock record of the timed region (CPU only: a fake stands in for
NVML's read-only queries).  The poller samples between start() and stop(),
reports the median SM clock and every clock-event reason it saw, and the
record falls back to nvidia-smi's when NVML cannot be read."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_poller_reports_median_clock_and_reasons():
    script = [(2070, 2070, 0, 900_000), (1950, 2070, 0x4, 1_390_000), (2070, 2070, 0, 950_000)]
    calls = {"n": 0}

    def reader():
        v = script[min(calls["n"], len(script) - 1)]
        calls["n"] += 1
        return v

    p = bench.NvmlClockPoller(period=0.001, reader=reader).start()
    time.sleep(0.02)
    p.stop()
    rec = p.summary()
    assert rec["samples"] == calls["n"] >= 3
    assert rec["sm_mhz"] == 2070 and rec["sm_min_mhz"] == 1950 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"]
    assert rec["power_w_max"] == 1390.0


def test_reason_bits_map_to_the_rejecting_names():
    p = bench.NvmlClockPoller(reader=lambda: (1200, 2070, 0x8 | 0x20 | 0x40, 500_000))
    p.start()
    p.stop()
    assert p.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_record_falls_back_to_nvidia_smi_without_nvml():
    class Sampler:
        def summary(self):
            return {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 6}

    p = bench.NvmlClockPoller.__new__(bench.NvmlClockPoller)
    p.samples, p.reader, p._thread = [], None, None
    assert p.start() is p
    p.stop()
    assert bench.clock_record(p, Sampler())["samples"] == 6
    assert bench.clock_record(None, Sampler())["sm_mhz"] == 2070.0
