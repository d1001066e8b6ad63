"""The bench's clock record: samples taken during the timed region, throttle reasons by name, and
the GEMMs' own clock counters read from the trace region.

NVML is replaced by a fake reader (no GPU here); the sampler must keep polling it for as long as
the timed region lasts and name every clock event reason any sample carried.
"""
import itertools
import time

import bench


def fake_reader(readings):
    it = itertools.cycle(readings)
    return lambda: next(it)


def test_samples_cover_a_short_timed_region():
    with bench.ClockSampler(0, reader=fake_reader([(1710.0, 2070.0, 0x4, 1395.0)])) as clk:
        time.sleep(0.05)
    s = clk.summary()
    assert s["source"] == "reader"
    assert s["samples"] >= 5  # a 50 ms region at a 2 ms period
    assert s["sm_mhz"] == 1710.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1395.0


def test_reasons_are_named_by_their_nvml_bits():
    readings = [(2070.0, 2070.0, 0x0, 900.0), (1500.0, 2070.0, 0x8 | 0x40, 1000.0),
                (1600.0, 2070.0, 0x20, 1000.0), (1900.0, 2070.0, 0x1, 300.0)]  # 0x1 = idle, not reported
    with bench.ClockSampler(0, reader=fake_reader(readings)) as clk:
        time.sleep(0.05)
    s = clk.summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz_min"] == 1500.0 and s["sm_mhz_distinct"] == 4


def test_a_clock_lock_is_named():
    with bench.ClockSampler(0, reader=fake_reader([(1200.0, 2070.0, 0x2, 500.0)])) as clk:
        time.sleep(0.02)
    assert clk.summary()["reasons"] == ["applications_clocks_setting"]


def test_a_reader_that_fails_leaves_the_record_unsampled():
    def broken():
        raise RuntimeError("NVML call failed")
    with bench.ClockSampler(0, reader=broken) as clk:
        time.sleep(0.01)
    assert clk.summary()["reasons"] == ["unsampled"]


class _FakeWorkspace:
    """A workspace whose trace region is a host tensor (the bench's clock-counter helpers only view
    it)."""

    def __init__(self, values):
        import torch
        self.trace = torch.tensor(values, dtype=torch.int64)

    def view(self, name):
        assert name == "trace"
        return self.trace


def test_kernel_clocks_from_the_trace_counters():
    """Slots 8-11 hold (SwiGLU cycles, ns, down-projection cycles, ns): the mean clock is cycles per
    microsecond; a GEMM with no recorded span reads None, and zeroing touches those four slots only."""
    ws = _FakeWorkspace([7] * 8 + [1_700_000, 1_000_000, 0, 0] + [9] * 4)
    got = bench.kernel_clocks(ws)
    assert got["swiglu_gemm"] == 1700.0 and got["down_projection"] is None
    bench.zero_kernel_clocks(ws)
    assert ws.trace.tolist() == [7] * 8 + [0, 0, 0, 0] + [9] * 4
