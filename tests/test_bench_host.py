"""Host-side parts of bench.py that need no GPU: the clock-sample parsing behind the
throttle check, and the CPU baseline's oracle sample (CPU)."""
import io

import bench
import dsa_workloads as W


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = _FakeProc()
    s.out = io.StringIO("\n".join(lines) + "\n")
    return s


def test_clock_samples_median_max_and_reasons():
    ok = "0, {sm}, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, {pc}"
    lines = [ok.format(sm=1950, pc="Not Active"), ok.format(sm=2070, pc="Active"), ok.format(sm=2010, pc="Not Active"),
             "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
             "garbage"]
    r = _sampler(lines).stop()
    assert r["samples"] == 3 and r["sm_mhz"] == 2010 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_samples_flag_slowdowns():
    line = "0, 1200, 2070, 1300.0, 0x8, Active, Not Active, Active, Not Active"
    r = _sampler([line]).stop()
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    r = s.stop()
    assert r["samples"] == 0 and r["reasons"] == ["nvidia-smi unavailable"]


def test_cpu_baseline_on_tiny_inputs():
    cfg = W.CONFIGS["tiny"]
    x = W.prefill_inputs(cfg, "cpu")
    r = bench.cpu_baseline(cfg, x)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["value"] > 0 and r["cores"] >= 1
    assert r["extrapolated_seconds_per_step"] > 0 and "query rows" in r["sample"]
