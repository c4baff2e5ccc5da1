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


def test_peak_is_burst_only_at_full_clock():
    held = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    v, how = bench.clock_adjusted(1914.7, held, "bf16")
    assert v == 1914.7 and "burst" in how
    low = {"sm_mhz": 1447.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    v, how = bench.clock_adjusted(1914.7, low, "bf16")
    assert abs(v - 1914.7 * 1447.0 / 2070.0) < 1e-9 and "1447/2070" in how
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.clock_adjusted(100.0, capped, "x")[0] == 100.0  # scaled by 1.0, but the reason is named
    v, how = bench.clock_adjusted(5.0, {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}, "x")
    assert v == 5.0 and "no clock record" in how


def test_run_peaks_measured_fp8_and_fallback():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    held = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    pk = bench.run_peaks(peaks, "measured", held, {"fp8_tflops": 3500.0})
    assert pk["bf16"] == 1900.0 and pk["fp8"] == 3500.0 and pk["fp8_derived"] == 3800.0
    assert "measured fp8" in pk["fp8_how"] and pk["bf16_sustained"] == 1700.0 and pk["hbm"] == 6800.0
    pk = bench.run_peaks(peaks, "measured", held, {"fp8_tflops": None})
    assert pk["fp8"] == 3800.0 and pk["fp8_how"].startswith("derived")


def test_stage_records_fractions():
    pk = {"bf16": 2000.0, "bf16_how": "b", "fp8": 4000.0, "fp8_how": "f", "fp8_derived": 4000.0,
          "bf16_sustained": 1600.0, "hbm": 8000.0}
    work = bench.prefill_work(4096, 2048, 64, 128, 128)
    r = bench.stage_records(work, [1.0, 0.5, 2.0], 4096, pk)
    assert abs(r["indexer"]["frac"] - work["indexer_flop"] / 1e-3 / 1e12 / 4000.0) < 1e-12
    assert abs(r["topk"]["frac"] - work["topk_bytes"] / 0.5e-3 / 1e9 / 8000.0) < 1e-12
    assert abs(r["sparse_mla"]["frac_sustained"] - work["mla_flop"] / 2e-3 / 1e12 / 1600.0) < 1e-12
    assert r["sparse_mla"]["tokens_per_s"] == 4096 / 2e-3
