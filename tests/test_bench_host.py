"""Host logic of the benchmark harness (no GPU): which clock records
disqualify a timed region."""
import bench


def _info(sm, smax=2032, reasons=()):
    return {"sm_mhz": sm, "sm_max_mhz": smax, "reasons": list(reasons), "samples": 20,
            "source": "nvml"}


def test_full_clock_no_reason_is_kept():
    assert not bench.clocks_rejected(_info(2032))
    assert not bench.clocks_rejected(_info(1900))


def test_power_cap_is_kept_even_at_low_clock():
    assert not bench.clocks_rejected(_info(1650, reasons=["sw_power_cap"]))


def test_slowdowns_are_rejected():
    for r in bench.REJECT_REASONS:
        assert bench.clocks_rejected(_info(2032, reasons=[r]))
        assert bench.clocks_rejected(_info(1500, reasons=["sw_power_cap", r]))


def test_clock_held_low_without_reason_is_rejected():
    assert bench.clocks_rejected(_info(1200))
    assert not bench.clocks_rejected(_info(1200), low_frac=0.5)


def test_missing_record_rejects_nothing():
    assert not bench.clocks_rejected(None)
    assert not bench.clocks_rejected({"error": "no NVML samples"})


class _FakeNvml:
    """Stands in for libnvidia-ml: a fixed SM clock and clock-event reason
    mask, written through the ctypes pointers the sampler passes."""

    def __init__(self, clocks, reasons):
        self.clocks = list(clocks)
        self.reasons = reasons
        self.i = 0

    def nvmlDeviceGetClockInfo(self, h, kind, ptr):
        ptr._obj.value = self.clocks[min(self.i, len(self.clocks) - 1)]
        self.i += 1
        return 0

    def reasons_fn(self, h, ptr):
        ptr._obj.value = self.reasons
        return 0


def _sample(monkeypatch, clocks, reasons):
    import time
    fake = _FakeNvml(clocks, reasons)
    s = bench.ClockSampler(0)
    monkeypatch.setattr(s, "_open", lambda: (fake, None, 2032, fake.reasons_fn))
    s.start()
    time.sleep(0.05)
    return s.stop()


def test_sampler_reports_median_clock_and_decodes_reason_bits(monkeypatch):
    info = _sample(monkeypatch, [2032], 0x4 | 0x40)
    assert info["sm_mhz"] == 2032 and info["sm_max_mhz"] == 2032
    assert info["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert info["samples"] >= 1 and info["source"] == "nvml"
    assert bench.clocks_rejected(info)


def test_sampler_without_reasons_keeps_the_run(monkeypatch):
    info = _sample(monkeypatch, [2032], 0)
    assert info["reasons"] == [] and not bench.clocks_rejected(info)


def test_sampler_without_nvml_reports_the_error(monkeypatch):
    s = bench.ClockSampler(0)

    def no_nvml():
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")

    monkeypatch.setattr(s, "_open", no_nvml)
    s.start()
    info = s.stop()
    assert "error" in info and "libnvidia-ml" in info["error"]
    assert not bench.clocks_rejected(info)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle on a bounded sample) prints
    one JSON line with the keys of the benchmark contract."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=root, env=env, check=True, capture_output=True,
                         text=True, timeout=600).stdout.strip().splitlines()
    line = json.loads(out[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TOPS"
    assert line["config"]["workload"] == bench.WORKLOAD
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
