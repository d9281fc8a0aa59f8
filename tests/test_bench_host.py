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
