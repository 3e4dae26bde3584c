"""The bench's clock record: the summary of nvidia-smi samples taken during the timed region,
and the rule that sends a measurement back (thermal or hardware slowdown, or an SM clock held
well below its maximum with no reason -- a leftover clock lock; a power cap alone is kept)."""

import bench


def _clocks(rows):
    c = bench.ClockSampler(0)
    c.rows = rows
    return c.summary()


def _row(sm, mx=2070, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return [str(sm), str(mx), "900.00", hw, hwt, swt, cap]


def test_summary_uses_the_timed_samples():
    rows = [(False, _row(345)), (True, _row(2070)), (True, _row(2055)), (True, _row(2070)), (False, _row(600))]
    s = _clocks(rows)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    assert not bench.clocks_rejected(s)


def test_summary_collects_active_reasons():
    rows = [(True, _row(1900, cap="Active")), (True, _row(1950)), (True, _row(1800, swt="Active"))]
    s = _clocks(rows)
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"] and s["sm_mhz"] == 1900.0


def test_rejection_rule():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    assert not bench.clocks_rejected(ok)
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1600.0, reasons=["sw_power_cap"]))  # kept, noted
    assert bench.clocks_rejected(dict(ok, sm_mhz=1500.0))   # held low with no reason: a lock
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1950.0))
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0})


def test_no_samples():
    assert _clocks([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_prefill_chunks_fit_the_call_limit():
    assert bench.chunk_prefills([100, 200, 300, 50], 400) == [[0, 1], [2, 3]]
    assert bench.chunk_prefills([500], 400) == [[0]]  # a sequence longer than the limit stands alone
    groups = bench.chunk_prefills([1024] * 32, 32768)
    assert groups == [list(range(32))]
