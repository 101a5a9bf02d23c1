"""bench.py's host-side helpers: the clock record's verdict, its parsing of
nvidia-smi lines, and the host CPU's name."""
from __future__ import annotations

import bench


def test_clock_verdicts():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clock_verdict(ok) == "ok"
    assert bench.clock_verdict(dict(ok, reasons=["hw_slowdown"])).startswith("rejected: hw_slowdown")
    assert bench.clock_verdict(dict(ok, reasons=["sw_thermal_slowdown", "sw_power_cap"])).startswith("rejected")
    assert bench.clock_verdict(dict(ok, reasons=["sw_power_cap"], sm_mhz=1500.0)) == "ok (sw_power_cap noted)"
    assert bench.clock_verdict(dict(ok, sm_mhz=1200.0)).startswith("rejected: SM clock 1200")
    assert bench.clock_verdict({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}) == "unsampled"
    assert bench.with_verdict(ok)["verdict"] == "ok" and bench.with_verdict(ok)["sm_mhz"] == 2070.0


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    s.out = ("0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
             "0, 2070, 2070, 1100.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "0, [N/A], 2070, 10.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    summary = s.summary()
    assert summary["samples"] == 2 and summary["sm_max_mhz"] == 2070.0
    assert summary["sm_mhz"] == (1965.0 + 2070.0) / 2
    assert summary["reasons"] == ["sw_power_cap"]
    assert bench.clock_verdict(summary) == "ok (sw_power_cap noted)"


def test_host_cpu_name_is_a_nonempty_string():
    name = bench.host_cpu_name()
    assert isinstance(name, str) and name
