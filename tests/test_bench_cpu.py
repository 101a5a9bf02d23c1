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


def test_the_value_is_the_slowest_point_with_at_most_16_tokens():
    pts = [{"M": 1, "tbps": 6.0}, {"M": 16, "tbps": 5.5}, {"M": 8, "tbps": 5.7}, {"M": 128, "tbps": 2.7}]
    assert bench.headline(pts) == {"M": 16, "tbps": 5.5}
    assert bench.headline([{"M": 64, "tbps": 4.0}, {"M": 32, "tbps": 5.0}]) == {"M": 64, "tbps": 4.0}


def test_repeats_cover_the_minimum_time_and_at_least_five():
    assert bench.repeats_for(15.0, 40.0) == 5
    assert bench.repeats_for(1.6, 40.0) == 25
    assert bench.repeats_for(0.11, 40.0) == 364
    assert bench.repeats_for(0.0, 40.0) == 5


def test_workload_keys_name_the_workloads_the_bench_accepts():
    from split_bf16_gemm_swapped_gb300 import workloads as W
    for w in list(W.ALL_FIXED) + W.all_sweep():
        assert bench.workload_by_name(bench.workload_key(w)) == w


def test_the_traffic_table_is_read_only_for_the_current_kernel(tmp_path, monkeypatch):
    table = tmp_path / "t.txt"
    table.write_text("# comment\nkernel_sha256: %s\ntraffic sweep_m16_s8: 470900000 B\n"
                     "traffic decode_m1: 29438208\n" % bench.kernel_sha())
    monkeypatch.setattr(bench, "TRAFFIC_TABLE", table)
    assert bench.traffic_table() == {"sweep_m16_s8": 470900000, "decode_m1": 29438208}
    table.write_text("kernel_sha256: 0000\ntraffic decode_m1: 29438208\n")
    assert bench.traffic_table() == {}
