"""bench.py's host logic, without a GPU: the clock summary of the nvidia-smi samples, the rule
that reports a committed profile's DRAM bytes only while its source hash matches, and the
measured-peak loading."""

import json

import bench

# index, clocks.sm, clocks.max.sm, power.draw, clocks_event_reasons.active, hw_slowdown,
# hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap (ClockSampler.QUERY, no units)
ROWS = [
    "0, 1965, 2070, 1180.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 1980, 2070, 1210.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 2010, 2070, 990.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
]


def test_clock_summary_median_max_and_reasons():
    out = bench.summarize_clocks(ROWS)
    assert out == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_each_rejecting_reason_once():
    rows = ROWS + ["0, 1500, 2070, 700.0, 0x48, Active, Not Active, Active, Not Active"] * 2
    out = bench.summarize_clocks(rows)
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert out["samples"] == 5 and out["sm_mhz"] == 1965.0


def test_clock_summary_skips_fields_that_are_not_numbers_and_short_rows():
    rows = ["0, [N/A], 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1900, [N/A], 900, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line", ""]
    out = bench.summarize_clocks(rows)
    assert out == {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}
    assert bench.summarize_clocks(["", "0, 1900"]) is None


def test_profile_bytes_only_while_the_hash_matches(tmp_path, monkeypatch):
    prof = tmp_path / "p.md"
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.profile_traffic() is None  # no profile
    prof.write_text(f"kernel_source_sha256_16: {bench.kernel_hash()}\ndram_bytes_per_launch: 2.5e9\n")
    assert bench.profile_traffic() == 2.5e9
    prof.write_text("kernel_source_sha256_16: 0123456789abcdef\ndram_bytes_per_launch: 2.5e9\n")
    assert bench.profile_traffic() is None  # taken on other sources
    prof.write_text(f"kernel_source_sha256_16: {bench.kernel_hash()}\n")
    assert bench.profile_traffic() is None  # no figure


def test_peaks_come_from_the_measured_file_when_present():
    p = bench.load_peaks()
    assert p["hbm"] > 0 and p["bf16"] > 0 and p["bf16_sustained"] > 0
    if p["source"] == "measured":
        with open(bench.os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        assert p["hbm"] == float(m["hbm_gbs"]) and p["bf16"] == float(m["bf16_tflops"])


def test_sampler_stop_reads_and_removes_its_file(tmp_path):
    # the sampler's stop() with a stand-in for the nvidia-smi process
    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(ROWS) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = Done(), str(path)
    assert s.stop()["sm_mhz"] == 1980.0
    assert not path.exists()
    assert bench.ClockSampler(0).stop() is None  # never started
