"""Host-side pieces of the benchmark's JSON line, without a GPU: the clock summary that
rejects throttled runs, and the decode roofline object."""
import bench


def test_clock_summary_takes_the_median_and_the_active_throttle_reasons():
    c = bench.Clocks(0)
    c.out = "\n".join([
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1100.5, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ])
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_of_no_samples_is_empty():
    c = bench.Clocks(0)
    c.out = ""
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_decode_roofline_is_algorithmic_bytes_over_time_against_the_peak():
    r = bench.roofline_decode({"launches": 1}, 2_000_000_000, 2000.0, 6800.0, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"] == "mega_decode_kernel"
    assert abs(r["frac"] - 2000.0 / 6800.0) < 1e-4
    assert r["traffic"] == round(2_000_000_000 * bench.MEGA_TRAFFIC_PER_BYTE)
    # more than one launch per step: no single kernel's traffic to report
    assert bench.roofline_decode({"launches": 5}, 2_000_000_000, 2000.0, 6800.0, "measured")["traffic"] is None


def test_reference_arm_prints_one_line_of_the_contract():
    """`bench.py --impl reference` (the CPU oracle, rank 0 alone): one JSON line with the
    arm's metric, unit and direction, its own cpu_baseline and an e2e object without host
    copies. About 10 s of CPU work at one step."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
