"""Host-side pieces of bench.py, on the CPU: the byte count and utilization
arithmetic against the pages' own figures, clock-sample parsing, and the
reference (oracle) arm's JSON line."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_byte_count_matches_case_c():
    """66 us at (7168, 16384) fp16 is 3.55 TB/s on the page."""
    for n, k, ib, ob, us, tbps, peak, util in _rows("case_c_bandwidth.txt"):
        b = bench.algorithmic_bytes(int(n), int(k), int(ib), int(ob))
        got = b / (float(us) * 1e-6) / 1e12
        assert abs(got - float(tbps)) / float(tbps) < 0.01
        assert round(100 * bench.frac_of_peak(float(tbps), float(peak))) == int(util)


def test_utilization_matches_case_b3():
    for n, k, dt, tbps, util in _rows("case_b3_utilization.txt"):
        assert abs(100 * bench.frac_of_peak(float(tbps), 4.8) - int(util)) <= 0.5 + 1e-9


def test_clock_parsing():
    header = ("index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], "
              "clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, "
              "clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, "
              "clocks_event_reasons.sw_power_cap")
    rows = ["0, 1965 MHz, 2070 MHz, 900.1 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 1980 MHz, 2070 MHz, 910.0 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 1950 MHz, 2070 MHz, 905.0 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    s = bench.parse_clock_rows(header, rows)
    assert s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3


def test_reference_arm_line(tmp_path):
    env = dict(os.environ, GEMV_REFERENCE_BUDGET_S="3", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, bench.__file__, "--impl", "reference", "--steps", "4", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_profiled_traffic_gated_by_sources_and_launch(gemv_lib):
    """The roofline's `traffic` comes from the committed ncu summary only
    while the kernel sources and the launch configuration are the ones it
    was captured with."""
    cfg = gemv_lib.gemv_plan(7168, 16384, 0, True, 152)
    got = bench.profiled_traffic("7168x16384_f16", cfg)
    text = open(os.path.join(bench.ROOT, "profiles", "gemv_7168x16384_f16.md")).read()
    if (f"source_digest: `{bench.kernel_source_digest()}`" in text
            and f"launch: `{bench.launch_signature(cfg)}`" in text):
        assert isinstance(got, int) and 234_928_128 <= got < 234_928_128 * 1.05
    else:
        assert got is None
    other = dict(cfg, warp_split=99)
    assert bench.profiled_traffic("7168x16384_f16", other) is None
    assert bench.profiled_traffic("no_such_workload", cfg) is None
    assert bench.launch_signature(cfg).startswith("variant=3 ")
