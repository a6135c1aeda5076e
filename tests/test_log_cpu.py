"""GEMV_LOG=1: one stderr line per launch configuration the planner builds,
in the documented key -> configuration format; nothing without it.  Run in a
child process so the variable is set before the library reads it (once).
No GPU: gemv_plan() is pure host arithmetic."""
from __future__ import annotations

import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys
sys.path.insert(0, %r)
import memory_bound_gemv_02_gb300 as g
L = g.lib()
out = g.GemvConfig()
for n, k, dt in ((7168, 16384, 0), (18433, 7169, 1), (256, 262144, 2)):
    assert L.gemv_plan(n, k, dt, 1, 152, None, ctypes.byref(out)) == 0
assert L.gemv_plan(4, 8, 9, 1, 152, None, ctypes.byref(out)) == g.GEMV_ERR_DTYPE  # no line for a failure
print("done")
""" % ROOT

LINE = re.compile(r"^gemv: plan dev=-1 n=(\d+) k=(\d+) dtype=(\d) aligned=([01]) -> variant=(\d) ctas=(\d+) "
                  r"warps_per_cta=(\d+) warp_split=(\d+) rows_per_warp=(\d) unroll=(\d) grid_split=(\d+) "
                  r"k_segment=(\d+) stages=(\d+) smem_bytes=(\d+)$")


def _run(env_value):
    env = dict(os.environ)
    env.pop("GEMV_LOG", None)
    if env_value is not None:
        env["GEMV_LOG"] = env_value
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("done")
    return [ln for ln in r.stderr.splitlines() if ln.startswith("gemv:")]


def test_log_lines_follow_the_format(gemv_lib):
    lines = _run("1")
    assert len(lines) == 3, lines
    want = [(7168, 16384, 0, 1), (18433, 7169, 1, 0), (256, 262144, 2, 1)]
    for ln, (n, k, dt, al) in zip(lines, want):
        m = LINE.match(ln)
        assert m, ln
        assert tuple(int(x) for x in m.groups()[:4]) == (n, k, dt, al)
        # the logged configuration is the one gemv_plan() returned
        cfg = gemv_lib.gemv_plan(n, k, dt, b_aligned16=True, sm_count=152)
        logged = dict(zip(("variant", "ctas", "warps_per_cta", "warp_split", "rows_per_warp", "unroll",
                           "grid_split", "k_segment", "stages", "smem_bytes"), (int(x) for x in m.groups()[4:])))
        assert logged == {kk: cfg[kk] for kk in logged}, (logged, cfg)


def test_no_log_by_default(gemv_lib):
    assert _run(None) == []
    assert _run("0") == []
