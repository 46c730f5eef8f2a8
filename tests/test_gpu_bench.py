"""The benchmark's own command on the GPU: a short default run prints one
JSON line with the keys its readers take (the metric, the roofline block,
the end-to-end leg with its host-link bound, the launch count and the clock
record), graph mode captures no graph inside the timed region, and the
host-link mode prints its nine cells. Needs a GPU."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_default_line_carries_the_contract_keys():
    lines = _run("--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "3",
                 "--no-extras")
    assert len(lines) == 1
    d = lines[0]
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "llama70b_t1024_h8192_n8"
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["algorithmic_bytes"] == (8 + 3) * 1024 * 8192 * 2 + 8192 * 2
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert 0 < roof["frac_per_launch"] <= roof["frac"] * 1.05
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 9 * 1024 * 8192 * 2 + 8192 * 2
    assert e2e["d2h_bytes_per_step"] == 2 * 1024 * 8192 * 2
    assert 0 < e2e["value"] < d["value"]
    link = e2e["link_bound"]
    # the copies alone cannot take longer than the copies plus the step, beyond noise
    assert 0 < link["frac"] <= 1.1 and link["GB_s"] > 0
    assert d["gpu_launches"] == 5
    assert "sm_mhz" in d["clocks"] and "edges" in d["clocks"]
    assert d["unfused"]["fused_speedup"] > 0


def test_link_mode_prints_nine_cells():
    lines = _run("--link", "--steps", "3")
    assert [(l["link"], l["streams"]) for l in lines] == [
        (w, k) for w in ("h2d", "d2h", "both") for k in (1, 2, 4)]
    n_in, n_out = 9 * 1024 * 8192 * 2 + 8192 * 2, 2 * 1024 * 8192 * 2
    for l in lines:
        want = {"h2d": n_in, "d2h": n_out, "both": n_in + n_out}[l["link"]]
        assert l["bytes"] == want and l["GB_s"] > 0


def test_graph_mode_captures_nothing_in_the_timed_region():
    """Graph mode replays one graph per rotating input set; every graph is
    captured during warm-up, so the timed steps are replays only."""
    lines = _run("--workload", "pr1_t128_h4096_n2", "--mode", "graph", "--steps", "50",
                 "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "3", "--no-extras",
                 "--no-unfused")
    assert len(lines) == 1
    d = lines[0]
    assert d["config"]["graph_captures_in_region"] == 0
    assert d["config"]["launch"].startswith("cuda graph")
    assert d["value"] > 0


def test_sweep_block_carries_every_form():
    """The default line's sweep block: the one-pipeline ring on the whole GPU,
    the two-pipeline forms under an 8-SM budget, and the direct form for the
    two small batches (one row per CTA; one CTA per row)."""
    lines = _run("--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "3",
                 "--no-unfused")
    cells = {(c["T"], c["H"], c["N"], c["sm_budget"]): c for c in lines[0]["sweep"]["cells"]}
    assert cells[(1024, 8192, 8, "full")]["form"] == "ring"
    assert cells[(4096, 8192, 2, 8)]["form"] == "two pipelines"
    assert cells[(4096, 8192, 12, 8)]["form"] == "two pipelines"
    assert cells[(128, 8192, 8, "full")]["form"] == "direct"
    d = cells[(304, 4096, 8, "full")]
    assert d["form"] == "direct" and d["ctas"] == 304 and d["sms_used"] <= 152
    for c in cells.values():
        assert c["GB_s"] > 0 and c["us_b2b"] > 0

