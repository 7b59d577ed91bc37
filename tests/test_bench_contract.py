"""bench.py's reference arm on CPU: one JSON line with the contract's keys.

The reference arm times the fp64 oracle on bounded samples of the workload, so
it runs without a GPU; the GPU arm's line carries the same keys plus the
roofline, clocks and launch count (checked on the GPU machine by running bench.py).
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _run(*args):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1", *args],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit", [("kl_b1h32_n65536_d128_causal", "TFLOP/s"),
                                           ("decode_b8h32_nq4_nk131072_d128", "GB/s")])
def test_reference_arm_line(workload, unit):
    d = _run("--workload", workload)
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["unit"] == unit and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None


@pytest.mark.parametrize("extra,flop_per_pair_per_d", [((), 12), (("--mutual",), 20)])
def test_reference_arm_full_workload(extra, flop_per_pair_per_d):
    """--full runs the oracle over every head and row: the value is the whole workload's counted FLOP (12D per
    unmasked pair for forward + one backward, 20D with both backwards) over the measured time."""
    d = _run("--workload", "kl_b1h1_n128_d64", "--full", *extra)
    cb = d["cpu_baseline"]
    assert cb["full_workload_s_is"] == "measured"
    assert cb["full_workload_s"] == pytest.approx(d["ms_per_step"] / 1e3, rel=1e-9)
    flop = flop_per_pair_per_d * 64 * 128 * 128  # B1 H1 N_Q = N_K = 128, D64, non-causal
    assert d["value"] * 1e12 * cb["full_workload_s"] == pytest.approx(flop, rel=1e-9)
    assert d["config"]["setting"] == ("mutual" if extra else 1)


def test_reference_arm_sample_extrapolates():
    d = _run("--workload", "kl_b2h32_n4096_d128_causal")
    cb = d["cpu_baseline"]
    assert cb["full_workload_s_is"].startswith("extrapolated")
    # 64 rows of one head sampled: the whole workload is 64 heads x 4096 x 4097 / 2 pairs
    sample_pairs = sum(min(4096, i + 1) for i in range(4096 - 64, 4096))
    ratio = 64 * 4096 * 4097 // 2 / sample_pairs
    assert cb["full_workload_s"] == pytest.approx(d["ms_per_step"] / 1e3 * ratio, rel=1e-9)
