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


def test_cpu_baseline_sampler_covers_every_kind_of_workload():
    """The GPU arm's cpu_baseline helper: forward + one backward, forward + both backwards, and decode (bytes)."""
    sys.path.insert(0, ROOT)
    import bench
    from attention_kl_divergence_streamkl_gb300 import synth

    w = synth.WORKLOADS["kl_b1h1_n128_d64"]
    v1, dt1, r1, d1 = bench.oracle_sample(w, (1,), 0.05)
    v12, dt12, r12, d12 = bench.oracle_sample(w, (1, 2), 0.05)
    assert v1 > 0 and v12 > 0 and 16 <= r1 <= 128 and 16 <= r12 <= 128
    assert "setting-1 backward" in d1 and "setting-1 + setting-2 backward" in d12
    # counted FLOP per unmasked pair: 12D for one backward, 20D for both (rows r of 128 keys each, non-causal)
    assert v1 * 1e12 * dt1 == pytest.approx(12 * 64 * r1 * 128, rel=1e-9)
    assert v12 * 1e12 * dt12 == pytest.approx(20 * 64 * r12 * 128, rel=1e-9)
    wd = synth.WORKLOADS["decode_b8h32_nq1_nk131072_d128"]
    vd, dtd, rd, dd = bench.oracle_sample(wd, (), 0.05)
    assert vd > 0 and rd == 1 and "K1, K2, Q1 and Q2" in dd
    b = bench.blas_threads()
    assert b is None or b >= 1


GPU_KEYS = KEYS - {"impl"} | {"roofline", "clocks", "gpu_launches", "per_kernel_ms", "extra_hbm"}


def _run_ours(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
@pytest.mark.parametrize("extra,unit", [(("--workload", "kl_b2h32_n4096_d128_causal"), "TFLOP/s"),
                                        (("--workload", "kl_b2h32_n4096_d128_causal", "--mutual"), "TFLOP/s"),
                                        (("--workload", "decode_b8h32_nq4_nk131072_d128"), "GB/s")])
def test_gpu_arm_line(extra, unit):
    """The GPU arm's JSON line on small workloads: every contract key, a roofline for the dominant kernel, a
    positive end-to-end figure with its copies counted, and a launch count."""
    d = _run_ours(*extra, "--steps", "3", "--warmup", "3", "--cpu-seconds", "0.5")
    assert GPU_KEYS <= set(d), GPU_KEYS - set(d)
    assert d["unit"] == unit and d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    roof = d["roofline"]
    assert roof["bound"] in ("tensor", "hbm") and roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-6)
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == unit and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= 3 * 1 and d["cpu_baseline"]["value"] > 0 and d["cpu_baseline"]["cores"] >= 1
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
