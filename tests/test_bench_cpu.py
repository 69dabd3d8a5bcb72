"""bench.py's host-side paths without a GPU: the reference arm (the CPU
oracle) runs end to end on the tiny workload and prints one JSON line with
the contract's keys; the CPU baseline reports its phases; the argument rules
hold."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"


def test_warmup_below_three_is_refused():
    r = _bench("--warmup", "2", timeout=120)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_cpu_baseline_reports_phases():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.cpu_baseline(1, 8192)
    assert c["kind"] == "oracle" and c["value"] > 0
    assert set(c["seconds_by_phase"]) == {"amax", "scale+cast_transpose", "gemm"}
    assert c["extrapolated_step_seconds"] > 0 and "extrapolated" in c["extrapolated_note"]
    assert "256 of 256 output rows" in c["sample"]
    empty = bench.cpu_baseline(1, 0)        # no GEMM rows: nothing to extrapolate from
    assert empty["extrapolated_step_seconds"] is None and empty["value"] == 0.0


def test_reference_arm_config_matches_ours():
    """Both arms print the same `config` (workload name, every linear with its
    M, K, N, flops per step) for the same arguments, so the two lines can be
    compared as one workload."""
    sys.path.insert(0, ROOT)
    import bench
    from float8_mixed_precision_gb300 import workloads as wl
    r = _bench("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    args = bench.main.__globals__["argparse"].Namespace(
        config=1, swiglu_input="given", fuse_shared_inputs=False, graph=1, groups=1)
    assert d["config"] == bench.config_dict(wl, args, 1)
    assert d["config"]["linears"] == ["tiny M=256 K=256 N=512"]
    assert d["config"]["flops_per_step"] == 6 * 256 * 256 * 512


def test_fp8_peak_follows_the_region_length():
    """A rate measured over less than a second is held to the burst peak,
    a longer one to the sustained (power-capped) peak; both x 2 for FP8."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.fp8_peak_for(0.05, peaks) == (3800.0, "burst")
    assert bench.fp8_peak_for(0.999, peaks) == (3800.0, "burst")
    assert bench.fp8_peak_for(2.0, peaks) == (3400.0, "sustained")
