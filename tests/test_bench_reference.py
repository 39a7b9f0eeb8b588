"""bench.py's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the keys the benchmark contract names, and sizes each step's
sample so that a run with many steps stays a few minutes long."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_budget_shrinks_with_steps():
    sys.path.insert(0, ROOT)
    import bench
    full = 15_000_000
    assert bench.reference_budget(full, 2, 1) == full           # few steps: full samples
    assert bench.reference_budget(full, 100, 5) == int(full * 12 / 105)
    for k, w in ((1, 0), (7, 3), (100, 5), (1000, 10)):
        total = (k + w) * bench.reference_budget(full, k, w)
        assert total <= max(12 * full, (k + w) * full) and total >= min(12 * full, (k + w) * full) * 0.99


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--oracle-pairs", "200000"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["vs_baseline"] is None
    assert line["steps"] == 1 and line["warmup"] == 0 and line["n_gpus"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def test_segment_stats_and_peak_choice():
    sys.path.insert(0, ROOT)
    import bench
    st = bench.segment_stats([3.0, 1.0, 2.0, 10.0, 2.0])
    assert st["median"] == 2.0 and st["min"] == 1.0 and st["max"] == 10.0 and st["p10"] <= st["p90"]
    peaks = {"bf16_tflops": 1919.3, "bf16_tflops_sustained": 1735.5, "hbm_gbs": 6682.2}
    assert bench.pick_bf16_peak(peaks, 0.12) == (1919.3, "bf16 burst")
    assert bench.pick_bf16_peak(peaks, 5.0) == (1735.5, "bf16 sustained")
    assert bench.pick_bf16_peak({"bf16_tflops": 1900.0}, 5.0)[0] == 1900.0


def test_reference_arm_other_config():
    # the tiny workload: the oracle covers the whole tree in one sample
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                          "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["config"]["workload"].startswith("Tiny") and line["value"] > 0
    assert "the whole workload" in line["cpu_baseline"]["sample"]


def test_profiles_match_the_kernel_sources():
    # The roofline's `traffic` comes from the ncu summaries under profiles/,
    # each naming the source it was captured from and that file's sha256
    # prefix; a kernel edited since its capture makes the figure null.
    sys.path.insert(0, ROOT)
    import bench
    for entry in bench.PROFILES:
        assert bench._profile_traffic(entry, 51809) is not None, entry
