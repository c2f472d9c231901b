"""bench.py's output contract, checked on the host: the reference arm (the
oracle timed on the CPU cores) prints exactly one JSON line carrying the keys
that the benchmark driver reads, with a cpu_baseline and an e2e object
describing that same run.  The smallest workload and a one-second sample per
step keep it to a few seconds."""
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def test_reference_arm_prints_one_contract_line():
    t0 = time.monotonic()
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_f32",
                        "--steps", "2", "--warmup", "1", "--cpu-seconds", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    wall = time.monotonic() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert REQUIRED <= d.keys(), sorted(REQUIRED - d.keys())
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] in ("weak", "strong")
    assert d["vs_baseline"] is None
    assert isinstance(d["config"], dict) and d["config"]["workload"].startswith("tiny_f32")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["steps"] * d["ms_per_step"] / 1000.0 <= wall     # the steps' own time, not a projection
    assert d["extrapolated_ms_per_full_workload"] > 0
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_rescaled_workload_is_named_for_its_sizes():
    """--batch / --heads (smaller cases for profiler captures) give the
    workload a name of its own, so a DRAM-traffic record taken on the full
    workload is never reported for it."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "deit_t", "--batch", "1",
                        "--heads", "2", "--steps", "1", "--warmup", "1", "--cpu-seconds", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    wl = d["config"]["workload"]
    assert wl.startswith("deit_t_B1_H2:") and "B=1 H=2" in wl
    sys.path.insert(0, ROOT)
    import bench
    assert bench.traffic_from_profiles("mita_fused", "deit_t_B1_H2") is None
