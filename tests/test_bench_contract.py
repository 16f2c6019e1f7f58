"""The benchmark's reference arm on the CPU: one JSON line with the keys the
benchmark contract names (the GPU arm prints the same keys plus the
roofline, clocks and kernel counts, and needs a GPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] >= 3  # the timing rules' floor, whatever was asked
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["unit"] == "TFLOP/s" and d["data"].startswith("synthetic")
    assert isinstance(d["config"]["workload"], str) and d["config"]["flops_per_step"] > 0
    # the GPU arm's config comes from the same function: same keys, same values
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_attention_prefill_gb300 import workloads
    assert d["config"] == bench.headline_config(
        workloads.make_workload(bench.HEADLINE_WORKLOAD, page_size=16), 1)
    # ms_per_step is the measured time of one (sampled) step, not an extrapolation
    assert d["ms_per_step"] < d["ms_whole_workload_extrapolated"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
