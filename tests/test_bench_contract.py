"""The benchmark's reference arm (the fp64 oracle on the host cores) runs
without a GPU and prints one JSON line with the fields the benchmark contract
names; the metric, unit and workload are the same as the GPU arm's."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_the_contract_line():
    line = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0")
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["higher_is_better"] is True and line["n_gpus"] == 1 and line["steps"] == 1
    assert line["config"]["workload"] == "decode-128k-b64-20L"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_oracle_baseline_of_the_chunked_prefill_is_bounded():
    """a workload of 8,192 queries per sequence is timed one query at a time, spread over the
    chunk, and stops at its time budget"""
    import time
    sys.path.insert(0, ROOT)
    import bench
    wl = bench.workload_of("prefill-chunk-8k-after-120k")
    units = bench.oracle_units(wl)
    assert len(units) == wl.n_q and sorted(u[0][0] for u in units) == list(range(wl.n_q))
    assert units[0][0][0] != 0 or units[1][0][0] != 1      # spread, not in chunk order
    t0 = time.perf_counter()
    cb = bench.cpu_baseline(wl, 24, budget_s=0.5)
    assert time.perf_counter() - t0 < 120
    assert cb["kind"] == "oracle" and cb["value"] > 0 and "of 1 sequences (of 1)" in cb["sample"]
