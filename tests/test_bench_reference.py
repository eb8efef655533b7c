"""The benchmark's reference arm, run here on the CPU.

`bench.py --impl reference` times the fp64 oracle on a bounded sample of the
benchmark's own workload and prints one JSON line with the keys every arm of
the benchmark carries.  Under torchrun only rank 0 does that work; the other
ranks exit 0 and print nothing.
"""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def _run(rank, world, *extra):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--steps", "2", "--warmup", "1", *extra],
        capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_line_with_the_benchmark_keys(oracle_lib):
    r = _run(0, 1)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d)
    assert d["impl"] == "reference"
    assert (d["metric"], d["unit"]) == (bench.METRIC, bench.UNIT)
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (2, 1, 1)
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD_DESC
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"],
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_on_one_case(oracle_lib):
    r = _run(0, 1, "--case", "C3")
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["config"]["workload"].startswith("C3 bf16 causal B2 H16 N_q4096 N_k4096 d128")
    assert d["value"] > 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run(1, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
