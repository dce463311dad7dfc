"""The benchmark's reference arm (`bench.py --impl reference`): the CPU oracle
timed on the host cores.  It needs no GPU, so its JSON line is checked here:
the keys the benchmark contract asks of it, values that agree with one
another, and that under torchrun only rank 0 runs and prints."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(extra_env=None, steps=1, warmup=3):
    env = dict(os.environ)
    env.update(extra_env or {})
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", str(steps), "--warmup", str(warmup)],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    return [ln for ln in proc.stdout.splitlines() if ln.strip()]


@pytest.fixture(scope="module")
def line():
    out = run_reference()
    assert len(out) == 1, out
    return json.loads(out[0])


def test_reference_line_has_the_contract_keys(line):
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 3
    assert line["higher_is_better"] is True
    assert line["vs_baseline"] is None
    assert line["unit"] == "GB/s"


def test_reference_line_agrees_with_itself(line):
    import bench
    assert line["metric"] == bench.METRIC
    assert line["config"]["workload"] == "mixtral-8x7b-moe-layer"
    assert 1 <= line["config"]["T_sample"] <= line["config"]["T"]
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1
    assert cpu["value"] == line["value"] and cpu["unit"] == line["unit"]
    assert str(line["config"]["T_sample"]) in cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_print_nothing():
    out = run_reference({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert out == []
