"""The reference arm of bench.py (the CPU oracle timed on the host cores) on
the CPU: one JSON line with the contract's keys, on the GPU arm's metric and
config; under more than one rank, rank 0 alone prints and the others exit 0
without work."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run({})
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    from mxfp8_norm_quant_gb300 import workloads as W
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"] == bench.make_config(W.get_workload(bench.DEFAULT_WORKLOAD), 1)
    assert d["config"]["workload"] == "m32768_stress"
    # the contract's floor of 3 warm-up steps applies to a smaller request
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3 and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("rank", [1])
def test_other_ranks_exit_without_work(rank):
    assert _run({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank)}) == []
