"""`bench.py --impl reference` on the host: the oracle's decode step timed on
this machine's cores, printed as one JSON line with the same metric, unit and
workload as the CUDA arm; under torchrun only rank 0 prints."""
import ast
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(extra_env, *args):
    env = dict(os.environ, **extra_env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    r = run_bench({"RANK": "1", "WORLD_SIZE": "2"}, "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_line_of_the_contract():
    r = run_bench({"RANK": "0", "WORLD_SIZE": "1"}, "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3  # at least 3 warm-up steps
    assert line["n_gpus"] == 1 and line["dtype"] == "f64"
    assert line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["batch"] == 64 and line["config"]["Hq"] == 32
    # the bytes the decode step must read: K and V of every live key, bf16
    assert line["config"]["kv_bytes_per_step"] % (2 * 8 * 128 * 2) == 0
    # the CUDA arm's metric and workload strings
    consts = {}
    for node in ast.parse(open(os.path.join(ROOT, "bench.py")).read()).body:
        if isinstance(node, ast.Assign) and getattr(node.targets[0], "id", "") in ("METRIC",
                                                                                  "WORKLOAD"):
            consts[node.targets[0].id] = node.value.value
    assert line["metric"] == consts["METRIC"]
    assert line["config"]["workload"] == consts["WORKLOAD"]
