"""The benchmark's JSON contract, on CPU: the reference arm (the fp64 oracle
timed on the host cores) prints one line with the keys the benchmark
contract names, and only rank 0 prints under a multi-rank launch."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "qwen3_4b_n8192", "--steps", "1",
           "--warmup", "3", "--oracle-rows", "32"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [line for line in r.stdout.splitlines() if line.strip()]


def test_reference_arm_line():
    lines = _run()
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "qwen3_4b_n8192"
    # the same config keys and values as the GPU arm prints for this workload
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_inputs import WORKLOADS
    args = argparse.Namespace(workload="qwen3_4b_n8192", seq_len=None)
    assert d["config"] == bench._config(WORKLOADS["qwen3_4b_n8192"], args, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}) == []
