"""bench.py's JSON line without a GPU: the reference arm (the oracle on the
host cores) carries every key of the contract, and the one-core oracle
timing that cpu_baseline starts in a child process prints its own line."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line_has_the_contract_keys():
    d = _run(["--impl", "reference", "--workload", "tiny_b1_f32", "--steps", "3", "--warmup", "1"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 1
    assert d["value"] > 0 and d["unit"] == "nodes/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_b1_f32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["sample"]
    assert cb["cores"] == os.cpu_count() and cb["blas_threads_per_process"] == 1
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_oracle_worker_waits_for_go_and_runs_exact_steps():
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny_b1_f32",
                        "--oracle-single-core", "32,16", "--oracle-worker", "--warmup", "1", "--cpu-seconds", "0",
                        "--steps", "3"], input="go\n", capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = r.stdout.splitlines()
    assert lines[0] == "ready"
    d = json.loads(lines[-1])
    assert d["requests"] == 3 and d["nodes"] == 30 and d["threads"] == 1


def test_single_core_oracle_timing_line():
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    d = _run(["--workload", "tiny_b1_f32", "--cpu-seconds", "0.5", "--oracle-single-core", "32"], env=env)
    assert d["value"] > 0 and d["requests"] == 1 and d["threads"] == 1
