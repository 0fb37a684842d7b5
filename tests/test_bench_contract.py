"""The benchmark's output contract, on the CPU: the reference arm (the oracle
timed on the host cores) prints one JSON line with every key the contract
names, on rank 0 only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_the_contract_line():
    r = _run(["--impl", "reference", "--workload", "tiny_ffn", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_ffn" and d["config"]["schedule"] == "gpipe"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] * 1e-3 * d["value"] - 32) < 1e-6 * 32   # tiny_ffn: 32 rows per step


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--workload", "tiny_ffn", "--steps", "1", "--warmup", "1"], {"RANK": "1"})
    assert r.returncode == 0 and not r.stdout.strip()


def test_library_options_are_named_in_the_config():
    r = _run(["--impl", "reference", "--workload", "tiny_ffn", "--steps", "1", "--warmup", "1",
              "--opt", "inflight=1", "--opt", "PIPELINE=0", "--schedule", "1f1b"])
    assert r.returncode == 0, r.stderr
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert d["config"]["options"] == {"INFLIGHT": 1, "PIPELINE": 0} and d["config"]["schedule"] == "1f1b"
