"""The benchmark script's command line and its CPU-only reference arm (the
fp64 oracle timed on host cores), run end to end on the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return out.stdout


def test_help_lists_the_contract_flags():
    text = run_bench("--help")
    for flag in ("--gpus", "--steps", "--warmup", "--impl", "--workload", "--mode", "--no-e2e"):
        assert flag in text


def test_reference_arm_prints_one_json_line():
    lines = [l for l in run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
             .splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
