"""bench.py's reference arm on the CPU: the float64 oracle timed on the host
cores prints one JSON line with the native arm's metric and unit, for a
forward, a backward and a decode workload (no GPU is touched)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,unit", [("f16_causal_1k", "TFLOP/s"), ("f16_decode_4k_q4", "GB/s")])
def test_reference_arm_prints_one_line(workload, unit):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--workload", workload], capture_output=True, text=True, env=env,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == unit and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["gpu_launches"] == 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
