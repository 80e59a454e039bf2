"""The benchmark's reference arm on the CPU (no GPU needed): it times the fp64
oracle on the host cores and must report the steps it actually ran, with the
native arm's config object."""
import json
import os
import subprocess
import sys
import time

import bench
from grouped_gemm_router_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_reports_what_it_ran():
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    w = inputs.WORKLOADS["tiny"]
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    assert line["config"] == bench.line_config(w, 1)
    n = line["sample_tokens"]
    assert 64 <= n <= w.T
    # value is the sample's tokens over one step's time, and the steps fit in the run
    assert abs(line["value"] - n / (line["ms_per_step"] / 1e3)) <= 1e-6 * line["value"]
    assert line["steps"] * line["ms_per_step"] / 1e3 <= wall
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
