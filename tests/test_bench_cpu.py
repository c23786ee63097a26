"""CPU checks of the benchmark's host paths: the reference arm (the oracle timed on the
host cores) keeps the JSON contract and its whole run stays within its time budget,
whatever the step count."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_ref(workload, steps, warmup, total):
    t = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          workload, "--steps", str(steps), "--warmup", str(warmup), "--ref-total-seconds",
                          str(total)], capture_output=True, text=True, check=True, cwd=ROOT, timeout=600)
    line = json.loads(out.stdout.strip().splitlines()[-1])
    return line, time.time() - t


@pytest.mark.parametrize("workload", ["tiny_mha", "gqa_tensorlist", "sfa_mla_small", "kv_append_int8"])
def test_reference_arm_line(workload):
    line, _ = run_ref(workload, 20, 3, 2.0)
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 20
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the config both arms print, L2 method included
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse(["--workload", workload])
    assert line["config"] == bench.line_config(args, bench.make_case(workload, 0), 1)
    assert line["config"]["l2"]


def test_reference_arm_time_is_bounded_for_many_steps():
    # 20000 steps (the default) must not take 20000 oracle rows of time
    line, wall = run_ref("gqa_padded", 20000, 20, 5.0)
    assert line["steps"] == 20000
    assert wall < 180
