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


def test_algorithmic_bytes_closed_forms():
    """The bytes behind every reported GB/s: only what the method must move.  The tiny MHA
    workload is exactly K + V (262 144 B) plus query and output (2 x 1 024 B); GQA counts the
    valid tokens' key/value rows, query, output and the mask over the valid windows; paging adds
    one block-table entry per block used; the sparse decode moves 2 176 B per selected token
    (key 1 024 + rope 128 + value 1 024; 1 152 B when value is key) plus one block-table entry,
    the query, the output and the index rows."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from kv_cache_incremental_split_gb300 import inputs as gen
    assert bench.algorithmic_bytes(bench.make_case("tiny_mha", 0)) == 264_192
    g = gen.gqa_padded(3, B=4, N=32, KV_N=8, D=128, Smax=512)
    toks = int(g.actual_seq_lengths.sum())
    assert bench.algorithmic_bytes(g) == 2 * toks * 8 * 128 * 2 + 2 * 4 * 32 * 128 * 2 + toks
    p = gen.paged_gqa(4, B=5, N=32, KV_N=8, D=128, block_size=128, len_lo=100, len_hi=1000)
    lens = p.actual_seq_lengths.astype(np.int64)
    assert bench.algorithmic_bytes(p) == (2 * int(lens.sum()) * 8 * 128 * 2 + 2 * 5 * 32 * 128 * 2
                                          + int(((lens + 127) // 128).sum()) * 4)
    s = gen.sfa_mla(5, B=3, Q_N=128, block_size=64, kv_len=4096, sparse_size=512, nvalid_lo=100, nvalid_hi=512)
    n = int(((s.sparse_indices >= 0) & (s.sparse_indices < s.actual_seq_lengths_kv[:, None, None, None])).sum())
    fixed = 3 * 128 * (512 + 64) * 2 + 3 * 128 * 512 * 2 + s.sparse_indices.nbytes
    assert bench.algorithmic_bytes(s) == n * (2_176 + 4) + fixed
    s.value = s.key
    assert bench.algorithmic_bytes(s) == n * (1_152 + 4) + fixed
