"""Host logic of multi-GPU runs, on CPU with the gloo backend (world size 2).

Each rank runs its own copy of the workload (weak scaling, no data-path
collective); the benchmark only reduces timings: the maximum elapsed time and
the total bytes over ranks.  The per-rank work here is the CPU oracle on a
rank-seeded small problem, so the test also checks that ranks stay
independent (every rank's output equals what it computes alone).
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from kv_cache_incremental_split_gb300 import inputs as gen
        case = gen.gqa_padded(rank, B=2, N=4, KV_N=2, D=16, Smax=40, layout="BNSD", dtype="fp16", mask=False)
        out = oracle.ifa_ref(case.query, case.key, case.value, num_heads=4, num_kv_heads=2, scale=case.scale,
                             layout="BNSD", actual_seq_lengths=case.actual_seq_lengths)
        elapsed = 10.0 * (rank + 1)
        nbytes = float(bench.algorithmic_bytes(case))
        agg_t, agg_b = bench.aggregate(elapsed, nbytes, world)
        q.put((rank, agg_t, agg_b, nbytes, out.sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, b0, n0, s0), (r1, t1, b1, n1, s1) = res
    assert t0 == t1 == 20.0            # max over ranks
    assert b0 == b1 == n0 + n1         # sum over ranks
    assert s0 != s1                    # rank-seeded, independent problems


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_algorithmic_bytes_counts_valid_windows_only():
    import bench
    from kv_cache_incremental_split_gb300 import inputs as gen
    case = gen.int8_leftpad(0, B=3, N=8, KV_N=2, D=128, Smax=100, len_lo=10, len_hi=60)
    case.actual_seq_lengths = np.array([10, 60, 95], dtype=np.int64)
    case.kv_padding_size = np.array([0, 50, 20], dtype=np.int64)   # b2 window start < 0: zero row
    assert bench.windows(case) == [(90, 10), (0, 0), (0, 0)]
    expect = 2 * 10 * 2 * 128 * 1 + 2 * 3 * 8 * 128 * 2 + 2 * case.antiquant_scale.nbytes
    assert bench.algorithmic_bytes(case) == expect


def test_bench_gpus_flag_launches_ranks_and_reduces():
    """`bench.py --gpus 2` without WORLD_SIZE relaunches itself under torch.distributed.run with two
    ranks; with --launch-check each rank stands in for its GPU leg (its workload's bytes and a
    time of rank + 1 ms), so the line checks the launch and the reduction: two ranks, the maximum
    time, the bytes of both rank-seeded workloads summed."""
    import json
    import subprocess
    import sys
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--launch-check",
                          "--workload", "tiny_mha", "--steps", "7"], capture_output=True, text=True, cwd=root,
                         env=env, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [json.loads(l) for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["launch_check"] is True and line["value"] is None
    assert line["n_gpus"] == 2 and line["max_rank_ms"] == 2.0
    expect = sum(bench.algorithmic_bytes(bench.make_case("tiny_mha", r)) for r in range(2)) * 7
    assert line["bytes_all_ranks"] == expect
