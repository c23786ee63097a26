"""CPU checks of the split planner (plan.cu: build_windows, choose_grid, build_bounds)
through a host-only driver (tests/plan_driver.cpp) compiled against it: the CTA tile
bounds partition the tiles, every CTA gets a tile, splitTiles gives equal shares, and the
cost-weighted split (16 per tile, plus piece_cost per whole sequence and cut_cost per
piece of a cut sequence, in 1/16 tiles) is better balanced than equal shares on mixes of
short and long sequences."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_incremental_split_gb300", "csrc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("plan") / "plan_driver")
    subprocess.check_call([nvcc, "-std=c++17", "-O1", "-I", CSRC, os.path.join(ROOT, "tests", "plan_driver.cpp"),
                           os.path.join(CSRC, "plan.cu"), "-o", out])
    return out


def run(driver, problems):
    text = "\n".join(" ".join(str(int(x)) for x in pr) for pr in problems) + "\n"
    res = subprocess.run([driver], input=text, capture_output=True, text=True, check=True).stdout.splitlines()
    out = []
    for line in res:
        f = line.split()
        assert f[0] != "error", line
        W, P, T, Ec, Ex = map(int, f[:5])
        out.append((W, P, T, (Ec, Ex), np.array(list(map(int, f[5:])), dtype=np.int64)))
    return out


def piece_costs(bounds, lens, T, RS, E):
    """Cost of every CTA range in 1/16 tiles: 16 per tile, Ec per whole sequence, Ex per piece
    of a sequence the range boundaries cut, on the real sequence layout."""
    Ec, Ex = E
    tiles = [(l + T - 1) // T for l in lens]
    seqs = []  # (first tile, end tile) of every sequence
    g = 0
    for t in tiles:
        for _ in range(RS):
            if t > 0:
                seqs.append((g, g + t))
            g += t
    costs = []
    for c in range(len(bounds) - 1):
        lo, hi = bounds[c], bounds[c + 1]
        cost = 16 * (hi - lo)
        for s, e in seqs:
            if e <= lo or s >= hi:
                continue
            cost += Ec if (s >= lo and e <= hi) else Ex
        costs.append(cost)
    return np.array(costs)


MIXES = [
    # (B, N, KV_N, D, kv, lens generator)
    (16, 32, 8, 128, 0, lambda r: r.integers(1, 4097, 16)),
    (32, 64, 8, 128, 2, lambda r: r.integers(256, 8193, 32)),
    (200, 32, 8, 128, 0, lambda r: r.integers(0, 301, 200)),
    (64, 32, 8, 128, 0, lambda r: np.where(r.random(64) < 0.8, r.integers(1, 200, 64), r.integers(8000, 30000, 64))),
    (3, 8, 8, 64, 0, lambda r: r.integers(40000, 60000, 3)),
    (1, 8, 8, 64, 0, lambda r: np.array([100])),
]


@pytest.mark.parametrize("mix", range(len(MIXES)))
@pytest.mark.parametrize("pmax", [152, 16, 1])
def test_bounds_partition_the_tiles(driver, mix, pmax):
    B, N, KVN, D, kv, gen = MIXES[mix]
    r = np.random.default_rng(100 + mix)
    probs = [[B, N, KVN, D, kv, 0, pmax] + list(gen(r)) for _ in range(4)]
    for W, P, T, E, b in run(driver, probs):
        assert len(b) == P + 1 and 1 <= P <= pmax
        if W == 0:
            continue
        assert b[0] == 0 and b[-1] == W
        assert (np.diff(b) >= 1).all(), "every CTA holds at least one tile"
        assert P <= W


@pytest.mark.parametrize("split", [1, 2, 7])
def test_split_tiles_gives_equal_shares(driver, split):
    r = np.random.default_rng(7)
    lens = list(r.integers(1, 4097, 16))
    ((W, P, T, E, b),) = run(driver, [[16, 32, 8, 128, 0, split, 152] + lens])
    assert P == min(152, math.ceil(W / split))
    assert (b == np.array([c * W // P for c in range(P + 1)])).all()


@pytest.mark.parametrize("mix", [0, 1, 2, 3])
def test_weighted_split_balances_piece_costs(driver, mix):
    B, N, KVN, D, kv, gen = MIXES[mix]
    r = np.random.default_rng(200 + mix)
    for _ in range(4):
        lens = [int(x) for x in gen(r)]
        ((W, P, T, E, b),) = run(driver, [[B, N, KVN, D, kv, 0, 152] + lens])
        tiles = sum((l + T - 1) // T for l in lens)
        RS = W // tiles
        weighted = piece_costs(b, lens, T, RS, E)
        equal = piece_costs(np.array([c * W // P for c in range(P + 1)]), lens, T, RS, E)
        assert weighted.max() <= equal.max()
        # every range sits within two cut pieces' fixed cost (plus a tile) of the mean
        assert weighted.max() - weighted.mean() <= 2 * E[1] + 16


def test_planner_is_deterministic(driver):
    r = np.random.default_rng(3)
    pr = [32, 64, 8, 128, 2, 0, 152] + list(r.integers(256, 8193, 32))
    a, b = run(driver, [pr, pr])
    assert a[:4] == b[:4] and (a[4] == b[4]).all()
