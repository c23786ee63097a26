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


# ---------------------------------------------------------------- window resolution (build_windows)

def windows(driver, B, smax, lens, pads=None, paged=False, cols=0, bs=128):
    lens = [-9] * B if lens is None else list(lens)
    pads = [] if pads is None else list(pads)
    line = f"w {B} {smax} {int(paged)} {cols} {bs} {len(pads)} " + " ".join(map(str, pads + lens)) + "\n"
    out = subprocess.run([driver], input=line, capture_output=True, text=True, check=True).stdout.split()
    if out[0] == "error":
        return int(out[1])
    W, T = int(out[0]), int(out[1])
    v = np.array(list(map(int, out[2:])), dtype=np.int64)
    return W, T, v[:B], v[B:]


def expected_window(smax, length, pad):
    """The IncreFlashAttention README's kv left padding rule: tokens [Smax - pad - len, Smax - pad),
    a negative pad counting as 0, an all-zero row (empty window) when the start or the end falls
    below 0; without padding sizes the first len tokens."""
    if pad is None:
        return 0, length
    pad = max(pad, 0)
    st, en = smax - pad - length, smax - pad
    if st < 0 or en < 0:
        return 0, 0
    return st, length


def test_windows_follow_the_left_padding_rule(driver):
    r = np.random.default_rng(11)
    smax = 1000
    lens = [0, 1, 1000, 999, 500, 700, 37, 1000] + list(r.integers(0, 1001, 24))
    pads = [0, 999, 0, 1, -5, 301, 963, 1] + list(r.integers(-20, 1001, 24))
    B = len(lens)
    W, T, st, ln = windows(driver, B, smax, lens, pads)
    for b in range(B):
        assert (st[b], ln[b]) == expected_window(smax, lens[b], pads[b]), b
    assert W == sum((int(x) + T - 1) // T for x in ln) * 2  # tiles of every (batch, kv head)
    # one broadcast padding size
    W1, _, st1, ln1 = windows(driver, 4, smax, [10, 200, 990, 995], [7])
    for b, L in enumerate([10, 200, 990, 995]):
        assert (st1[b], ln1[b]) == expected_window(smax, L, 7)


def test_windows_without_padding_and_rejected_lengths(driver):
    # right padding: the first len tokens; without lengths every batch uses maxSeqLen
    _, _, st, ln = windows(driver, 3, 300, [0, 17, 300])
    assert list(st) == [0, 0, 0] and list(ln) == [0, 17, 300]
    _, _, st, ln = windows(driver, 2, 300, None)
    assert list(ln) == [300, 300]
    # padding sizes without lengths leave the window right padded
    _, _, st, ln = windows(driver, 2, 300, None, [5, 9])
    assert list(st) == [0, 0] and list(ln) == [300, 300]
    # a length above the cache, or negative, is refused (161002)
    assert windows(driver, 2, 300, [301, 1]) == 161002
    assert windows(driver, 2, 300, [-1, 1]) == 161002
    assert windows(driver, 2, 300, [-1, 1], [0]) == 161002
    # paged: up to blockTableCols * blockSize tokens
    _, _, st, ln = windows(driver, 2, 0, [512, 1], paged=True, cols=4, bs=128)
    assert list(ln) == [512, 1]
    assert windows(driver, 2, 0, [513, 1], paged=True, cols=4, bs=128) == 161002
