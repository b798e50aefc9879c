"""The decode indexer's sample estimate of a row's K-th key (the streaming Top-K admits only keys at
or above the r-th largest of a segment's first tiles; the merge checks the estimate and rescores the
row when it was too high). Results never depend on it; how often the check fails does. The rule's
constants are read from the kernel source, and the probability that a sample of S keys from a row
of n holds r or more of the row's K largest keys (hypergeometric, exact) must stay below 4e-11 at
every row length for which the rule takes an estimate."""
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = os.path.join(ROOT, "indexer_top_sparse_paged_gb300", "csrc", "common.cuh")
TILE_KEYS = 128


def _rule():
    src = open(COMMON).read()
    tiles = int(re.search(r"constexpr int kEstTiles = (\d+);", src).group(1))
    m = re.search(r"ceilf\(mu \+ ([0-9.]+)f \* sqrtf\(mu\) \+ ([0-9.]+)f\)", src)
    assert m, "estimate rank rule not found in common.cuh"
    a, b = float(m.group(1)), float(m.group(2))
    cond = re.search(r"return \(4 \* r < 3 \* sample\) \? r : 0u;", src)
    assert cond, "estimate applicability condition not found in common.cuh"
    return tiles, a, b


def _rank(sample: int, n: int, K: int, a: float, b: float) -> int:
    """The kernel's rank (0: no estimate), computed in float32 as the kernel does."""
    import numpy as np
    if n <= K:
        return 0
    mu = np.float32(sample) * np.float32(K) / np.float32(n)
    r = int(np.ceil(np.float32(mu + np.float32(a) * np.sqrt(mu, dtype=np.float32) + np.float32(b))))
    return r if 4 * r < 3 * sample else 0


@pytest.mark.parametrize("K", [512, 2048])
def test_estimate_failure_probability_bound(K):
    stats = pytest.importorskip("scipy.stats")
    tiles, a, b = _rule()
    worst, n_checked = 0.0, 0
    lengths = sorted(set(list(range(K + 64, 40000, 97)) + list(range(40000, 300000, 4999)) +
                         [1 << 19, 1 << 20, 1 << 21, 1 << 22]))
    for sample in (tiles * TILE_KEYS // 2, tiles * TILE_KEYS):  # a full sample, and one of rows with invalid keys
        for n in lengths:
            r = _rank(sample, n, K, a, b)
            if r == 0:
                continue
            p = stats.hypergeom.sf(r - 1, n, K, sample)
            worst = max(worst, p)
            n_checked += 1
    assert n_checked > 100
    assert worst < 4e-11, worst


def test_estimate_applies_to_long_rows_only():
    """Short rows (where the estimate would admit most keys anyway) take none; long ones do."""
    tiles, a, b = _rule()
    S = tiles * TILE_KEYS
    assert _rank(S, 2048, 2048, a, b) == 0
    assert _rank(S, 2500, 2048, a, b) == 0
    assert _rank(S, 24576, 2048, a, b) > 0
    assert _rank(S, 1 << 20, 2048, a, b) > 0
    # longer rows take smaller ranks (mu = S K / n shrinks), never below ceil(b), the limit as mu -> 0
    ranks = [_rank(S, n, 2048, a, b) for n in (24576, 1 << 17, 1 << 20, 1 << 22, 1 << 26)]
    assert all(x >= y for x, y in zip(ranks, ranks[1:])), ranks
    assert ranks[-1] >= math.ceil(b)
