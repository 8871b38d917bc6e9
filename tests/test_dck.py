"""Dynamic chunk sizing (the SGLang article's "DCK 12288 (sigma=0.65)", read as stated in
oracle/dck.py): the plain restatement is pinned to a hand-derived example, to brute-force pair
counts and to the two limits sigma = 0 (fixed chunks) and sigma = 1 (chunks of equal cost); the
library's planner then matches it size for size (CPU only)."""
import json
import math
import os
import types

import numpy as np
import pytest

import ring_attention_slope_gb300 as slope
from _lib import built_lib
from oracle import dck as odck

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "dck_small.json")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def visible_pairs(s, n, window):
    """Visible (query, key) pairs of rows [s, s + n) counted on a materialised mask."""
    i = np.arange(s, s + n)[:, None]
    j = np.arange(0, s + n)[None, :]
    m = j <= i
    if window:
        m &= (i - j) < window
    return int(m.sum())


# ---------------------------------------------------------------- pins of the restatement

def test_golden_small_example():
    g = json.load(open(GOLDEN))
    c = g["case"]
    assert odck.dck_chunk_sizes(c["S"], c["initial"], c["sigma"], c["window"], c["align"]) == g["sizes"]


@pytest.mark.parametrize("s,n,window", [(0, 1, 0), (0, 37, 0), (5, 40, 0), (100, 33, 16), (3, 60, 16), (0, 20, 64)])
def test_chunk_cost_is_the_mask_count(s, n, window):
    assert odck.chunk_cost(s, n, window) == visible_pairs(s, n, window)


def test_sigma_zero_is_fixed_chunking():
    """No smoothing towards the equal-cost size: every chunk keeps the initial size (the 64K workload's
    5 x 12288 + 4096)."""
    assert odck.dck_chunk_sizes(65536, 12288, 0.0) == [12288] * 5 + [4096]
    assert odck.dck_chunk_sizes(1000, 300, 0.0, window=50) == [300, 300, 300, 100]


@pytest.mark.parametrize("sigma", [0.0, 0.65, 1.0])
def test_window_one_keeps_the_initial_size(sigma):
    """With a window of 1 every row sees one key, so a chunk of the initial size costs exactly the target:
    the equal-cost size is the initial size and the chunks stay fixed whatever sigma is."""
    assert odck.dck_chunk_sizes(10, 4, sigma, window=1) == [4, 4, 2]
    assert odck.dck_chunk_sizes(65536, 12288, sigma, window=1) == [12288] * 5 + [4096]


@pytest.mark.parametrize("S,initial,window", [(3000, 400, 0), (5000, 256, 100), (777, 777, 0), (2048, 100, 0)])
def test_sigma_one_is_the_equal_cost_partition(S, initial, window):
    """Every chunk but the last is the longest run of rows whose pairs stay within the first chunk's."""
    sizes = odck.dck_chunk_sizes(S, initial, 1.0, window)
    target = visible_pairs(0, min(initial, S), window)
    s = 0
    for c, n in enumerate(sizes):
        cost = visible_pairs(s, n, window)
        if n > 1:
            assert cost <= target
        if s + n < S:
            assert visible_pairs(s, n + 1, window) > target or n == 1 and cost > target
        s += n
    assert s == S


@pytest.mark.parametrize("sigma", [0.0, 0.3, 0.65, 1.0])
@pytest.mark.parametrize("align", [1, 64])
def test_sizes_sum_to_S_and_never_grow(sigma, align):
    sizes = odck.dck_chunk_sizes(65536, 12288, sigma, align=align)
    assert sum(sizes) == 65536 and all(n > 0 for n in sizes)
    assert all(a >= b for a, b in zip(sizes, sizes[1:]))
    assert all(n % align == 0 for n in sizes[1:-1])


def test_dynamic_chunks_balance_attention_cost():
    """The point of shrinking the chunks: their attention costs stay far closer to the first chunk's than
    fixed 12K chunks do (whose last full chunk costs about 9x the first)."""
    S = 65536

    def spread(sizes):
        costs, s = [], 0
        for n in sizes[:-1]:
            costs.append(odck.chunk_cost(s, n))
            s += n
        return max(costs) / costs[0]

    fixed = spread(odck.dck_chunk_sizes(S, 12288, 0.0))
    dck = spread(odck.dck_chunk_sizes(S, 12288, 0.65))
    assert fixed > 8.0 and dck < 2.5, (fixed, dck)


def _mutant(old, new):
    src = open(odck.__file__).read()
    assert old in src
    mod = types.ModuleType("dck_mutant")
    exec(compile(src.replace(old, new), "dck_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", [
    ("sigma * ideal + (1.0 - sigma) * sizes[-1]", "(1.0 - sigma) * ideal + sigma * sizes[-1]"),  # weights swapped
    ("math.floor(smoothed + 0.5)", "math.floor(smoothed)"),                                        # rounds down
    ("cost + row_keys(s + n, window) <= target", "cost + row_keys(s + n, window) < target"),       # strict target
    ("return i + 1 if window <= 0 else min(i + 1, window)", "return i if window <= 0 else min(i, window)"),  # no self
])
def test_pins_catch_plausible_mistakes(old, new):
    """Each planted mistake in the restatement fails at least one of the pins above."""
    m = _mutant(old, new)
    g = json.load(open(GOLDEN))
    c = g["case"]
    caught = m.dck_chunk_sizes(c["S"], c["initial"], c["sigma"], c["window"], c["align"]) != g["sizes"]
    caught |= any(m.chunk_cost(s, n, w) != visible_pairs(s, n, w) for s, n, w in [(0, 37, 0), (100, 33, 16)])
    caught |= m.dck_chunk_sizes(65536, 12288, 0.0) != [12288] * 5 + [4096]
    caught |= m.dck_chunk_sizes(10, 4, 1.0, window=1) != [4, 4, 2]
    assert caught


# ---------------------------------------------------------------- the library's planner

CASES = [(S, init, sigma, window, align)
         for S in (1, 5, 1000, 65536, 102400)
         for init in (1, 7, 4096, 12288)
         for sigma in (0.0, 0.25, 0.65, 1.0)
         for window in (0, 128)
         for align in (1, 128)
         if align <= init]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_library_matches_restatement(case):
    S, init, sigma, window, align = case
    assert slope.dck_chunk_sizes(S, init, sigma, window=window, align=align) == \
        odck.dck_chunk_sizes(S, init, sigma, window, align)


def test_library_default_is_dck_12288_sigma_065():
    sizes = slope.dck_chunk_sizes(65536)
    assert sizes[0] == 12288 and sum(sizes) == 65536
    assert sizes == odck.dck_chunk_sizes(65536, 12288, 0.65)


def test_library_argument_errors():
    lib = slope.load()
    E_SHAPE, E_NULL = -3, -1
    assert lib.slope_dck_chunk_sizes(0, 12288, 0.65, 0, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 0, 0.65, 0, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, -0.1, 0, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, 1.5, 0, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, math.nan, 0, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, 0.5, -1, 1, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, 0.5, 0, 101, None, 0) == E_SHAPE
    assert lib.slope_dck_chunk_sizes(1000, 100, 0.5, 0, 1, None, 5) == E_NULL
    # capacity smaller than the count: the count still comes back
    n = lib.slope_dck_chunk_sizes(1000, 100, 0.5, 0, 1, None, 0)
    assert n == len(odck.dck_chunk_sizes(1000, 100, 0.5))
