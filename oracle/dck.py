"""Plain restatement of the dynamic chunk sizing reading, for tests.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``; never by the product package.
It shares no code with the library's planner (``slope_dck_chunk_sizes``), which
uses a closed-form pair count and a bisection; here every cost is a running sum
over rows and every equal-cost size a row-by-row scan, so that the two can be
compared size for size.

The SGLang pipeline-parallelism article (TL;DR, the caption of its throughput
figure) names dynamic chunking with an initial chunked-prefill size of 12K and a
smoothing factor of 0.65, and stops before the algorithm.  The reading:

* a chunk's cost is its visible (query, key) pairs: query row i sees keys
  0..i under the causal mask (its last ``window`` keys with a window);
* the target is the first chunk's cost, the first chunk being ``initial``
  tokens (or S if shorter);
* each later chunk starting at token s moves from the previous size towards
  the largest size whose cost stays within the target (at least one token),
  by exponential smoothing with factor sigma, rounded half up, then down to a
  multiple of ``align`` (at least ``align``), and clipped to the tokens left.
"""
from __future__ import annotations

import math


def row_keys(i: int, window: int) -> int:
    """Keys that query row i sees under the causal mask (and the window)."""
    return i + 1 if window <= 0 else min(i + 1, window)


def chunk_cost(s: int, n: int, window: int = 0) -> int:
    """Visible pairs of the chunk of rows [s, s + n)."""
    return sum(row_keys(i, window) for i in range(s, s + n))


def equal_cost_size(s: int, S: int, target: int, window: int = 0) -> int:
    """Largest n >= 1 (and <= S - s) with chunk_cost(s, n) <= target, by adding rows one at a time."""
    cost, n = 0, 0
    while s + n < S and cost + row_keys(s + n, window) <= target:
        cost += row_keys(s + n, window)
        n += 1
    return max(1, n)


def dck_chunk_sizes(S: int, initial: int = 12288, sigma: float = 0.65, window: int = 0, align: int = 1) -> list:
    first = min(initial, S)
    target = chunk_cost(0, first, window)
    sizes = [first]
    s = first
    while s < S:
        ideal = equal_cost_size(s, S, target, window)
        smoothed = sigma * ideal + (1.0 - sigma) * sizes[-1]
        n = math.floor(smoothed + 0.5)
        n = max(align, (n // align) * align)
        n = min(n, S - s)
        sizes.append(n)
        s += n
    return sizes
