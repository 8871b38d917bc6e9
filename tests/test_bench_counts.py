"""The bench's algorithmic counts (FLOPs per step, attention-kernel bytes per launch, merge
bytes per launch) against brute force over the visibility matrix on small plans (CPU only)."""
import numpy as np
import pytest

import bench
import ring_attention_slope_gb300 as slope
import slope_workloads as wl
from _lib import built_lib


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def visible(S, window):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    m = j <= i
    if window:
        m &= (i - j) < window
    return m


def seen_rows(it, V):
    """Rows of a plan item that see at least one key of its ranges (from the matrix)."""
    q0, q1 = it["q_row0"], it["q_row0"] + it["q_len"]
    seen = np.zeros(q1 - q0, dtype=bool)
    for k0, ln in it["kv"]:
        seen |= V[q0:q1, k0:k0 + ln].any(axis=1)
    return seen


def launch_groups(items, n_launch):
    """Plan launches merged into kernel launches: consecutive ones share a launch while their items
    of live planes (plane 0, or a plane with an item that has a key range) fit in 32."""
    live = {0} | {it["plane"] for it in items if it["kv"]}
    groups, cur = [], []
    for lch in range(n_launch):
        step = [it for it in items if it["launch"] == lch and it["plane"] in live]
        if cur and len(cur) + len(step) > 32:
            groups.append(cur)
            cur = []
        cur += step
    if cur:
        groups.append(cur)
    return groups, live


CASES = [("zigzag", 4, None, 0, 1024), ("zigzag", 4, None, 37, 1024), ("contiguous", 8, None, 0, 1024),
         ("chunked", 3, [300, 1, 723], 0, 1024), ("chunked", 3, [300, 1, 723], 50, 1024),
         ("zigzag", 8, None, 100, 2048), ("zigzag", 16, None, 0, 2048)]


@pytest.mark.parametrize("layout,n,sizes,window,S", CASES)
def test_counts_match_brute_force(layout, n, sizes, window, S):
    w = wl.Workload("t", S, 4, 2, 64, 64, 1.0, layout, n)
    V = visible(S, window)
    items, n_launch, n_planes = slope.cp_prefill_plan(S, n, layout, chunk_sizes=sizes, window=window)
    # FLOPs: every visible pair once per query head
    assert bench.workload_flops(w, window) == V.sum() * w.Hq * 2 * (w.dqk + w.dv)
    # attention kernel: distinct Q rows that see a key, distinct K/V rows, partial writes
    groups, live = launch_groups(items, n_launch)
    per_launch = []
    for g in groups:
        qrows = np.zeros(S, dtype=bool)
        kvrows = np.zeros(S, dtype=bool)
        writes = 0
        for it in g:
            s = seen_rows(it, V)
            qrows[it["q_row0"]:it["q_row0"] + it["q_len"]] |= s
            for k0, ln in it["kv"]:
                kvrows[k0:k0 + ln] = True
            writes += int(s.sum()) * w.Hq * (4 * w.dv + 4) + int((~s).sum()) * w.Hq * 4
        per_launch.append(qrows.sum() * w.Hq * w.dqk * 2 + kvrows.sum() * w.Hkv * (w.dqk + w.dv) * 2 + writes)
    got, n_groups = bench.k1_bytes_per_launch(slope, w, n, sizes, window)
    assert n_groups == len(groups)
    assert got == pytest.approx(sum(per_launch) / len(per_launch), rel=1e-12)
    # merge: lse of every (row, head) of each live plane, the partial of each (row, plane) that saw a
    # key, and the bf16 out + fp32 lse written once
    partial_rows = sum(int(seen_rows(it, V).sum()) for it in items if it["plane"] in live)
    expect = w.Hq * (len(live) * S * 4 + partial_rows * w.dv * 4 + S * (2 * w.dv + 4))
    assert bench.merge_bytes_per_launch(slope, w, n, sizes, window) == expect
