"""Host-side work decomposition: ring steps (zigzag / contiguous), chunked
prefill items and Ulysses head groups cover every visible (query, key, head)
triple exactly once."""
import numpy as np
import pytest

import ring_attention_slope_gb300 as slope
from _lib import built_lib


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def visible(S, window, causal=True):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    m = np.ones((S, S), dtype=bool)
    if causal:
        m &= j <= i
    if window:
        m &= (i - j) < window
    return m


def coverage(items, S, window, causal=True):
    vis = visible(S, window, causal)
    cnt = np.zeros((S, S), dtype=np.int32)
    for it in items:
        q0, q1 = it["q_row0"], it["q_row0"] + it["q_len"]
        for k0, kl in it["kv"]:
            cnt[q0:q1, k0:k0 + kl] += vis[q0:q1, k0:k0 + kl]
    return cnt, vis


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("window", [0, 1, 37, 128])
def test_ring_plan_covers_each_visible_pair_once(layout, N, window):
    parts = 2 * N if layout == "zigzag" else N
    S = parts * 24
    items, n_launches, n_planes = slope.cp_prefill_plan(S, N, layout, window=window)
    assert n_launches == N and n_planes == N
    cnt, vis = coverage(items, S, window)
    assert np.array_equal(cnt, vis.astype(np.int32)), "some visible pair missing or counted twice"
    # The key blocks each rank holds at step t, from the ring's definition (rank r holds the blocks of
    # rank (r - t) mod N): a query row is in at most one item of step t, and a row in none sees no key
    # of its rank's step-t blocks (its partial is the -inf lse written before the launches).
    parts = 2 * N if layout == "zigzag" else N
    sub = S // parts
    owned = (lambda r: [r, 2 * N - 1 - r]) if layout == "zigzag" else (lambda r: [r])
    owner = np.zeros(S, dtype=np.int64)
    for r in range(N):
        for c in owned(r):
            owner[c * sub:(c + 1) * sub] = r
    for t in range(N):
        rows = np.zeros(S, dtype=np.int32)
        for it in items:
            if it["launch"] == t:
                assert it["plane"] == t
                rows[it["q_row0"]:it["q_row0"] + it["q_len"]] += 1
        assert np.all(rows <= 1)
        held = np.zeros((S, S), dtype=bool)
        for r in range(N):
            keys = np.zeros(S, dtype=bool)
            for c in owned((r - t) % N):
                keys[c * sub:(c + 1) * sub] = True
            held[owner == r] = keys
        sees = (vis & held).any(axis=1)
        assert not np.any(sees & (rows == 0)), "a row that sees a key of its step is in no item"
    # zigzag ownership: the ranks' query sub-chunks are r and 2N-1-r (step 0 holds every diagonal)
    if layout == "zigzag":
        starts = sorted({it["q_row0"] // sub for it in items if it["launch"] == 0})
        assert starts == list(range(2 * N))


def test_zigzag_balances_causal_work():
    """Zigzag gives every rank the same causal work; contiguous does not."""
    S, N = 64 * 16, 8
    vis = visible(S, 0)

    def per_rank(layout):
        items, _, _ = slope.cp_prefill_plan(S, N, layout)
        parts = 2 * N if layout == "zigzag" else N
        sub = S // parts
        work = np.zeros(N)
        for it in items:
            a = it["q_row0"] // sub
            r = a if a < N else 2 * N - 1 - a
            if layout == "contiguous":
                r = a
            for k0, kl in it["kv"]:
                work[r] += vis[it["q_row0"]:it["q_row0"] + it["q_len"], k0:k0 + kl].sum()
        return work

    zz = per_rank("zigzag")
    ct = per_rank("contiguous")
    assert zz.max() / zz.min() < 1.01
    assert ct.max() / ct.min() > 5


@pytest.mark.parametrize("sizes", [[300], [100, 200], [12, 40, 7, 141, 100], None])
@pytest.mark.parametrize("window", [0, 16])
def test_chunked_plan(sizes, window):
    S = 300
    n = len(sizes) if sizes else 4
    items, n_launches, n_planes = slope.cp_prefill_plan(S, n, "chunked", chunk_sizes=sizes, window=window)
    assert n_launches == n and n_planes == 2
    cnt, vis = coverage(items, S, window)
    assert np.array_equal(cnt, vis.astype(np.int32))
    starts = np.cumsum([0] + (sizes or [75] * 4))[:-1]
    lens = sizes or [75] * 4
    for c in range(n):
        its = [it for it in items if it["launch"] == c]
        # the first chunk has no prefix to see, so no prefix partial; every other chunk's first rows see
        # the tokens before it (with a window, only rows within the window of them do)
        assert sorted(it["plane"] for it in its) == ([0, 1] if c > 0 else [1])
        for it in its:
            assert it["q_row0"] == starts[c] and 1 <= it["q_len"] <= lens[c]
            if it["plane"] == 1 or window == 0:
                assert it["q_len"] == lens[c]
            else:
                assert it["q_len"] == min(lens[c], window - 1)
            for k0, kl in it["kv"]:
                if it["plane"] == 0:
                    assert k0 + kl <= starts[c]  # prefix partial: earlier tokens only
                else:
                    assert k0 >= starts[c]       # own partial: the chunk itself


def test_plan_errors():
    with pytest.raises(slope.SlopeError):
        slope.cp_prefill_plan(1000, 8, "zigzag")
    with pytest.raises(slope.SlopeError):
        slope.cp_prefill_plan(1000, 2, "chunked", chunk_sizes=[400, 500])


@pytest.mark.parametrize("N", [1, 2, 4, 8, 32])
@pytest.mark.parametrize("window", [0, 1, 37])
def test_ulysses_plan_covers_each_head_and_visible_pair_once(N, window):
    """Rank u owns head group u of N over every token; together the ranks cover every
    (head, visible pair) once, with one item per rank, no partial plane and no merge."""
    S, Hq = 200, 64
    items, n_launches, n_planes = slope.cp_prefill_plan(S, N, "ulysses", window=window)
    assert n_launches == N and n_planes == 1 and len(items) == N
    cnt_heads = np.zeros((Hq, S, S), dtype=np.int32)
    vis = visible(S, window)
    for it in items:
        assert it["n_head_groups"] == N and it["plane"] == 0 and it["launch"] == it["head_group"]
        assert it["q_row0"] == 0 and it["q_len"] == S
        h0, h1 = it["head_group"] * Hq // N, (it["head_group"] + 1) * Hq // N
        cnt, _ = coverage([it], S, window)
        cnt_heads[h0:h1] += cnt
    assert np.array_equal(cnt_heads, np.broadcast_to(vis.astype(np.int32), cnt_heads.shape))
    # every other layout lists all heads in every entry
    for layout, n in (("zigzag", 4), ("chunked", 3)):
        its, _, _ = slope.cp_prefill_plan(240, n, layout)
        assert all(it["head_group"] == 0 and it["n_head_groups"] == 1 for it in its)


def test_ulysses_plan_errors():
    for N in (0, 33):
        with pytest.raises(slope.SlopeError):
            slope.cp_prefill_plan(256, N, "ulysses")


@pytest.mark.parametrize("layout,N,u,sizes", [("zigzag", 4, 2, None), ("contiguous", 8, 8, None),
                                              ("chunked", 3, 4, [50, 1, 141]), ("zigzag", 1, 32, None)])
@pytest.mark.parametrize("window", [0, 37])
def test_ulysses_ring_plan_splits_each_item_by_head_group(layout, N, u, sizes, window):
    """Ulysses x Ring: every base item becomes u head-group items of the same launch and plane; together
    they cover every (head, visible pair) once."""
    S = 192 if sizes is None else sum(sizes)
    Hq = 64
    base, nl0, np0 = slope.cp_prefill_plan(S, N, layout, chunk_sizes=sizes, window=window)
    items, nl, npl = slope.cp_prefill_plan(S, N, slope.layout_code(layout, u), chunk_sizes=sizes, window=window)
    assert (nl, npl) == (nl0, np0) and len(items) == u * len(base)
    for i, it in enumerate(items):
        b = base[i // u]
        assert it["head_group"] == i % u and it["n_head_groups"] == u
        assert {k: it[k] for k in ("launch", "plane", "q_row0", "q_len", "kv")} == \
            {k: b[k] for k in ("launch", "plane", "q_row0", "q_len", "kv")}
    vis = visible(S, window)
    cnt = np.zeros((Hq, S, S), dtype=np.int32)
    for it in items:
        h0, h1 = it["head_group"] * Hq // u, (it["head_group"] + 1) * Hq // u
        c, _ = coverage([it], S, window)
        cnt[h0:h1] += c
    assert np.array_equal(cnt, np.broadcast_to(vis.astype(np.int32), cnt.shape))


def test_ulysses_ring_plan_errors():
    with pytest.raises(slope.SlopeError):
        slope.cp_prefill_plan(256, 4, slope.layout_code("ulysses", 2))   # Ulysses takes no extra degree
    with pytest.raises(slope.SlopeError):
        slope.cp_prefill_plan(256, 4, slope.layout_code("zigzag", 33))   # more than 32 groups
    with pytest.raises(slope.SlopeError):
        slope.cp_prefill_plan(256, 4, 1 | (1 << 16))                      # bits above the degree


@pytest.mark.parametrize("layout,N,sizes", [("zigzag", 1, None), ("zigzag", 4, None), ("zigzag", 16, None),
                                            ("contiguous", 3, None), ("contiguous", 8, None),
                                            ("chunked", 3, [100, 250, 170]), ("chunked", 5, None)])
@pytest.mark.parametrize("window", [0, 1, 37, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_fused_plan_covers_each_visible_pair_once(layout, N, sizes, window, causal):
    """SLOPE_CP_FUSED: one item per query sub-chunk (ring) or chunk, each over one key range, writing the
    final output directly (one plane); together they cover every visible pair exactly once, and every
    query row belongs to exactly one item."""
    S = 520 if layout == "chunked" else (2 * N if layout == "zigzag" else N) * 24
    items, n_launches, n_planes = slope.cp_prefill_plan(S, N, layout, chunk_sizes=sizes, causal=causal,
                                                        window=window, fused=True)
    assert n_planes == 1 and n_launches == N
    assert all(it["plane"] == 0 and len(it["kv"]) <= 1 for it in items)
    cnt, vis = coverage(items, S, window, causal)
    assert np.array_equal(cnt, vis.astype(np.int32)), "some visible pair missing or counted twice"
    rows = np.zeros(S, dtype=np.int32)
    for it in items:
        rows[it["q_row0"]:it["q_row0"] + it["q_len"]] += 1
    assert np.all(rows == 1)
    # each item's range is exactly the union of the keys its rows see (nothing wider)
    for it in items:
        q0, q1 = it["q_row0"], it["q_row0"] + it["q_len"]
        seen = np.flatnonzero(vis[q0:q1].any(axis=0))
        if it["kv"]:
            (k0, kl), = it["kv"]
            assert k0 == seen[0] and k0 + kl == seen[-1] + 1
        else:
            assert seen.size == 0
    # the ring's items per rank: zigzag r owns sub-chunks r and 2N-1-r
    if layout == "zigzag":
        sub = S // (2 * N)
        for r in range(N):
            mine = sorted(it["q_row0"] // sub for it in items if it["launch"] == r)
            assert mine == sorted({r, 2 * N - 1 - r})


def test_plan_ex_flags():
    """plan_ex with flags 0 is the plain plan; conflicting or unknown flags are refused."""
    lib = slope.load()
    assert lib.slope_cp_prefill_plan_ex(1024, 4, 1, None, 1, 0, 3, None, 0, None, None) == -8
    assert lib.slope_cp_prefill_plan_ex(1024, 4, 1, None, 1, 0, 8, None, 0, None, None) == -8
    a, la, pa = slope.cp_prefill_plan(1024, 4, "zigzag", window=64)
    b = lib.slope_cp_prefill_plan(1024, 4, 1, None, 1, 64, None, 0, None, None)
    assert len(a) == b and la == 4 and pa == 4
