"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances (bf16 inputs, fp32 accumulation): output max-abs <= 2e-2 and
relative L2 <= 5e-3, log-sum-exp max-abs <= 1e-3; rows that see no key must
give exactly out = 0 and lse = -inf on both sides.
"""
import math
import os
import re

import numpy as np
import pytest
import torch

import oracle
import ring_attention_slope_gb300 as slope
import slope_workloads as wl

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_REL_L2, LSE_MAX = 2e-2, 5e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    slope.build()
    slope.load()
    st, _ = slope.device_status()
    assert st == 0


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what):
    og = np.asarray(out_gpu, dtype=np.float64)
    lg = np.asarray(lse_gpu, dtype=np.float64)
    assert og.shape == out_ref.shape, f"{what}: out shape {og.shape} vs {out_ref.shape}"
    assert lg.shape == lse_ref.shape, f"{what}: lse shape {lg.shape} vs {lse_ref.shape}"
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), f"{what}: -inf rows differ"
    assert not np.any(np.isnan(lg)), f"{what}: NaN lse"
    fin = ~empty
    if fin.any():
        le = np.max(np.abs(lg[fin] - lse_ref[fin]))
        assert le <= LSE_MAX, f"{what}: lse max-abs {le:.3e}"
    d = og - out_ref
    me = np.max(np.abs(d)) if d.size else 0.0
    nr = np.linalg.norm(out_ref)
    rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
    assert me <= OUT_MAX, f"{what}: out max-abs {me:.3e}"
    assert rel <= OUT_REL_L2, f"{what}: out rel-L2 {rel:.3e}"
    # empty rows: exactly zero output
    emp_rows = empty.T  # [rows, heads]
    if emp_rows.any():
        assert np.all(og[emp_rows] == 0.0), f"{what}: nonzero output for rows with no visible key"
    return me, rel


def qkv(S, Hq, Hkv, dqk, dv, seed, Skv=None, scale_v=1.0, device="cuda"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Skv = S if Skv is None else Skv
    q = (torch.randn(S, Hq, dqk, generator=g) * scale_v).to(torch.bfloat16)
    k = (torch.randn(Skv, Hkv, dqk, generator=g) * scale_v).to(torch.bfloat16)
    v = (torch.randn(Skv, Hkv, dv, generator=g) * scale_v).to(torch.bfloat16)
    return q.to(device), k.to(device), v.to(device)


# ---------------------------------------------------------------- device status / bounded waits

def test_timeout_selftest_reports_and_context_survives():
    slope.timeout_selftest(2_000_000)  # 2 ms limit on a barrier nothing completes
    st, site = slope.device_status()
    assert st == -7 and site == 99
    assert slope.device_status() == (0, 0)  # cleared by the read
    q, k, v = qkv(256, 2, 1, 64, 64, seed=1)
    out, lse = slope.attn_partial(q, k, v, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    compare(out.cpu(), lse.cpu(), ro, rl, "after timeout self-test")
    assert slope.device_status() == (0, 0)


# ---------------------------------------------------------------- work tiles claimed at run time

# The attention kernels for dqk >= 128 claim their work tiles from device counters that the
# library hands out round robin, SLOPE_TILE_COUNTERS of them per device (each 0 between launches).
TILE_COUNTERS = int(re.search(r"#define SLOPE_TILE_COUNTERS (\d+)",
                              open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                                "include", "slope.h")).read()).group(1))


@pytest.mark.parametrize("S,H", [(1100, 6), (2100, 48)])
def test_claimed_tiles_same_bits_every_launch(S, H):
    """Five MLA-shaped launches in a row, each claiming its tiles from the next counter (so CTAs take the
    tiles in a different order each time; at S = 2100 with 48 heads, 432 tiles give most CTAs several):
    the same bits every time, and the oracle's values (on a subset of heads at the larger size)."""
    q, k, v = qkv(S, H, H, 192, 128, seed=31 + S)
    runs = []
    for _ in range(5):
        out, lse = slope.attn_partial(q, k, v, causal=True)
        runs.append((out, lse))
    torch.cuda.synchronize()
    heads = None if H <= 8 else [0, 1, 23, 46, 47]
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, heads=heads)
    og, lg = runs[0][0].cpu(), runs[0][1].cpu()
    if heads is not None:
        og, lg = og[:, heads], lg[heads]
    compare(og, lg, ro, rl, f"claimed tiles S={S} H={H}")
    for out, lse in runs[1:]:
        assert torch.equal(out, runs[0][0]) and torch.equal(lse, runs[0][1])
    assert slope.device_status() == (0, 0)


def test_claimed_tile_counter_returns_to_zero_after_an_abort():
    """A launch that starts while the status word holds an error computes nothing, yet its CTAs still claim
    past the end and put the counter back to 0: every later launch, up to and past the one that reuses
    that counter, computes every tile."""
    S, H = 700, 4
    q, k, v = qkv(S, H, H, 192, 128, seed=33)
    out = torch.empty((S, H, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((H, S), dtype=torch.float32, device="cuda")
    ref_out, ref_lse = slope.attn_partial(q, k, v, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    compare(ref_out.cpu(), ref_lse.cpu(), ro, rl, "before the aborted launch")
    slope.timeout_selftest(2_000_000)  # the status word now holds a timeout
    slope.attn_partial(q, k, v, causal=True, out=out, lse=lse)  # its CTAs see it and return at once
    st, site = slope.device_status()
    assert st == -7 and site == 99
    bad = torch.zeros((), dtype=torch.bool, device="cuda")
    for _ in range(TILE_COUNTERS + 3):
        out.fill_(math.nan)
        lse.fill_(math.nan)
        slope.attn_partial(q, k, v, causal=True, out=out, lse=lse)
        bad |= ~(out == ref_out).all()  # a tile left uncomputed keeps its NaN
        bad |= ~(lse == ref_lse).all()
    torch.cuda.synchronize()
    assert not bool(bad)
    assert slope.device_status() == (0, 0)


# ---------------------------------------------------------------- partial attention

PARTIAL_CASES = [
    # Sq, Skv, Hq, Hkv, dqk, dv, q_off, kv_off, causal, window
    (256, 256, 2, 1, 64, 64, 0, 0, True, 0),
    (300, 300, 4, 2, 64, 64, 0, 0, True, 0),          # ragged query tail, several tiles
    (517, 700, 4, 1, 64, 64, 183, 0, True, 0),        # queries after a longer key prefix
    (384, 384, 8, 8, 64, 64, 1000, 0, False, 0),      # unmasked
    (260, 390, 4, 2, 64, 64, 390, 0, True, 0),        # keys all earlier: full tiles + ragged key tail
    (200, 333, 2, 1, 64, 64, 0, 100, True, 0),        # keys partly in the future; first rows see none
    (640, 640, 2, 1, 64, 64, 0, 0, True, 128),        # sliding window 128
    (500, 500, 2, 2, 64, 64, 0, 0, True, 1),          # window 1: out = v
    (333, 333, 4, 1, 64, 64, 0, 0, True, 77),
    (256, 256, 4, 2, 128, 64, 0, 0, True, 0),
    (300, 410, 2, 1, 128, 128, 110, 0, True, 0),
    (384, 384, 2, 2, 192, 128, 0, 0, True, 0),        # MLA-shaped
    (270, 513, 3, 3, 192, 128, 243, 0, True, 0),
    (1, 1, 1, 1, 64, 64, 0, 0, True, 0),
    (129, 1, 2, 1, 64, 64, 5, 4, True, 0),
    (300, 410, 4, 2, 64, 128, 110, 0, True, 0),       # dqk 64, dv 128 (P over S, turns)
    (384, 384, 2, 2, 64, 128, 0, 0, True, 77),
    (270, 513, 3, 3, 192, 64, 243, 0, True, 0),       # dqk 192, dv 64 (separate P)
    (333, 333, 4, 4, 192, 64, 0, 0, False, 0),
]


@pytest.mark.parametrize("case", PARTIAL_CASES, ids=lambda c: "x".join(map(str, c)))
def test_attn_partial_matches_oracle(case):
    Sq, Skv, Hq, Hkv, dqk, dv, q_off, kv_off, causal, window = case
    q, k, v = qkv(Sq, Hq, Hkv, dqk, dv, seed=hash(case) % 10000, Skv=Skv, scale_v=1.0)
    out, lse = slope.attn_partial(q, k, v, q_off=q_off, kv_off=kv_off, causal=causal, window=window)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), q_pos0=q_off, kv_pos0=kv_off, causal=causal,
                              window=window)
    compare(out.cpu(), lse.cpu(), ro, rl, f"partial {case}")
    assert slope.device_status() == (0, 0)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d,dv", [(64, 64), (64, 128), (128, 64), (128, 128), (192, 64), (192, 128)])
def test_attn_partial_score_jumps_inside_a_key_tile(causal, d, dv):
    """Keys whose scores jump by tens of log2 units inside one 128-key tile and again in
    later tiles: the running max moves many times and the row sum and O are rescaled
    by factors down to 2^-100 and below (with P in its own TMEM columns at dv = 64 and
    over S at dv = 128)."""
    S, Hq, Hkv = 640, 2, 1
    g = torch.Generator().manual_seed(77)
    u = torch.randn(d, generator=g)
    u = u / u.norm() * 8.0  # |u|^2 = 64: key a*u scores about 64a*scale against q ~ u + noise
    q = (torch.randn(S, Hq, d, generator=g) + u).to(torch.bfloat16)
    k = torch.randn(S, Hkv, d, generator=g) * 0.1
    v = torch.randn(S, Hkv, dv, generator=g)
    for j, a in [(40, 1.5), (70, 4.0), (100, 8.0), (170, 12.0), (300, 20.0), (333, 3.0), (520, 30.0)]:
        k[j, :] = a * u
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    out, lse = slope.attn_partial(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, causal=causal)
    compare(out.cpu(), lse.cpu(), ro, rl, f"score jumps causal={causal} d={d}/{dv}")
    assert slope.device_status() == (0, 0)


def test_attn_partial_no_keys_and_future_keys():
    q, k, v = qkv(200, 4, 2, 64, 64, seed=5, Skv=300)
    out, lse = slope.attn_partial(q, k, v, q_off=0, kv_off=500, causal=True)  # every key in the future
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    out, lse = slope.attn_partial(q, k[:0], v[:0], causal=True)  # no keys at all
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("q_off,kv_off,causal,window", [
    (2**28 - 300, 2**28 - 300 - 250, True, 0),       # the last positions allowed
    (-2**28 + 250, -2**28, True, 100),               # the first positions allowed
    (2**28 - 300, -2**28, False, 0),                 # query - key position differences near 2^29
    (-2**28, 2**28 - 250, False, 2**30),             # keys all "after" the queries, the largest window
    (2**28 - 300, 2**28 - 450, True, 2**30),
])
def test_attn_partial_extreme_positions(q_off, kv_off, causal, window):
    """Positions at the ends of the accepted range [-2^28, 2^28]: the kernel's 32-bit position differences
    (less the window) do not overflow, and the masks match the oracle's 64-bit ones."""
    q, k, v = qkv(300, 4, 2, 64, 64, seed=q_off % 9973, Skv=250)
    out, lse = slope.attn_partial(q, k, v, q_off=q_off, kv_off=kv_off, causal=causal, window=window)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), q_pos0=q_off, kv_pos0=kv_off, causal=causal, window=window)
    compare(out.cpu(), lse.cpu(), ro, rl, f"positions {q_off} {kv_off}")
    assert slope.device_status() == (0, 0)


def test_attn_partial_window1_is_exact_identity():
    q, k, v = qkv(300, 2, 1, 64, 64, seed=6)
    out, lse = slope.attn_partial(q, k, v, causal=True, window=1)
    torch.cuda.synchronize()
    G = 2
    ref = v.float().repeat_interleave(G, dim=1)
    torch.testing.assert_close(out, ref, rtol=1e-6, atol=0)
    sii = (q.float() * k.float().repeat_interleave(G, dim=1)).sum(-1) / 8.0  # scale 1/sqrt(64)
    torch.testing.assert_close(lse, sii.T.contiguous(), rtol=0, atol=1e-5)


def test_attn_partial_strided_views():
    """Q/K/V as head-slices of larger packed tensors; out/lse as views with padding."""
    S, Hq, Hkv, d = 300, 4, 2, 64
    g = torch.Generator().manual_seed(11)
    qkv_packed = torch.randn(S, Hq + 2 * Hkv, d, generator=g).to(torch.bfloat16).cuda()
    q, k, v = qkv_packed[:, :Hq], qkv_packed[:, Hq:Hq + Hkv], qkv_packed[:, Hq + Hkv:]
    out_big = torch.full((S, Hq + 1, d), 7.0, device="cuda")
    lse_big = torch.full((Hq, S + 16), 7.0, device="cuda")
    out, lse = slope.attn_partial(q, k, v, causal=True, out=out_big[:, :Hq], lse=lse_big[:, :S])
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    compare(out.cpu(), lse.cpu(), ro, rl, "strided views")
    assert torch.all(out_big[:, Hq] == 7.0) and torch.all(lse_big[:, S:] == 7.0)


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("dv", [64, 128, 192])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 16, 32])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge_matches_oracle(dv, n, out_dtype):
    S, H = 333, 6
    g = torch.Generator().manual_seed(n * 100 + dv)
    outs = [torch.randn(S, H, dv, generator=g) for _ in range(n)]
    lses = [torch.randn(H, S, generator=g) * 4 + 2 for _ in range(n)]
    for i, l in enumerate(lses):  # some partials see nothing for some rows
        l[:, (torch.arange(S) % (i + 2)) == 0] = -math.inf
    lses[0][:, :5] = -math.inf
    for l in lses:
        l[:, :3] = -math.inf  # rows 0..2 see nothing at all
    out, lse = slope.lse_merge([o.cuda() for o in outs], [x.cuda() for x in lses], out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rl = oracle.merge([o.double().numpy() for o in outs], [x.double().numpy() for x in lses])
    compare(out.float().cpu(), lse.cpu(), ro, rl, f"merge n={n} dv={dv} {out_dtype}")


# ---------------------------------------------------------------- whole prefill: tiny workload, all layouts

def tiny():
    return wl.WORKLOADS[0]


@pytest.mark.parametrize("layout,n", [("zigzag", 4), ("zigzag", 2), ("zigzag", 1), ("contiguous", 4),
                                      ("contiguous", 8), ("chunked", 3), ("chunked", 1)])
@pytest.mark.parametrize("window", [0, 128])
def test_cp_prefill_tiny_all_layouts(layout, n, window):
    w = tiny()
    q, k, v = wl.workload_qkv(w, device="cuda")
    out, lse = slope.cp_prefill(q, k, v, n, layout, window=window)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    compare(out.float().cpu(), lse.cpu(), ro, rl, f"tiny {layout} n={n} W={window}")
    assert slope.device_status() == (0, 0)


def test_cp_prefill_skips_ring_steps_without_keys():
    """With a window shorter than a sub-chunk, zigzag ring steps 2..N-2 see no key: no launch, no merge input."""
    S, Hq, Hkv, d, N, W = 2048, 4, 2, 64, 8, 100
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=17)
    items, n_steps, _ = slope.cp_prefill_plan(S, N, "zigzag", window=W)
    live = {it["plane"] for it in items if it["kv"]} | {0}
    assert live == {0, 1, N - 1}
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps + 2)]
    out, lse, n_launches, kinds = slope.cp_prefill_timed(q, k, v, N, "zigzag", events, window=W)
    torch.cuda.synchronize()
    # the live planes' lse filled with -inf, then one attention launch (the 16 items of step 0 and the 14 of
    # steps 1 and 7 whose rows see the previous sub-chunk's last keys: 30 <= 32), then the merge
    assert kinds == [2, 0, 1] and n_launches == 3
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=W)
    compare(out.float().cpu(), lse.cpu(), ro, rl, "zigzag-8 window 100")
    assert slope.device_status() == (0, 0)


def test_cp_prefill_chunked_ragged_sizes_and_fp32_out():
    S, Hq, Hkv, d = 1000, 4, 2, 64
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=21, scale_v=0.8)
    sizes = [130, 1, 257, 255, 357]
    out, lse = slope.cp_prefill(q, k, v, len(sizes), "chunked", chunk_sizes=sizes, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    compare(out.cpu(), lse.cpu(), ro, rl, "chunked ragged")


def test_cp_prefill_layout_invariance():
    """Zigzag, contiguous and chunked decompositions agree with each other."""
    S, Hq, Hkv, d = 2048, 4, 1, 64
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=31)
    res = []
    for layout, n in (("zigzag", 4), ("contiguous", 8), ("chunked", 5), ("zigzag", 1)):
        o, l = slope.cp_prefill(q, k, v, n, layout, out_dtype=torch.float32)
        res.append((o, l))
    torch.cuda.synchronize()
    base_o, base_l = res[0][0].cpu().double().numpy(), res[0][1].cpu().double().numpy()
    for o, l in res[1:]:
        compare(o.cpu(), l.cpu(), base_o, base_l, "layout invariance")


def test_cp_prefill_mla_shape_small():
    S, H = 1536, 4
    q, k, v = qkv(S, H, H, 192, 128, seed=41, scale_v=0.3)
    sizes = [700, 500, 336]
    out, lse = slope.cp_prefill(q, k, v, 3, "chunked", chunk_sizes=sizes)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    compare(out.float().cpu(), lse.cpu(), ro, rl, "mla small")


# ---------------------------------------------------------------- full-size workloads, sampled rows/heads

def check_full_workload(w, window, rows_random=4096, bf16_partials=False, fused=False, sizes=None):
    q, k, v = wl.workload_qkv(w, device="cuda")
    sizes = wl.chunk_sizes(w) if sizes is None else sizes
    n = len(sizes) if sizes is not None else wl.n_chunks(w)
    out, lse = slope.cp_prefill(q, k, v, n, w.layout, chunk_sizes=sizes, window=window, bf16_partials=bf16_partials,
                                fused=fused)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    rows = wl.sample_rows(w, n_random=rows_random)
    if sizes is not None:  # the first and last rows of every chunk actually used
        edges = np.cumsum([0] + list(sizes))
        extra = [np.arange(a, min(b, a + 64)) for a, b in zip(edges[:-1], edges[1:])]
        extra += [np.arange(max(a, b - 64), b) for a, b in zip(edges[:-1], edges[1:])]
        rows = np.unique(np.concatenate([rows] + extra)).astype(np.int64)
    heads = wl.sample_heads(w)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    ro, rl = oracle.attention(qc, kc, vc, causal=True, window=window, rows=rows, heads=heads)
    og = out[torch.from_numpy(rows).cuda()][:, heads].float().cpu()
    lg = lse[heads][:, torch.from_numpy(rows).cuda()].cpu()
    compare(og, lg, ro, rl, f"{w.name} W={window} bf16_partials={bf16_partials} fused={fused}")
    # properties at every row: finite outputs, lse >= the log of... finite and bounded
    assert torch.isfinite(out.float()).all()
    assert torch.isfinite(lse).all()


def test_full_causal_gqa_s32k_zigzag8():
    check_full_workload(wl.WORKLOADS[1], 0)


def test_full_chunked_prefill_s64k():
    check_full_workload(wl.WORKLOADS[2], 0)


@pytest.mark.parametrize("window", [0, 128])
def test_full_s100k_zigzag16(window):
    check_full_workload(wl.WORKLOADS[3], window, rows_random=2048)


def test_full_mla_s64k_chunked_var():
    check_full_workload(wl.WORKLOADS[4], 0)


@pytest.mark.parametrize("layout,n,dims", [("zigzag", 4, (8, 2, 64, 64)), ("chunked", 3, (8, 2, 64, 64)),
                                           ("zigzag", 4, (4, 4, 192, 128))])
def test_cp_prefill_host_buffers_overlapped_calls(layout, n, dims):
    """Three host-buffer prefills on two alternating device-buffer sets and three streams: each host
    result equals slope_cp_prefill on the same inputs, bit for bit (the third call reuses the first
    call's device buffers while the second call's work may still run).  With the MLA head sizes the
    attention launches of overlapping calls claim their work tiles from separate counters."""
    S = 2048
    Hq, Hkv, d, dv = dims
    calls = [qkv(S, Hq, Hkv, d, dv, seed=90 + i, device="cpu") for i in range(3)]
    hosts = [tuple(t.pin_memory() for t in c) for c in calls]
    sets = [dict(q=torch.empty(S, Hq, d, dtype=torch.bfloat16, device="cuda"),
                 k=torch.empty(S, Hkv, d, dtype=torch.bfloat16, device="cuda"),
                 v=torch.empty(S, Hkv, dv, dtype=torch.bfloat16, device="cuda"),
                 out=torch.empty(S, Hq, dv, dtype=torch.bfloat16, device="cuda"),
                 lse=torch.empty(Hq, S, dtype=torch.float32, device="cuda")) for _ in range(2)]
    houts = [torch.empty(S, Hq, dv, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    hlses = [torch.empty(Hq, S, dtype=torch.float32).pin_memory() for _ in range(3)]
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ws = None
    for i in range(3):
        b = sets[i % 2]
        ws = slope.cp_prefill_host(*hosts[i], houts[i], hlses[i], b["q"], b["k"], b["v"], b["out"], b["lse"], n,
                                   layout, workspace=ws, copy_in_stream=s_in, compute_stream=s_c,
                                   copy_out_stream=s_out)
    torch.cuda.synchronize()
    for i in range(3):
        ro, rl = slope.cp_prefill(*(t.cuda() for t in calls[i]), n, layout)
        torch.cuda.synchronize()
        assert torch.equal(houts[i], ro.cpu()), f"call {i}: out differs"
        assert torch.equal(hlses[i], rl.cpu()), f"call {i}: lse differs"
    assert slope.device_status() == (0, 0)


@pytest.mark.parametrize("Sq,Hq,Hkv,d,window", [(1000, 8, 2, 64, 0), (777, 4, 4, 64, 100), (640, 4, 4, 128, 0)])
def test_attn_partial_bf16_out_is_the_fp32_out_rounded(Sq, Hq, Hkv, d, window):
    """bf16 output: the same normalised rows as the fp32 output, rounded to bf16 (same kernel arithmetic),
    including rows of ragged 32-row chunks that are stored directly."""
    q, k, v = qkv(Sq, Hq, Hkv, d, d, seed=Sq + d)
    o32, l32 = slope.attn_partial(q, k, v, causal=True, window=window)
    o16, l16 = slope.attn_partial(q, k, v, causal=True, window=window, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)
    assert slope.device_status() == (0, 0)


@pytest.mark.parametrize("layout,n", [("zigzag", 8), ("chunked", 3)])
def test_fused_single_launch_matches_ring_and_oracle(layout, n):
    """The whole causal attention in one attention launch (bf16 out, no partials, no merge) agrees with
    the ring / chunked decomposition and with the oracle on sampled rows."""
    S, Hq, Hkv, d = 4096, 8, 2, 64
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=123, scale_v=0.5)
    fo, fl = slope.attn_partial(q, k, v, causal=True, out_dtype=torch.bfloat16)
    ro, rl = slope.cp_prefill(q, k, v, n, layout)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(S - 130, S),
                                     np.random.default_rng(5).integers(0, S, 600)]))
    oo, ol = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, rows=rows)
    compare(fo.float().cpu()[rows], fl.cpu()[:, rows], oo, ol, f"fused vs oracle ({layout})")
    d_out = (fo.float() - ro.float()).abs().max().item()
    d_lse = (fl - rl).abs().max().item()
    assert d_out <= 2e-2 and d_lse <= 1e-3, (d_out, d_lse)
    assert slope.device_status() == (0, 0)


def test_cp_prefill_host_more_buffer_sets_than_tracked():
    """18 device-buffer sets in rotation (the library tracks 16: older sets are waited for and their
    slots reused), the first set reused at the end, and no lse: every result equals cp_prefill."""
    S, Hq, Hkv, d, n = 512, 4, 1, 64, 2
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sets = [dict(q=torch.empty(S, Hq, d, dtype=torch.bfloat16, device="cuda"),
                 k=torch.empty(S, Hkv, d, dtype=torch.bfloat16, device="cuda"),
                 v=torch.empty(S, Hkv, d, dtype=torch.bfloat16, device="cuda"),
                 out=torch.empty(S, Hq, d, dtype=torch.bfloat16, device="cuda")) for _ in range(18)]
    order = list(range(18)) + [0, 1]
    inputs, outs = [], []
    ws = None
    for j, i in enumerate(order):
        hq, hk, hv = (t.pin_memory() for t in qkv(S, Hq, Hkv, d, d, seed=300 + j, device="cpu"))
        ho = torch.empty(S, Hq, d, dtype=torch.bfloat16).pin_memory()
        b = sets[i]
        ws = slope.cp_prefill_host(hq, hk, hv, ho, None, b["q"], b["k"], b["v"], b["out"], None, n, "zigzag",
                                   workspace=ws, copy_in_stream=s_in, compute_stream=s_c, copy_out_stream=s_out)
        inputs.append((hq, hk, hv))
        outs.append(ho)
    torch.cuda.synchronize()
    for j in range(len(order)):
        ro, _ = slope.cp_prefill(*(t.cuda() for t in inputs[j]), n, "zigzag", want_lse=False)
        torch.cuda.synchronize()
        assert torch.equal(outs[j], ro.cpu()), f"call {j} (buffer set {order[j]})"
    assert slope.device_status() == (0, 0)


# ---------------------------------------------------------------- bf16 partials (slope_cp_prefill_ex)

@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("n", [2, 5, 32])
def test_lse_merge_bf16_partials_are_widened_exactly(dv, n):
    """bf16 partials merge to exactly what their fp32 copies merge to (the merge widens each
    element and then runs the fp32 arithmetic), and match the oracle on those partials."""
    S, H = 333, 6
    g = torch.Generator().manual_seed(7 * n + dv)
    outs = [torch.randn(S, H, dv, generator=g).to(torch.bfloat16) for _ in range(n)]
    lses = [torch.randn(H, S, generator=g) * 4 + 2 for _ in range(n)]
    for i, l in enumerate(lses):
        l[:, (torch.arange(S) % (i + 3)) == 1] = -math.inf
    for l in lses:
        l[:, :2] = -math.inf
    lc = [x.cuda() for x in lses]
    ob, lb = slope.lse_merge([o.cuda() for o in outs], lc, out_dtype=torch.float32)
    of, lf = slope.lse_merge([o.float().cuda() for o in outs], lc, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(ob, of) and torch.equal(lb, lf)
    ro, rl = oracle.merge([o.double().numpy() for o in outs], [x.double().numpy() for x in lses])
    compare(ob.cpu(), lb.cpu(), ro, rl, f"bf16-partial merge n={n} dv={dv}")


def _workspace_planes(ws, S, Hq, dv, n_planes, dtype):
    """The partial planes [n_planes, S, Hq, dv] and fp32 lse planes [n_planes, S, Hq] (at the next
    256-byte boundary) that a prefill leaves in its workspace."""
    elem = 2 if dtype == torch.bfloat16 else 4
    out_bytes = n_planes * S * Hq * dv * elem
    lse_off = (out_bytes + 255) // 256 * 256
    planes = ws[:out_bytes].view(dtype).view(n_planes, S, Hq, dv)
    lses = ws[lse_off:lse_off + n_planes * S * Hq * 4].view(torch.float32).view(n_planes, S, Hq)
    return planes, lses


@pytest.mark.parametrize("layout,n,window,dqk,dv,sizes", [
    ("zigzag", 4, 0, 64, 64, None), ("contiguous", 8, 0, 128, 128, None), ("zigzag", 8, 100, 64, 64, None),
    ("chunked", 3, 0, 128, 64, [700, 1, 1347]), ("chunked", 2, 300, 192, 128, [1000, 1048])])
def test_cp_prefill_bf16_partials_are_the_fp32_partials_rounded(layout, n, window, dqk, dv, sizes):
    """SLOPE_CP_BF16_PARTIALS changes nothing but the rounding of each written partial element:
    every written element is the fp32 path's element rounded to bf16 (round to nearest even),
    the lse planes are bit-identical, and the result stays within the oracle tolerances and within
    one bf16 rounding of the largest |v| of the fp32-partial result."""
    S, Hq, Hkv = 2048, 4, 2
    q, k, v = qkv(S, Hq, Hkv, dqk, dv, seed=53 + n + dqk)
    n_planes = 2 if layout == "chunked" else n
    ws32 = torch.full((slope.cp_prefill_workspace_size(S, Hq, dv, n, layout, sizes),), 0xFF, dtype=torch.uint8,
                      device="cuda")
    ws16 = torch.full((slope.cp_prefill_workspace_size(S, Hq, dv, n, layout, sizes, bf16_partials=True),), 0xFF,
                      dtype=torch.uint8, device="cuda")
    assert ws16.numel() < ws32.numel()
    o32, l32 = slope.cp_prefill(q, k, v, n, layout, chunk_sizes=sizes, window=window, workspace=ws32,
                                out_dtype=torch.float32)
    o16, l16 = slope.cp_prefill(q, k, v, n, layout, chunk_sizes=sizes, window=window, workspace=ws16,
                                out_dtype=torch.float32, bf16_partials=True)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    p32, lp32 = _workspace_planes(ws32, S, Hq, dv, n_planes, torch.float32)
    p16, lp16 = _workspace_planes(ws16, S, Hq, dv, n_planes, torch.bfloat16)
    # same lse planes bit for bit, including the rows and planes neither run wrote
    assert torch.equal(lp16.view(torch.int32), lp32.view(torch.int32))
    written = torch.isfinite(lp32)  # rows of live planes that see a key (their out elements are written)
    assert written.any()
    assert torch.equal(p16[written].view(torch.int16), p32[written].to(torch.bfloat16).view(torch.int16))
    assert torch.equal(l16, l32)
    # a partial element is a convex combination of v (up to the bf16 rounding of P): |x| <= 1.01 max|v|
    bound = 2.0 ** -8 * 1.01 * v.float().abs().max().item() + 1e-5
    assert (o16 - o32).abs().max().item() <= bound
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    compare(o16.cpu(), l16.cpu(), ro, rl, f"bf16 partials {layout} n={n} W={window}")


def test_full_causal_gqa_s32k_zigzag8_bf16_partials():
    check_full_workload(wl.WORKLOADS[1], 0, rows_random=2048, bf16_partials=True)


# ---------------------------------------------------------------- Ulysses head-sharded layout

@pytest.mark.parametrize("S,Hq,Hkv,dqk,dv,U,window", [
    (2048, 8, 4, 64, 64, 4, 0), (2048, 8, 4, 64, 64, 2, 100), (1000, 8, 2, 128, 128, 2, 0),
    (1536, 4, 4, 192, 128, 4, 0), (777, 6, 3, 64, 64, 3, 37), (2048, 8, 4, 64, 64, 1, 0)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_cp_prefill_ulysses_matches_oracle_and_fused(S, Hq, Hkv, dqk, dv, U, window, out_dtype):
    """Each Ulysses rank computes the whole attention of its head group: the result matches the
    oracle and is bit-identical to the single launch over all heads (the same tiles, listed per
    head group)."""
    q, k, v = qkv(S, Hq, Hkv, dqk, dv, seed=61 + U + dqk, scale_v=0.7)
    out, lse = slope.cp_prefill(q, k, v, U, "ulysses", window=window, out_dtype=out_dtype)
    ref_o = torch.empty_like(out)
    ref_l = torch.empty_like(lse)
    slope.attn_partial(q, k, v, causal=True, window=window, out=ref_o, lse=ref_l)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    compare(out.float().cpu(), lse.cpu(), ro, rl, f"ulysses U={U} W={window} {out_dtype}")


def test_cp_prefill_ulysses_strided_out_and_no_lse():
    """A padded fp32 out (the row/head strides of a wider buffer; the padding stays untouched) and
    no lse (the kernel writes the workspace's lse plane instead)."""
    S, Hq, Hkv, d, U = 1024, 8, 4, 64, 4
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=71)
    big = torch.full((S, Hq, d + 4), 7.0, dtype=torch.float32, device="cuda")
    out = big[:, :, :d]
    ws = torch.empty((slope.cp_prefill_workspace_size(S, Hq, d, U, "ulysses"),), dtype=torch.uint8, device="cuda")
    o, l = slope.cp_prefill(q, k, v, U, "ulysses", out=out, workspace=ws, want_lse=False)
    torch.cuda.synchronize()
    assert l is None and o.data_ptr() == big.data_ptr()
    assert torch.all(big[:, :, d:] == 7.0)  # the padding is untouched
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    lse_ws = ws[:S * Hq * 4].view(torch.float32).view(S, Hq).T.cpu()  # [S, Hq] plane, head fastest
    compare(out.cpu(), lse_ws, ro, rl, "ulysses strided out, lse in the workspace")


def test_full_causal_gqa_s32k_ulysses8():
    """The 32K GQA workload (8 KV heads) as 8 Ulysses ranks, sampled rows of one KV group."""
    w = wl.WORKLOADS[1]
    q, k, v = wl.workload_qkv(w, device="cuda")
    out, lse = slope.cp_prefill(q, k, v, 8, "ulysses")
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    rows = wl.sample_rows(w, n_random=2048)
    heads = wl.sample_heads(w)
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, rows=rows, heads=heads)
    og = out[torch.from_numpy(rows).cuda()][:, heads].float().cpu()
    lg = lse[heads][:, torch.from_numpy(rows).cuda()].cpu()
    compare(og, lg, ro, rl, "s32k ulysses8")


def test_head_grouped_tile_order_with_one_query_head_per_kv_head():
    """With Hq / Hkv < 4 and dqk >= 128 the launch orders its tiles head group by head group (here 8 heads
    per group over 32 row blocks for the single launch and for 4 Ulysses ranks, 1 per group for 32 ranks):
    every (row block, head) is computed once, by the same arithmetic, whatever the grouping."""
    S, H, d = 8192, 32, 128
    q, k, v = qkv(S, H, H, d, d, seed=83, scale_v=0.6)
    fo = torch.empty((S, H, d), dtype=torch.bfloat16, device="cuda")
    fl = torch.empty((H, S), dtype=torch.float32, device="cuda")
    slope.attn_partial(q, k, v, causal=True, out=fo, lse=fl)
    res = [slope.cp_prefill(q, k, v, U, "ulysses") for U in (32, 4)]
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    for o, l in res:
        assert torch.equal(o, fo) and torch.equal(l, fl)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(S - 128, S), rng.integers(0, S, 384)]))
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, rows=rows)
    rt = torch.from_numpy(rows).cuda()
    compare(fo[rt].float().cpu(), fl[:, rt].cpu(), ro, rl, "head-grouped tile order")


@pytest.mark.parametrize("layout,n,u,window,sizes,dims", [
    ("zigzag", 4, 2, 0, None, (8, 4, 64, 64)), ("zigzag", 8, 4, 100, None, (8, 4, 64, 64)),
    ("contiguous", 4, 4, 0, None, (8, 4, 64, 64)), ("chunked", 3, 2, 0, [700, 1, 1347], (8, 4, 64, 64)),
    ("chunked", 2, 2, 0, [1000, 1048], (4, 4, 192, 128))])
def test_cp_prefill_ulysses_ring_equals_the_ring(layout, n, u, window, sizes, dims):
    """Ulysses x Ring (the layout word's degree u): each step's partial is computed as u head-group
    items writing the same planes, so the result is bit-identical to the plain ring (or chunks) and
    matches the oracle."""
    S = 2048
    Hq, Hkv, dqk, dv = dims
    q, k, v = qkv(S, Hq, Hkv, dqk, dv, seed=91 + u + n, scale_v=0.7)
    bo, bl = slope.cp_prefill(q, k, v, n, layout, chunk_sizes=sizes, window=window, out_dtype=torch.float32)
    o, l = slope.cp_prefill(q, k, v, n, slope.layout_code(layout, u), chunk_sizes=sizes, window=window,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    assert torch.equal(o, bo) and torch.equal(l, bl)
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    compare(o.cpu(), l.cpu(), ro, rl, f"ulysses x ring {layout} n={n} u={u} W={window}")


# ---------------------------------------------------------------- fused layouts (slope_cp_prefill_ex, SLOPE_CP_FUSED)

@pytest.mark.parametrize("layout,n,u,window,sizes,dims", [
    ("zigzag", 4, 1, 0, None, (8, 4, 64, 64)), ("zigzag", 8, 1, 100, None, (8, 4, 64, 64)),
    ("contiguous", 4, 1, 0, None, (8, 4, 64, 64)), ("zigzag", 2, 2, 0, None, (8, 4, 128, 128)),
    ("chunked", 3, 1, 0, [700, 1, 1347], (8, 4, 64, 64)), ("chunked", 2, 1, 300, [1000, 1048], (4, 4, 192, 128)),
    ("chunked", 4, 2, 0, [300, 700, 548, 500], (4, 2, 64, 128)), ("zigzag", 16, 1, 0, None, (4, 1, 192, 64))])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_cp_prefill_fused_matches_oracle(layout, n, u, window, sizes, dims, out_dtype):
    """SLOPE_CP_FUSED: each rank's (or chunk's) query rows over all their visible keys in one item, written
    directly.  It matches the oracle and the partials-and-merge result; without a window every item's key
    range starts at key 0, like the single launch over the whole sequence, and the result is bit-identical
    to that launch."""
    S = 2048
    Hq, Hkv, dqk, dv = dims
    q, k, v = qkv(S, Hq, Hkv, dqk, dv, seed=131 + n + dqk + u, scale_v=0.7)
    lay = slope.layout_code(layout, u)
    o, l = slope.cp_prefill(q, k, v, n, lay, chunk_sizes=sizes, window=window, out_dtype=out_dtype, fused=True)
    mo, ml = slope.cp_prefill(q, k, v, n, lay, chunk_sizes=sizes, window=window, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    compare(o.float().cpu(), l.cpu(), ro, rl, f"fused {layout} n={n} u={u} W={window} {out_dtype}")
    compare(o.float().cpu(), l.cpu(), mo.float().cpu().double().numpy(), ml.cpu().double().numpy(),
            f"fused vs partials+merge {layout} n={n}")
    if window == 0:
        fo = torch.empty_like(o)
        fl = torch.empty_like(l)
        slope.attn_partial(q, k, v, causal=True, out=fo, lse=fl)
        torch.cuda.synchronize()
        assert torch.equal(o, fo) and torch.equal(l, fl)


def test_cp_prefill_fused_without_lse_uses_the_workspace_plane():
    S, Hq, Hkv, d, n = 1024, 4, 2, 64, 4
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=141)
    nbytes = slope.cp_prefill_workspace_size(S, Hq, d, n, "zigzag", fused=True)
    assert nbytes == S * Hq * 4
    ws = torch.empty((nbytes,), dtype=torch.uint8, device="cuda")
    o, l = slope.cp_prefill(q, k, v, n, "zigzag", workspace=ws, want_lse=False, fused=True)
    torch.cuda.synchronize()
    assert l is None
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    lse_ws = ws.view(torch.float32).view(S, Hq).T.cpu()
    compare(o.float().cpu(), lse_ws, ro, rl, "fused, lse in the workspace")


def test_full_causal_gqa_s32k_zigzag8_fused():
    check_full_workload(wl.WORKLOADS[1], 0, rows_random=2048, fused=True)


def test_full_chunked_prefill_s64k_fused():
    check_full_workload(wl.WORKLOADS[2], 0, rows_random=2048, fused=True)


# ---------------------------------------------------------------- dynamic chunk sizes (slope_dck_chunk_sizes)

def test_full_chunked_prefill_s64k_dck():
    """The 64K GQA workload chunked by the dynamic sizes (initial 12288, sigma 0.65): 27 chunks shrinking
    from 12288 to about 1200 tokens, partials and merge, against the oracle on sampled rows."""
    w = wl.WORKLOADS[2]
    sizes = slope.dck_chunk_sizes(w.S, 12288, 0.65)
    assert len(sizes) > 6 and sizes[0] == 12288
    check_full_workload(w, 0, rows_random=2048, sizes=sizes)


def test_full_mla_s64k_dck_fused():
    """The MLA-shaped workload chunked by the dynamic sizes, in the fused form (one item per chunk)."""
    w = wl.WORKLOADS[4]
    check_full_workload(w, 0, rows_random=1024, sizes=slope.dck_chunk_sizes(w.S), fused=True)


def test_full_mla_s64k_dck():
    w = wl.WORKLOADS[4]
    check_full_workload(w, 0, rows_random=1024, sizes=slope.dck_chunk_sizes(w.S))
