"""Checks that pin the fp64 oracle to mathematics it does not itself contain.

Each ``check_*`` function raises ``AssertionError`` when the oracle currently
bound in :mod:`oracle` disagrees with an independent source:

* hand-derived worked examples under ``tests/golden/`` (closed-form values),
* a pure-Python loop brute force on tiny inputs,
* a materialised numpy score matrix with an explicitly built mask,
* torch's CPU ``scaled_dot_product_attention`` / ``logsumexp`` in fp64,
* closed forms (zero keys -> mean of visible values and lse = ln count; a
  single visible key -> that value and its score; constant values),
* merge algebra (identity, permutation, -inf partial, associativity),
* chunk-layout invariance: ring (contiguous / zigzag) and chunked-prefill
  partials merged equal unchunked attention.

They are plain functions so that ``test_oracle_mutants.py`` can run all of
them against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_ENV = {"e": math.e, "log": math.log, "exp": math.exp, "sqrt": math.sqrt, "inf": math.inf}


def _val(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, _ENV))  # expressions of the fixtures only
    return float(x)


def _bf16(a):
    return torch.tensor(a, dtype=torch.float64).to(torch.bfloat16)


def rand_qkv(S, Hq, Hkv, dqk, dv, seed, Skv=None, scale_v=1.0):
    g = torch.Generator().manual_seed(seed)
    Skv = S if Skv is None else Skv
    q = (torch.randn(S, Hq, dqk, generator=g) * scale_v).to(torch.bfloat16)
    k = (torch.randn(Skv, Hkv, dqk, generator=g) * scale_v).to(torch.bfloat16)
    v = (torch.randn(Skv, Hkv, dv, generator=g) * scale_v).to(torch.bfloat16)
    return q, k, v


def _mask(Sq, Skv, q_pos0, kv_pos0, causal, window):
    pq = q_pos0 + np.arange(Sq)[:, None]
    pk = kv_pos0 + np.arange(Skv)[None, :]
    m = np.ones((Sq, Skv), dtype=bool)
    if causal:
        m &= pk <= pq
    if window > 0:
        m &= (pq - pk) < window
    return m


def brute_numpy(q, k, v, q_pos0=0, kv_pos0=0, causal=True, window=0, scale=None):
    """Materialised S x S softmax with an explicit boolean mask (fp64)."""
    Q, K, V = (t.double().numpy() for t in (q, k, v))
    Sq, Hq, dqk = Q.shape
    Skv, Hkv, dv = V.shape
    G = Hq // Hkv
    scale = 1 / math.sqrt(dqk) if scale is None else scale
    mask = _mask(Sq, Skv, q_pos0, kv_pos0, causal, window)
    out = np.zeros((Sq, Hq, dv))
    lse = np.full((Hq, Sq), -np.inf)
    for h in range(Hq):
        Kg, Vg = K[:, h // G, :], V[:, h // G, :]
        s = scale * (Q[:, h, :] @ Kg.T)
        s = np.where(mask, s, -np.inf)
        any_vis = mask.any(axis=1)
        m = np.where(any_vis, s.max(axis=1, initial=-np.inf), 0.0)
        p = np.where(mask, np.exp(s - m[:, None]), 0.0)
        l = p.sum(axis=1)
        safe = np.where(any_vis, l, 1.0)
        out[:, h, :] = np.where(any_vis[:, None], (p @ Vg) / safe[:, None], 0.0)
        lse[h] = np.where(any_vis, m + np.log(safe), -np.inf)
    return out, lse


def brute_python(q, k, v, causal=True, window=0, scale=None):
    """Pure-Python loops, one score at a time (tiny inputs only)."""
    Q, K, V = (t.double().tolist() for t in (q, k, v))
    Sq, Hq, dqk = len(Q), len(Q[0]), len(Q[0][0])
    Skv, Hkv, dv = len(V), len(V[0]), len(V[0][0])
    G = Hq // Hkv
    scale = 1 / math.sqrt(dqk) if scale is None else scale
    out = [[[0.0] * dv for _ in range(Hq)] for _ in range(Sq)]
    lse = [[-math.inf] * Sq for _ in range(Hq)]
    for h in range(Hq):
        g = h // G
        for i in range(Sq):
            vis = [j for j in range(Skv) if (not causal or j <= i) and (window == 0 or i - j < window)]
            if not vis:
                continue
            sc = {j: scale * math.fsum(Q[i][h][d] * K[j][g][d] for d in range(dqk)) for j in vis}
            m = max(sc.values())
            w = {j: math.exp(sc[j] - m) for j in vis}
            l = math.fsum(w.values())
            for e in range(dv):
                out[i][h][e] = math.fsum(w[j] * V[j][g][e] for j in vis) / l
            lse[h][i] = m + math.log(l)
    return np.array(out), np.array(lse)


def close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: -inf pattern differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite values differ"
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin]))
        assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- golden examples

def check_golden_attention():
    for name in ("two_keys_causal.json", "gqa_group_map.json", "window_edge.json"):
        fx = json.load(open(os.path.join(GOLDEN, name)))
        q, k, v = _bf16(fx["q"]), _bf16(fx["k"]), _bf16(fx["v"])
        for case in fx["cases"]:
            out, lse = oracle.attention(q, k, v, causal=bool(case["causal"]), window=case["window"],
                                        scale=fx["scale"])
            exp_out = np.array([[_val(x) for x in row] for row in case["out"]])
            exp_lse = np.array([[_val(x) for x in row] for row in case["lse"]])
            S, Hq, dv = out.shape
            if exp_out.shape == (S, dv):  # one head
                exp_out = exp_out[:, None, :]
            else:  # one row, heads listed
                exp_out = exp_out.reshape(S, Hq, dv)
            exp_lse = exp_lse.reshape(Hq, S)
            close(out, exp_out, 1e-12, f"{name} out {case}")
            close(lse, exp_lse, 1e-12, f"{name} lse {case}")


def check_golden_merge():
    fx = json.load(open(os.path.join(GOLDEN, "merge_two_partials.json")))
    outs = [np.array(p["out"], dtype=np.float64) for p in fx["partials"]]
    lses = [np.array([[_val(x) for x in r] for r in p["lse"]]) for p in fx["partials"]]
    out, lse = oracle.merge(outs, lses)
    exp_out = np.array([[[_val(x) for x in c] for c in r] for r in fx["expected"]["out"]])
    exp_lse = np.array([[_val(x) for x in r] for r in fx["expected"]["lse"]])
    close(out, exp_out, 1e-12, "golden merge out")
    close(lse, exp_lse, 1e-12, "golden merge lse")


# ---------------------------------------------------------------- brute force

def check_brute_python():
    cases = [(7, 2, 1, 3, 2, True, 0), (9, 4, 2, 2, 3, True, 3), (6, 2, 2, 4, 4, False, 0),
             (8, 3, 1, 2, 5, True, 1)]
    for n, (S, Hq, Hkv, dqk, dv, causal, window) in enumerate(cases):
        q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=100 + n)
        o, l = oracle.attention(q, k, v, causal=causal, window=window)
        bo, bl = brute_python(q, k, v, causal=causal, window=window)
        close(o, bo, 1e-12, f"python brute out {n}")
        close(l, bl, 1e-12, f"python brute lse {n}")


def check_brute_numpy():
    cases = [
        # S, Skv, Hq, Hkv, dqk, dv, q_pos0, kv_pos0, causal, window
        (256, 256, 4, 1, 16, 16, 0, 0, True, 0),
        (200, 200, 4, 2, 32, 24, 0, 0, True, 17),
        (96, 160, 4, 4, 24, 40, 300, 200, True, 0),
        (64, 128, 2, 1, 8, 8, 0, 64, True, 0),   # keys entirely in the future: all masked
        (70, 50, 6, 3, 12, 20, 1000, 0, False, 0),
        (120, 120, 4, 1, 16, 8, 0, 0, True, 1),
    ]
    for n, (S, Skv, Hq, Hkv, dqk, dv, qp, kp, causal, window) in enumerate(cases):
        q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=200 + n, Skv=Skv, scale_v=1.5)
        o, l = oracle.attention(q, k, v, q_pos0=qp, kv_pos0=kp, causal=causal, window=window)
        bo, bl = brute_numpy(q, k, v, qp, kp, causal, window)
        close(o, bo, 1e-12, f"numpy brute out {n}")
        close(l, bl, 1e-12, f"numpy brute lse {n}")


def check_torch_sdpa():
    """torch's CPU SDPA (fp64) with an explicit boolean mask and explicit head repeat."""
    cases = [(128, 8, 2, 64, 64, 0), (96, 4, 4, 48, 32, 0), (160, 4, 1, 32, 16, 40)]
    for n, (S, Hq, Hkv, dqk, dv, window) in enumerate(cases):
        q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=300 + n, scale_v=1.2)
        scale = 0.37 + 0.01 * n
        o, l = oracle.attention(q, k, v, causal=True, window=window, scale=scale)
        G = Hq // Hkv
        Q = q.double().permute(1, 0, 2)
        K = k.double().permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = v.double().permute(1, 0, 2).repeat_interleave(G, dim=0)
        mask = torch.from_numpy(_mask(S, S, 0, 0, True, window))
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        scores = torch.where(mask, scale * (Q @ K.transpose(1, 2)), torch.tensor(-math.inf, dtype=torch.float64))
        ref_lse = torch.logsumexp(scores, dim=-1)
        close(o, ref.permute(1, 0, 2).numpy(), 1e-12, f"sdpa out {n}")
        close(l, ref_lse.numpy(), 1e-12, f"sdpa lse {n}")


# ---------------------------------------------------------------- closed forms

def check_closed_forms():
    S, Hq, Hkv, dqk, dv = 150, 4, 2, 16, 12
    q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=400)
    V = v.double().numpy()
    G = Hq // Hkv
    # zero keys: every visible score is 0 -> mean of visible values, lse = ln(count)
    kz = torch.zeros_like(k)
    for window in (0, 5):
        o, l = oracle.attention(q, kz, v, causal=True, window=window)
        for i in range(S):
            lo = 0 if window == 0 else max(0, i - window + 1)
            cnt = i - lo + 1
            for h in range(Hq):
                np.testing.assert_allclose(o[i, h], V[lo:i + 1, h // G].mean(axis=0), rtol=0, atol=1e-12)
                assert abs(l[h, i] - math.log(cnt)) <= 1e-12, "zero-key lse"
    # one visible key (window 1): out = v_i, lse = s_ii
    scale = 0.25
    o, l = oracle.attention(q, k, v, causal=True, window=1, scale=scale)
    Q, K = q.double().numpy(), k.double().numpy()
    for h in range(Hq):
        np.testing.assert_allclose(o[:, h], V[:, h // G], rtol=0, atol=1e-12)
        sii = scale * np.einsum("sd,sd->s", Q[:, h], K[:, h // G])
        np.testing.assert_allclose(l[h], sii, rtol=0, atol=1e-12)
    # causal row 0 sees only key 0
    o, l = oracle.attention(q, k, v, causal=True, scale=scale)
    for h in range(Hq):
        np.testing.assert_allclose(o[0, h], V[0, h // G], rtol=0, atol=1e-12)
    # constant values c: output is c wherever a key is visible
    vc = torch.full_like(v, 0.75)
    o, _ = oracle.attention(q, k, vc, causal=True)
    np.testing.assert_allclose(o, 0.75, rtol=0, atol=1e-12)
    # no visible key: out 0, lse -inf
    o, l = oracle.attention(q[:10], k, v, q_pos0=0, kv_pos0=100, causal=True)
    assert np.all(o == 0.0) and np.all(l == -np.inf), "empty rows"


# ---------------------------------------------------------------- merge algebra

def check_merge_algebra():
    rng = np.random.default_rng(500)
    R, H, dv = 37, 3, 5
    parts = [(rng.normal(size=(R, H, dv)), rng.normal(size=(H, R)) * 3) for _ in range(4)]
    o1, l1 = oracle.merge([parts[0][0]], [parts[0][1]])
    close(o1, parts[0][0], 1e-12, "merge identity out")
    close(l1, parts[0][1], 1e-12, "merge identity lse")
    oa, la = oracle.merge([p[0] for p in parts], [p[1] for p in parts])
    perm = [2, 0, 3, 1]
    ob, lb = oracle.merge([parts[i][0] for i in perm], [parts[i][1] for i in perm])
    close(oa, ob, 1e-12, "merge permutation out")
    close(la, lb, 1e-12, "merge permutation lse")
    dead = (rng.normal(size=(R, H, dv)) * 1e6, np.full((H, R), -np.inf))
    oc, lc = oracle.merge([parts[0][0], dead[0]], [parts[0][1], dead[1]])
    close(oc, parts[0][0], 1e-12, "merge -inf identity out")
    close(lc, parts[0][1], 1e-12, "merge -inf identity lse")
    o01, l01 = oracle.merge([parts[0][0], parts[1][0]], [parts[0][1], parts[1][1]])
    od, ld = oracle.merge([o01, parts[2][0], parts[3][0]], [l01, parts[2][1], parts[3][1]])
    close(od, oa, 1e-12, "merge associativity out")
    close(ld, la, 1e-12, "merge associativity lse")
    # closed form: lse = log sum exp, with a huge offset that a non-shifted sum overflows
    big = [p[1] + 800.0 for p in parts]
    _, lbig = oracle.merge([p[0] for p in parts], big)
    close(lbig, la + 800.0, 1e-9, "merge shift")
    oe, le = oracle.merge([dead[0], dead[0]], [dead[1], dead[1]])
    assert np.all(oe == 0.0) and np.all(le == -np.inf), "merge of empties"


# ---------------------------------------------------------------- invariance

def ring_owned(r, N, layout):
    """Sub-chunks a ring rank holds: zigzag -> {r, 2N-1-r} of 2N; contiguous -> {r} of N."""
    return [r, 2 * N - 1 - r] if layout == "zigzag" else [r]


def ring_reference(q, k, v, N, layout, window=0):
    """Ring decomposition with the oracle: at step t rank r holds the K/V of rank
    (r - t) mod N; every (own Q sub-chunk, held KV sub-chunk) pair gives one partial,
    and a row's partials are merged.  Returns out [S,Hq,dv], lse [Hq,S]."""
    S, Hq, _ = q.shape
    dv = v.shape[2]
    parts = 2 * N if layout == "zigzag" else N
    c = S // parts
    out = np.zeros((S, Hq, dv))
    lse = np.zeros((Hq, S))
    for r in range(N):
        for a in ring_owned(r, N, layout):
            po, pl = [], []
            for t in range(N):
                src = (r - t) % N
                for b in ring_owned(src, N, layout):
                    o, l = oracle.attention(q[a * c:(a + 1) * c], k[b * c:(b + 1) * c], v[b * c:(b + 1) * c],
                                            q_pos0=a * c, kv_pos0=b * c, causal=True, window=window)
                    po.append(o)
                    pl.append(l)
            mo, ml = oracle.merge(po, pl)
            out[a * c:(a + 1) * c] = mo
            lse[:, a * c:(a + 1) * c] = ml
    return out, lse


def chunked_reference(q, k, v, sizes, window=0):
    """Chunked prefill: chunk [s, e) attends to KV[0, s) (prefix partial) and
    causally to KV[s, e) (its own partial); the two partials are merged."""
    S, Hq, _ = q.shape
    dv = v.shape[2]
    out = np.zeros((S, Hq, dv))
    lse = np.zeros((Hq, S))
    s0 = 0
    for c in sizes:
        s1 = s0 + c
        o1, l1 = oracle.attention(q[s0:s1], k[:s0], v[:s0], q_pos0=s0, kv_pos0=0, causal=True, window=window)
        o2, l2 = oracle.attention(q[s0:s1], k[s0:s1], v[s0:s1], q_pos0=s0, kv_pos0=s0, causal=True,
                                  window=window)
        mo, ml = oracle.merge([o1, o2], [l1, l2])
        out[s0:s1] = mo
        lse[:, s0:s1] = ml
        s0 = s1
    return out, lse


def check_invariance():
    S, Hq, Hkv, dqk, dv = 240, 4, 2, 16, 8
    q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=600, scale_v=1.3)
    for window in (0, 23):
        full_o, full_l = oracle.attention(q, k, v, causal=True, window=window)
        for layout in ("contiguous", "zigzag"):
            for N in (1, 2, 3, 4, 8):
                parts = 2 * N if layout == "zigzag" else N
                if S % parts:
                    continue
                o, l = ring_reference(q, k, v, N, layout, window)
                close(o, full_o, 1e-12, f"ring {layout} N={N} W={window} out")
                close(l, full_l, 1e-12, f"ring {layout} N={N} W={window} lse")
        rng = np.random.default_rng(601)
        for trial in range(3):
            sizes, left = [], S
            while left:
                sizes.append(min(left, int(rng.integers(1, 90))))
                left -= sizes[-1]
            o, l = chunked_reference(q, k, v, sizes, window)
            close(o, full_o, 1e-12, f"chunked {sizes} W={window} out")
            close(l, full_l, 1e-12, f"chunked {sizes} W={window} lse")


def check_head_and_row_subsets():
    """The oracle's row/head subsets (used on the large workloads) and the Ulysses split (each rank's
    contiguous query-head group over all tokens, KV heads of that group) equal the matching slices of
    the materialised attention; a subset head keeps its global KV head (h // G, not its index in the
    subset)."""
    S, Hq, Hkv, dqk, dv = 96, 8, 2, 16, 8
    q, k, v = rand_qkv(S, Hq, Hkv, dqk, dv, seed=700, scale_v=1.1)
    for window in (0, 17):
        full_o, full_l = brute_numpy(q, k, v, causal=True, window=window)
        for heads in ([4, 5, 6, 7], [1, 6], [7], [6, 1]):
            for rows in (None, [0, 5, 95, 40]):
                o, l = oracle.attention(q, k, v, causal=True, window=window, heads=heads, rows=rows)
                r = np.arange(S) if rows is None else np.array(rows)
                close(o, full_o[r][:, heads], 1e-12, f"heads {heads} rows {rows} W={window} out")
                close(l, full_l[heads][:, r], 1e-12, f"heads {heads} rows {rows} W={window} lse")
        for U in (1, 2):
            hq, hk = Hq // U, Hkv // U
            outs, lses = [], []
            for u in range(U):
                o, l = oracle.attention(q[:, u * hq:(u + 1) * hq], k[:, u * hk:(u + 1) * hk], v[:, u * hk:(u + 1) * hk],
                                        causal=True, window=window)
                outs.append(o)
                lses.append(l)
            close(np.concatenate(outs, axis=1), full_o, 1e-12, f"Ulysses U={U} W={window} out")
            close(np.concatenate(lses, axis=0), full_l, 1e-12, f"Ulysses U={U} W={window} lse")


ALL_CHECKS = [check_golden_attention, check_golden_merge, check_brute_python, check_brute_numpy,
              check_torch_sdpa, check_closed_forms, check_merge_algebra, check_invariance,
              check_head_and_row_subsets]
