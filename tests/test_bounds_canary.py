"""Guard regions in place of a device memory checker.

Every buffer the library writes (out, lse, the prefill workspace) is a view inside a larger buffer
whose other bytes hold a canary pattern; after each call the pattern must be intact, and the view
itself must hold the oracle's values.  Sizes are odd (S = 1, 127, 129, ...), positions unaligned,
and the views padded between rows and heads where the ABI allows strides.  The environment variable
SLOPE_DEBUG_BOUNDS=1 widens the sweep.
"""
import itertools
import math
import os

import pytest
import torch

import oracle
import ring_attention_slope_gb300 as slope

pytestmark = pytest.mark.gpu

WIDE = os.environ.get("SLOPE_DEBUG_BOUNDS", "0") not in ("", "0")
CANARY32 = 0x7FC0DEAD  # a NaN payload no kernel writes
CANARY16 = 0x7FAD
CANARY8 = 0xA5
FRONT = 64  # elements (256 bytes for fp32, 128 for bf16): keeps the views 16-byte aligned


@pytest.fixture(scope="module", autouse=True)
def _built():
    slope.build()
    slope.load()


def guarded(shape, dtype, pad_last=0):
    """A view of `shape` (with `pad_last` spare elements after each innermost row) inside a buffer of
    canaries; returns (view, raw buffer as integers, mask of the bytes the view covers)."""
    itype, canary = (torch.int32, CANARY32) if dtype == torch.float32 else (torch.int16, CANARY16)
    inner = shape[-1] + pad_last
    outer = math.prod(shape[:-1])
    n = outer * inner
    raw = torch.full((FRONT + n + FRONT + 37,), canary, dtype=itype, device="cuda")
    covered = torch.zeros_like(raw, dtype=torch.bool)
    body = raw[FRONT:FRONT + n].view(*shape[:-1], inner)
    covered[FRONT:FRONT + n].view(*shape[:-1], inner)[..., :shape[-1]] = True
    view = body[..., :shape[-1]].view(dtype)
    return view, raw, covered, canary


def assert_intact(raw, covered, canary, what):
    outside = raw[~covered]
    bad = int((outside != canary).sum())
    assert bad == 0, f"{what}: {bad} guard elements overwritten"


def qkv(S, Hq, Hkv, dqk, dv, seed, Skv=None):
    g = torch.Generator().manual_seed(seed)
    Skv = S if Skv is None else Skv
    q = torch.randn(S, Hq, dqk, generator=g).to(torch.bfloat16)
    k = torch.randn(Skv, Hkv, dqk, generator=g).to(torch.bfloat16)
    v = torch.randn(Skv, Hkv, dv, generator=g).to(torch.bfloat16)
    return q.cuda(), k.cuda(), v.cuda()


def close(got, ref, what, atol=2e-2):
    got = got.double().cpu()
    ref = torch.as_tensor(ref)
    fin = torch.isfinite(ref)
    assert torch.equal(torch.isneginf(got), torch.isneginf(ref)), f"{what}: -inf pattern differs"
    assert float((got[fin] - ref[fin]).abs().max()) <= atol if fin.any() else True, f"{what}: values"


SIZES = [1, 127, 129, 300] + ([2, 255, 257, 1000] if WIDE else [])
DIMS = [(64, 64), (192, 128)] + ([(128, 64), (64, 128), (192, 64)] if WIDE else [])


@pytest.mark.parametrize("S", SIZES)
@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attn_partial_writes_only_its_outputs(S, dims, out_dtype):
    dqk, dv = dims
    Hq, Hkv = (4, 2) if dqk == 64 else (3, 3)
    q_off, kv_off, window = 5, 3, (77 if S > 100 else 0)
    q, k, v = qkv(S, Hq, Hkv, dqk, dv, seed=S * 7 + dqk, Skv=S + 3)
    out, oraw, ocov, oc = guarded((S, Hq, dv), out_dtype, pad_last=8)  # a gap after every head's row
    lse, lraw, lcov, lc = guarded((Hq, S), torch.float32, pad_last=3)
    slope.attn_partial(q, k, v, q_off=q_off, kv_off=kv_off, causal=True, window=window, out=out, lse=lse)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    assert_intact(oraw, ocov, oc, f"out S={S} {dims}")
    assert_intact(lraw, lcov, lc, f"lse S={S} {dims}")
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), q_pos0=q_off, kv_pos0=kv_off, causal=True, window=window)
    close(lse, rl, "lse", atol=1e-3)
    close(out.float(), ro, "out")


@pytest.mark.parametrize("S", SIZES)
@pytest.mark.parametrize("n", [1, 3, 8])
def test_lse_merge_writes_only_its_outputs(S, n):
    H, dv = 3, 64
    g = torch.Generator().manual_seed(S + n)
    outs = [torch.randn(S, H, dv, generator=g).cuda() for _ in range(n)]
    lses = [(torch.randn(H, S, generator=g) * 3).cuda() for _ in range(n)]
    lses[0][:, 0] = -math.inf
    out, oraw, ocov, oc = guarded((S, H, dv), torch.bfloat16, pad_last=8)
    lse, lraw, lcov, lc = guarded((H, S), torch.float32, pad_last=1)
    slope.lse_merge(outs, lses, out=out, lse=lse)
    torch.cuda.synchronize()
    assert_intact(oraw, ocov, oc, "merge out")
    assert_intact(lraw, lcov, lc, "merge lse")
    ro, rl = oracle.merge([o.double().cpu().numpy() for o in outs], [x.double().cpu().numpy() for x in lses])
    close(lse, rl, "merge lse", atol=1e-3)
    close(out.float(), ro, "merge out")


PREFILL = [("zigzag", 4, 0), ("contiguous", 3, 0), ("chunked", 3, 0), ("zigzag", 2, 77)]
if WIDE:
    PREFILL += [("zigzag", 8, 0), ("chunked", 5, 128), ("contiguous", 1, 0)]


@pytest.mark.parametrize("S", [129, 300] + ([257, 1000] if WIDE else []))
@pytest.mark.parametrize("layout,n,window", PREFILL)
@pytest.mark.parametrize("flags", [(False, False), (True, False), (False, True)], ids=["fp32", "bf16p", "fused"])
def test_cp_prefill_writes_only_out_lse_and_its_workspace(S, layout, n, window, flags):
    bf16_partials, fused = flags
    if layout == "zigzag" and S % (2 * n):
        S += 2 * n - S % (2 * n)
    if layout == "contiguous" and S % n:
        S += n - S % n
    Hq, Hkv, d = 4, 2, 64
    q, k, v = qkv(S, Hq, Hkv, d, d, seed=S + n + window)
    sizes = None
    if layout == "chunked":
        base = S // n
        sizes = [base] * (n - 1) + [S - base * (n - 1)]
    nbytes = slope.cp_prefill_workspace_size(S, Hq, d, n, layout, sizes, bf16_partials=bf16_partials, fused=fused)
    wraw = torch.full((256 + nbytes + 4096,), CANARY8, dtype=torch.uint8, device="cuda")
    ws = wraw[256:256 + nbytes]
    out, oraw, ocov, oc = guarded((S, Hq, d), torch.bfloat16, pad_last=8)
    lse, lraw, lcov, lc = guarded((Hq, S), torch.float32, pad_last=5)
    slope.cp_prefill(q, k, v, n, layout, chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=ws,
                     bf16_partials=bf16_partials, fused=fused)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    assert int((wraw[:256] != CANARY8).sum()) == 0 and int((wraw[256 + nbytes:] != CANARY8).sum()) == 0, \
        "writes outside the workspace"
    assert_intact(oraw, ocov, oc, "prefill out")
    assert_intact(lraw, lcov, lc, "prefill lse")
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True, window=window)
    close(lse, rl, "prefill lse", atol=1e-3)
    close(out.float(), ro, "prefill out")


def test_sweep_flag_is_read():
    """The wide sweep is selected by the environment, as the module docstring says."""
    assert (len(SIZES) > 4) == WIDE and list(itertools.islice(SIZES, 4)) == [1, 127, 129, 300]
