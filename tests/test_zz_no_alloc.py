"""slope_cp_prefill_static_scratch against slope_cp_prefill.

Some callers of this library cannot allocate device memory: a process that
reserved its whole device memory up front for its own pools, or a latency
critical path where an allocation would synchronise the device.  For them the
library offers a variant of slope_cp_prefill that keeps its partials in a fixed
64 MiB array it holds itself.  These tests call it through the C ABI and check
that it gives the results of the workspace entry point, on two calls in a row
with different shapes (the array is shared and keeps the previous call's
contents), and that a request too large for the array is refused.

The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import ring_attention_slope_gb300 as slope
import slope_workloads as wl

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_REL_L2, LSE_MAX = 2e-2, 5e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    slope.build()
    slope.load()


def _close(out, lse, ref_out, ref_lse, what):
    o, r = out.float().cpu().double().numpy(), ref_out.float().cpu().double().numpy()
    lo, lr = lse.cpu().double().numpy(), ref_lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(lo), np.isneginf(lr)), what
    fin = np.isfinite(lr)
    assert np.max(np.abs(lo[fin] - lr[fin])) <= LSE_MAX, what
    assert np.max(np.abs(o - r)) <= OUT_MAX, what
    assert np.linalg.norm(o - r) <= OUT_REL_L2 * np.linalg.norm(r), what


def test_static_scratch_matches_workspace_call_twice():
    # call 1: S=1024, 4 query heads on 1 KV head, zigzag ring of 4 ranks
    w = wl.WORKLOADS[0]
    q, k, v = wl.workload_qkv(w, device="cuda")
    ref_o, ref_l = slope.cp_prefill(q, k, v, 4, "zigzag")
    o1, l1 = slope.cp_prefill_static_scratch(q, k, v, 4, "zigzag")
    # call 2: other inputs and layout (ragged chunked prefill, 2 KV heads, fp32 out)
    g = torch.Generator().manual_seed(77)
    S, Hq, Hkv, d = 1000, 4, 2, 64
    q2 = (torch.randn(S, Hq, d, generator=g) * 0.7).to(torch.bfloat16).cuda()
    k2 = (torch.randn(S, Hkv, d, generator=g) * 0.7).to(torch.bfloat16).cuda()
    v2 = (torch.randn(S, Hkv, d, generator=g) * 0.7).to(torch.bfloat16).cuda()
    sizes = [300, 257, 443]
    ref_o2, ref_l2 = slope.cp_prefill(q2, k2, v2, 3, "chunked", chunk_sizes=sizes, out_dtype=torch.float32)
    o2, l2 = slope.cp_prefill_static_scratch(q2, k2, v2, 3, "chunked", chunk_sizes=sizes, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert slope.device_status() == (0, 0)
    _close(o1, l1, ref_o, ref_l, "first call")
    _close(o2, l2, ref_o2, ref_l2, "second call")


def test_static_scratch_refuses_requests_larger_than_the_array():
    # S = 32768, 64 heads, ring of 8: the partials need about 4.4 GB
    base_q = torch.zeros(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    q = base_q.expand(32768, 64, 64)
    kv = base_q.expand(32768, 8, 64)
    with pytest.raises(slope.SlopeError) as e:
        slope.cp_prefill_static_scratch(q, kv, kv, 8, "zigzag", out=torch.empty(1, 1, 64, device="cuda").expand(
            32768, 64, 64), want_lse=False)
    assert e.value.status == -9
    assert "64" in str(e.value) or "67108864" in str(e.value)
