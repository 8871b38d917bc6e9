"""Python binding of libslope: context-parallel causal GQA prefill attention on GB300.

Thin ctypes marshalling over the C ABI declared in ``include/slope.h``; every
step of the computation runs in the library's CUDA kernels.  PyTorch only
provides device memory, streams and events.  There is no fallback: if the
compiled library is missing, every call raises.

The calls mirror the C ABI:

* :func:`attn_partial` - partial attention of a query block against a
  key/value block (one Ring Attention step of one device), returning the
  normalised output and its log-sum-exp.
* :func:`lse_merge` - exact log-sum-exp merge of partials.
* :func:`cp_prefill` - the whole context-parallel prefill attention: ring
  steps (zigzag or contiguous) or chunked prefill, run in order, then merged.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH

__all__ = [
    "SlopeError", "load", "build", "attn_partial", "lse_merge", "cp_prefill", "cp_prefill_timed",
    "cp_prefill_workspace_size", "cp_prefill_plan", "device_status", "timeout_selftest", "LAYOUTS", "version",
    "cp_prefill_static_scratch", "dck_chunk_sizes",
]

LAYOUTS = {"contiguous": 0, "zigzag": 1, "chunked": 2, "ulysses": 3}
_BF16, _F32 = 0, 1


class SlopeTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3), ("stride", ctypes.c_int64 * 3)]


class SlopePlanItem(ctypes.Structure):
    _fields_ = [("launch", ctypes.c_int32), ("plane", ctypes.c_int32), ("q_row0", ctypes.c_int64),
                ("q_len", ctypes.c_int64), ("n_kv", ctypes.c_int32), ("kv_row0", ctypes.c_int64 * 2),
                ("kv_len", ctypes.c_int64 * 2), ("head_group", ctypes.c_int32), ("n_head_groups", ctypes.c_int32)]


class SlopeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status in (-6, -9):
            detail = " [" + load().slope_last_error().decode() + "]"
        super().__init__(f"{what}: {status_string(status)} ({status}){detail}")


_lib = None

EXPORTED = ["slope_attn_partial", "slope_lse_merge", "slope_cp_prefill", "slope_cp_prefill_workspace_size",
            "slope_cp_prefill_timed", "slope_cp_prefill_plan", "slope_device_status",
            "slope_debug_timeout_selftest", "slope_status_string", "slope_version", "slope_last_error",
            "slope_cp_prefill_static_scratch", "slope_cp_prefill_host", "slope_cp_prefill_ex",
            "slope_cp_prefill_workspace_size_ex", "slope_cp_prefill_plan_ex", "slope_dck_chunk_sizes"]

# flags of slope_cp_prefill_ex (include/slope.h)
CP_BF16_PARTIALS = 1
CP_FUSED = 2


def build(force: bool = False) -> str:
    """Compile libslope.so in-tree for sm_103a (nvcc) and return its path."""
    from ._build import build as _b
    return _b(force=force)


def load():
    """Load libslope.so (built by :func:`build`); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libslope.so is not built ({LIB_PATH}); call ring_attention_slope_gb300.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    T = P(SlopeTensor)
    i64, c_int, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    lib.slope_attn_partial.argtypes = [T, T, T, i64, i64, c_int, i64, f32, T, T, vp]
    lib.slope_attn_partial.restype = c_int
    lib.slope_lse_merge.argtypes = [T, T, c_int, T, T, vp]
    lib.slope_lse_merge.restype = c_int
    lib.slope_cp_prefill.argtypes = [T, T, T, c_int, c_int, P(i64), c_int, i64, f32, T, T, vp, ctypes.c_size_t, vp]
    lib.slope_cp_prefill.restype = c_int
    lib.slope_cp_prefill_timed.argtypes = [T, T, T, c_int, c_int, P(i64), c_int, i64, f32, T, T, vp,
                                           ctypes.c_size_t, vp, P(vp), c_int, P(c_int), P(c_int)]
    lib.slope_cp_prefill_timed.restype = c_int
    lib.slope_cp_prefill_workspace_size.argtypes = [i64, i64, i64, c_int, c_int, P(i64)]
    lib.slope_cp_prefill_workspace_size.restype = ctypes.c_size_t
    lib.slope_cp_prefill_plan.argtypes = [i64, c_int, c_int, P(i64), c_int, i64, P(SlopePlanItem), i64,
                                          P(ctypes.c_int32), P(ctypes.c_int32)]
    lib.slope_cp_prefill_plan.restype = i64
    lib.slope_cp_prefill_plan_ex.argtypes = [i64, c_int, c_int, P(i64), c_int, i64, ctypes.c_uint, P(SlopePlanItem),
                                             i64, P(ctypes.c_int32), P(ctypes.c_int32)]
    lib.slope_cp_prefill_plan_ex.restype = i64
    lib.slope_dck_chunk_sizes.argtypes = [i64, i64, ctypes.c_double, i64, i64, P(i64), i64]
    lib.slope_dck_chunk_sizes.restype = i64
    lib.slope_device_status.argtypes = [vp, P(c_int)]
    lib.slope_device_status.restype = c_int
    lib.slope_debug_timeout_selftest.argtypes = [ctypes.c_uint64, vp]
    lib.slope_debug_timeout_selftest.restype = c_int
    lib.slope_status_string.argtypes = [c_int]
    lib.slope_status_string.restype = ctypes.c_char_p
    lib.slope_version.argtypes = []
    lib.slope_version.restype = ctypes.c_char_p
    lib.slope_last_error.argtypes = []
    lib.slope_last_error.restype = ctypes.c_char_p
    lib.slope_cp_prefill_static_scratch.argtypes = [T, T, T, c_int, c_int, P(i64), c_int, i64, f32, T, T, vp]
    lib.slope_cp_prefill_static_scratch.restype = c_int
    lib.slope_cp_prefill_host.argtypes = [T, T, T, T, T, T, T, T, T, T, c_int, c_int, P(i64), c_int, i64, f32, vp,
                                          ctypes.c_size_t, vp, vp, vp]
    lib.slope_cp_prefill_host.restype = c_int
    lib.slope_cp_prefill_ex.argtypes = [T, T, T, c_int, c_int, P(i64), c_int, i64, f32, ctypes.c_uint, T, T, vp,
                                        ctypes.c_size_t, vp]
    lib.slope_cp_prefill_ex.restype = c_int
    lib.slope_cp_prefill_workspace_size_ex.argtypes = [i64, i64, i64, c_int, c_int, P(i64), ctypes.c_uint]
    lib.slope_cp_prefill_workspace_size_ex.restype = ctypes.c_size_t
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().slope_status_string(int(status)).decode()


def version() -> str:
    return load().slope_version().decode()


# ---------------------------------------------------------------- marshalling helpers

def _torch():
    import torch
    return torch


def _desc(t, expect_dtype=None, host=False):
    """slope_tensor describing a CUDA tensor (or, with host=True, a CPU tensor) of rank 2 or 3."""
    torch = _torch()
    if t.dtype == torch.bfloat16:
        dt = _BF16
    elif t.dtype == torch.float32:
        dt = _F32
    else:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if expect_dtype is not None and t.dtype != expect_dtype:
        raise TypeError(f"expected {expect_dtype}, got {t.dtype}")
    if t.numel() > 0 and t.device.type != ("cpu" if host else "cuda"):
        raise TypeError("expected a host (CPU) tensor" if host else "libslope operates on CUDA tensors")
    if t.dim() not in (2, 3):
        raise ValueError("tensors must be rank 2 or 3")
    d = SlopeTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = dt
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream_ptr(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != 0:
        raise SlopeError(status, what)


def _chunk_array(chunk_sizes):
    if chunk_sizes is None:
        return None, None
    arr = (ctypes.c_int64 * len(chunk_sizes))(*[int(c) for c in chunk_sizes])
    return arr, ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64))


def _layout(layout):
    if isinstance(layout, str):
        return LAYOUTS[layout]
    return int(layout)


def layout_code(layout, ulysses=1):
    """Layout word of the C ABI: a base layout (name or code) and, for the ring and chunked layouts,
    a Ulysses degree (SLOPE_ULYSSES_DEGREE: the head groups of a Ulysses x Ring split)."""
    code = _layout(layout)
    return code | (int(ulysses) << 8) if int(ulysses) > 1 else code


# ---------------------------------------------------------------- public calls

def attn_partial(q, k, v, *, q_off=0, kv_off=0, causal=True, window=0, scale=0.0, out=None, lse=None,
                 out_dtype=None, stream=None):
    """Partial attention of q [Sq,Hq,dqk] against k [Skv,Hkv,dqk], v [Skv,Hkv,dv] (bf16, CUDA).

    Returns ``(out, lse)``: out fp32 (default) or bf16 [Sq,Hq,dv], lse fp32 [Hq,Sq] (natural log).
    Over the whole sequence with bf16 out this is the whole attention in one launch.
    """
    torch = _torch()
    Sq, Hq, _ = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((Sq, Hq, dv), dtype=out_dtype or torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((Hq, Sq), dtype=torch.float32, device=q.device)
    dq, dk, dvv, do, dl = _desc(q), _desc(k), _desc(v), _desc(out), _desc(lse)
    st = load().slope_attn_partial(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dvv), int(q_off), int(kv_off),
                                   int(bool(causal)), int(window), float(scale), ctypes.byref(do),
                                   ctypes.byref(dl), _stream_ptr(stream))
    _check(st, "slope_attn_partial")
    return out, lse


def lse_merge(outs, lses, *, out=None, lse=None, out_dtype=None, stream=None):
    """Exact log-sum-exp merge of partials outs[k] fp32 or bf16 [S,H,dv] (one dtype), lses[k] fp32 [H,S]."""
    torch = _torch()
    n = len(outs)
    if n != len(lses) or n == 0:
        raise ValueError("need the same, non-zero number of outs and lses")
    S, H, dv = outs[0].shape
    if out is None:
        out = torch.empty((S, H, dv), dtype=out_dtype or torch.bfloat16, device=outs[0].device)
    if lse is None:
        lse = torch.empty((H, S), dtype=torch.float32, device=outs[0].device)
    od = (SlopeTensor * n)(*[_desc(o) for o in outs])
    ld = (SlopeTensor * n)(*[_desc(x) for x in lses])
    do, dl = _desc(out), _desc(lse)
    st = load().slope_lse_merge(od, ld, n, ctypes.byref(do), ctypes.byref(dl), _stream_ptr(stream))
    _check(st, "slope_lse_merge")
    return out, lse


def _flags(bf16_partials=False, fused=False):
    return (CP_BF16_PARTIALS if bf16_partials else 0) | (CP_FUSED if fused else 0)


def cp_prefill_workspace_size(S, Hq, dv, n_chunks, layout, chunk_sizes=None, bf16_partials=False,
                              fused=False) -> int:
    arr, ptr = _chunk_array(chunk_sizes)
    flags = _flags(bf16_partials, fused)
    if flags:
        return int(load().slope_cp_prefill_workspace_size_ex(int(S), int(Hq), int(dv), int(n_chunks), _layout(layout),
                                                             ptr, flags))
    return int(load().slope_cp_prefill_workspace_size(int(S), int(Hq), int(dv), int(n_chunks), _layout(layout), ptr))


def _prep_cp(q, v, n_chunks, layout, chunk_sizes, out, lse, workspace, out_dtype, want_lse, bf16_partials=False,
             fused=False):
    torch = _torch()
    S, Hq, _ = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((S, Hq, dv), dtype=out_dtype or torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((Hq, S), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = cp_prefill_workspace_size(S, Hq, dv, n_chunks, layout, chunk_sizes, bf16_partials, fused)
        if nbytes == 0:
            raise SlopeError(-5, "slope_cp_prefill_workspace_size")
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=q.device)
    return out, lse, workspace


def cp_prefill(q, k, v, n_chunks, layout="zigzag", *, chunk_sizes=None, causal=True, window=0, scale=0.0,
               out=None, lse=None, workspace=None, out_dtype=None, want_lse=True, stream=None, bf16_partials=False,
               fused=False):
    """Context-parallel prefill attention of one layer (ring steps or chunks run in order, then merged).

    Returns ``(out, lse)``: out bf16 (default) or fp32 [S,Hq,dv], lse fp32 [Hq,S] (None if not wanted).
    ``bf16_partials`` keeps the partial outputs in bf16 between the attention launches and the merge
    (SLOPE_CP_BF16_PARTIALS); ``fused`` merges each rank's or chunk's partials online in the kernel, with no
    partial planes and no merge launch (SLOPE_CP_FUSED).  Either runs slope_cp_prefill_ex; otherwise
    slope_cp_prefill runs.
    """
    out, lse, workspace = _prep_cp(q, v, n_chunks, layout, chunk_sizes, out, lse, workspace, out_dtype, want_lse,
                                   bf16_partials, fused)
    arr, ptr = _chunk_array(chunk_sizes)
    dq, dk, dvv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    dl = _desc(lse) if lse is not None else None
    args_head = (ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dvv), int(n_chunks), _layout(layout), ptr,
                 int(bool(causal)), int(window), float(scale))
    args_tail = (ctypes.byref(do), ctypes.byref(dl) if dl is not None else None,
                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    flags = _flags(bf16_partials, fused)
    if flags:
        st = load().slope_cp_prefill_ex(*args_head, flags, *args_tail)
        _check(st, "slope_cp_prefill_ex")
    else:
        st = load().slope_cp_prefill(*args_head, *args_tail)
        _check(st, "slope_cp_prefill")
    return out, lse


def cp_prefill_host(q_host, k_host, v_host, out_host, lse_host, q, k, v, out, lse, n_chunks, layout="zigzag", *,
                    chunk_sizes=None, causal=True, window=0, scale=0.0, workspace=None, copy_in_stream=None,
                    compute_stream=None, copy_out_stream=None):
    """cp_prefill on host tensors: queues host->device copies of q/k/v into the device buffers q/k/v on
    ``copy_in_stream``, the prefill on ``compute_stream`` and device->host copies of out/lse into
    out_host/lse_host on ``copy_out_stream`` (streams default to the current stream).  All tensors are dense;
    host tensors should be pinned.  Returns immediately; the host outputs are valid once
    ``copy_out_stream`` has reached this point.  Calls on different device buffers overlap (see
    slope_cp_prefill_host in include/slope.h)."""
    if workspace is None:
        S, Hq, _ = q.shape
        nbytes = cp_prefill_workspace_size(S, Hq, v.shape[2], n_chunks, layout, chunk_sizes)
        if nbytes == 0:
            raise SlopeError(-5, "slope_cp_prefill_workspace_size")
        workspace = _torch().empty((nbytes,), dtype=_torch().uint8, device=q.device)
    arr, ptr = _chunk_array(chunk_sizes)
    hq, hk, hv, ho = (_desc(t, host=True) for t in (q_host, k_host, v_host, out_host))
    hl = _desc(lse_host, host=True) if lse_host is not None else None
    dq, dk, dvv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    dl = _desc(lse) if lse is not None else None
    ref = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    st = load().slope_cp_prefill_host(ref(hq), ref(hk), ref(hv), ref(ho), ref(hl), ref(dq), ref(dk), ref(dvv),
                                      ref(do), ref(dl), int(n_chunks), _layout(layout), ptr, int(bool(causal)),
                                      int(window), float(scale), ctypes.c_void_p(workspace.data_ptr()),
                                      workspace.numel(), _stream_ptr(copy_in_stream), _stream_ptr(compute_stream),
                                      _stream_ptr(copy_out_stream))
    _check(st, "slope_cp_prefill_host")
    return workspace


def cp_prefill_static_scratch(q, k, v, n_chunks, layout="zigzag", *, chunk_sizes=None, causal=True, window=0,
                              scale=0.0, out=None, lse=None, out_dtype=None, want_lse=True, stream=None):
    """cp_prefill for callers that cannot allocate device memory.

    The partials live in the library's fixed 64 MiB scratch array instead of a
    caller workspace; larger requests raise SlopeError (SLOPE_ERR_WORKSPACE).
    Calls that overlap on the GPU share that array and race.  Returns ``(out, lse)``.
    """
    torch = _torch()
    S, Hq, _ = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((S, Hq, dv), dtype=out_dtype or torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((Hq, S), dtype=torch.float32, device=q.device)
    arr, ptr = _chunk_array(chunk_sizes)
    dq, dk, dvv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    dl = _desc(lse) if lse is not None else None
    st = load().slope_cp_prefill_static_scratch(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dvv),
                                                int(n_chunks), _layout(layout), ptr, int(bool(causal)),
                                                int(window), float(scale), ctypes.byref(do),
                                                ctypes.byref(dl) if dl is not None else None, _stream_ptr(stream))
    _check(st, "slope_cp_prefill_static_scratch")
    return out, lse


def cp_prefill_timed(q, k, v, n_chunks, layout, events, *, chunk_sizes=None, causal=True, window=0, scale=0.0,
                     out=None, lse=None, workspace=None, out_dtype=None, want_lse=True, stream=None):
    """cp_prefill that records ``events`` (list of (start, end) torch.cuda.Event pairs) around each launch.

    Returns ``(out, lse, n_launches, kinds)`` with kinds[i] = 0 (attention) or 1 (merge).
    """
    out, lse, workspace = _prep_cp(q, v, n_chunks, layout, chunk_sizes, out, lse, workspace, out_dtype, want_lse)
    arr, ptr = _chunk_array(chunk_sizes)
    handles = []
    for a, b in events:
        for e in (a, b):
            if e.cuda_event == 0:  # torch creates the CUDA event lazily, at its first record
                e.record()
        handles += [a.cuda_event, b.cuda_event]
    ev = (ctypes.c_void_p * len(handles))(*handles)
    kinds = (ctypes.c_int * len(events))()
    nl = ctypes.c_int(0)
    dq, dk, dvv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    dl = _desc(lse) if lse is not None else None
    st = load().slope_cp_prefill_timed(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dvv), int(n_chunks),
                                       _layout(layout), ptr, int(bool(causal)), int(window), float(scale),
                                       ctypes.byref(do), ctypes.byref(dl) if dl is not None else None,
                                       ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                       _stream_ptr(stream), ev, len(events), ctypes.byref(nl), kinds)
    _check(st, "slope_cp_prefill_timed")
    return out, lse, nl.value, list(kinds)[:nl.value]


def cp_prefill_plan(S, n_chunks, layout, *, chunk_sizes=None, causal=True, window=0, fused=False):
    """Host-only work decomposition: (items, n_launches, n_planes); items are dicts.  ``fused`` gives the
    decomposition of SLOPE_CP_FUSED."""
    lib = load()
    arr, ptr = _chunk_array(chunk_sizes)
    nl, npl = ctypes.c_int32(0), ctypes.c_int32(0)
    flags = _flags(fused=fused)
    n = lib.slope_cp_prefill_plan_ex(int(S), int(n_chunks), _layout(layout), ptr, int(bool(causal)), int(window),
                                     flags, None, 0, ctypes.byref(nl), ctypes.byref(npl))
    if n < 0:
        raise SlopeError(int(n), "slope_cp_prefill_plan")
    items = (SlopePlanItem * max(1, n))()
    n2 = lib.slope_cp_prefill_plan_ex(int(S), int(n_chunks), _layout(layout), ptr, int(bool(causal)), int(window),
                                      flags, items, n, None, None)
    assert n2 == n
    res = []
    for it in items[:n]:
        res.append({"launch": it.launch, "plane": it.plane, "q_row0": it.q_row0, "q_len": it.q_len,
                    "kv": [(it.kv_row0[r], it.kv_len[r]) for r in range(it.n_kv)],
                    "head_group": it.head_group, "n_head_groups": it.n_head_groups})
    return res, nl.value, npl.value


def dck_chunk_sizes(S, initial=12288, sigma=0.65, *, window=0, align=1):
    """Dynamic chunk sizes for the chunked layout (slope_dck_chunk_sizes): from an initial chunk, later
    chunks move towards the size whose attention cost equals the first chunk's, smoothed with factor sigma.
    Returns a list of ints summing to S."""
    lib = load()
    n = lib.slope_dck_chunk_sizes(int(S), int(initial), float(sigma), int(window), int(align), None, 0)
    if n < 0:
        raise SlopeError(int(n), "slope_dck_chunk_sizes")
    arr = (ctypes.c_int64 * n)()
    n2 = lib.slope_dck_chunk_sizes(int(S), int(initial), float(sigma), int(window), int(align),
                                   ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)), n)
    assert n2 == n
    return [int(x) for x in arr]


def device_status(stream=None):
    """(status, site): synchronises the stream, reads and clears the device status word."""
    site = ctypes.c_int(0)
    st = load().slope_device_status(_stream_ptr(stream), ctypes.byref(site))
    return st, site.value


def timeout_selftest(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test kernel (its wait is meant to run out)."""
    _check(load().slope_debug_timeout_selftest(int(limit_ns), _stream_ptr(stream)), "slope_debug_timeout_selftest")
