"""fp64 CPU oracle for context-parallel causal GQA prefill attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package
``ring_attention_slope_gb300``.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C99, fp64, OpenMP over
(head, row)); this module only builds that file with gcc and marshals arrays.

What it computes (Moreh, "Optimizing long-context prefill on multiple
older-generation GPU nodes", section "Introduction to Context Parallelism",
Ring Attention item: attention on each device from partial Q/K/V, combined
across the ring):

* :func:`attention` - softmax attention of a query block against a key/value
  block under a causal and optional sliding-window mask on *global*
  positions, grouped-query heads ``g = h // (Hq // Hkv)``; returns the
  normalised output and the natural-log log-sum-exp of the scaled scores
  (``-inf`` and a zero output for a row that sees no key).  Called on the
  whole sequence it is plain causal attention; called on a sub-block it is
  one ring partial.
* :func:`merge` - the exact log-sum-exp combination of partials computed
  over disjoint key sets.

Pins (tests under ``-m "not gpu"``): brute force on tiny inputs (pure-Python
loops and a materialised numpy score matrix), torch's CPU scaled-dot-product
attention in fp64 with an explicit mask, closed forms (zero keys, a single
visible key, constant values), merge algebra, chunk-layout invariance, and
row/head subsets (with the Ulysses head split) against the full materialised
attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    lib.oracle_attention.restype = _int
    lib.oracle_attention.argtypes = [
        _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
        _i64, _i64, _int, _int, _int, _int,
        _i64, _i64, _int, _i64, _dbl,
        _vp, _i64, _vp, _int, _vp, _vp]
    lib.oracle_merge.restype = _int
    lib.oracle_merge.argtypes = [_vp, _vp, _int, _i64, _int, _int, _vp, _vp]
    lib.oracle_num_threads.restype = _int
    lib.oracle_num_threads.argtypes = []
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's parallel regions use on this host."""
    return int(_load().oracle_num_threads())


def _bf16_bits(x):
    """Return (uint16 ndarray or tensor keeping memory alive, ptr, strides in elements).

    Accepts a torch bf16 tensor of rank 3 (any strides, CPU) or a numpy
    uint16 array holding bf16 bit patterns.
    """
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.dtype != torch.bfloat16 or x.dim() != 3:
            raise TypeError("oracle expects a rank-3 bfloat16 tensor")
        if x.device.type != "cpu":
            x = x.cpu()
        if x.stride(2) != 1:
            x = x.contiguous()
        bits = x.view(torch.int16)
        return bits, bits.data_ptr(), (bits.stride(0), bits.stride(1)), tuple(x.shape)
    a = np.asarray(x)
    if a.dtype != np.uint16 or a.ndim != 3:
        raise TypeError("oracle expects a rank-3 uint16 array of bf16 bits")
    if a.strides[2] != 2:
        a = np.ascontiguousarray(a)
    return a, a.ctypes.data, (a.strides[0] // 2, a.strides[1] // 2), a.shape


def attention(q, k, v, *, q_pos0: int = 0, kv_pos0: int = 0, causal: bool = True,
              window: int = 0, scale: float | None = None, rows=None, heads=None):
    """Softmax attention of q[Sq,Hq,dqk] against k[Skv,Hkv,dqk], v[Skv,Hkv,dv] in fp64.

    ``rows``/``heads`` select a subset of query rows / query heads (default all).
    Returns ``(out, lse)``: out float64 [n_rows, n_heads, dv], lse float64
    [n_heads, n_rows] (natural log; ``-inf`` for a row with no visible key).
    ``scale`` defaults to ``1/sqrt(dqk)``.
    """
    qa, qp, (qsr, qsh), (Sq, Hq, dqk) = _bf16_bits(q)
    ka, kp, (ksr, ksh), (Skv, Hkv, dk2) = _bf16_bits(k)
    va, vp, (vsr, vsh), (Sv, Hv, dv) = _bf16_bits(v)
    if dk2 != dqk or Sv != Skv or Hv != Hkv or Hq % Hkv:
        raise ValueError("inconsistent q/k/v shapes")
    if scale is None:
        scale = 1.0 / float(np.sqrt(dqk))
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    heads_a = None if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
    n_rows = Sq if rows_a is None else len(rows_a)
    n_heads = Hq if heads_a is None else len(heads_a)
    out = np.empty((n_rows, n_heads, dv), dtype=np.float64)
    lse = np.empty((n_heads, n_rows), dtype=np.float64)
    rc = _load().oracle_attention(
        qp, qsr, qsh, kp, ksr, ksh, vp, vsr, vsh,
        Sq, Skv, Hq, Hkv, dqk, dv, int(q_pos0), int(kv_pos0), int(bool(causal)), int(window),
        float(scale),
        None if rows_a is None else rows_a.ctypes.data, n_rows,
        None if heads_a is None else heads_a.ctypes.data, n_heads,
        out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    del qa, ka, va
    return out, lse


def merge(outs, lses):
    """Exact log-sum-exp merge.  outs: list of [R,H,dv], lses: list of [H,R] (fp64)."""
    if len(outs) != len(lses):
        raise ValueError("outs and lses differ in length")
    o64 = [np.ascontiguousarray(o, dtype=np.float64) for o in outs]
    l64 = [np.ascontiguousarray(x, dtype=np.float64) for x in lses]
    if not o64:
        raise ValueError("merge of zero partials")
    R, H, dv = o64[0].shape
    for o, x in zip(o64, l64):
        if o.shape != (R, H, dv) or x.shape != (H, R):
            raise ValueError("partials differ in shape")
    optrs = (ctypes.c_void_p * len(o64))(*[o.ctypes.data for o in o64])
    lptrs = (ctypes.c_void_p * len(l64))(*[x.ctypes.data for x in l64])
    out = np.empty((R, H, dv), dtype=np.float64)
    lse = np.empty((H, R), dtype=np.float64)
    rc = _load().oracle_merge(ctypes.cast(optrs, _vp), ctypes.cast(lptrs, _vp), len(o64),
                              R, H, dv, out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return out, lse
