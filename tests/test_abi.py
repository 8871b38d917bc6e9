"""The C ABI library loads without a GPU and exports every declared symbol;
argument errors are reported as statuses before anything touches the GPU."""
import ctypes

import pytest

import ring_attention_slope_gb300 as slope
from _lib import built_lib, declared_symbols

S_OK, E_NULL, E_DTYPE, E_SHAPE, E_STRIDE, E_LAYOUT, E_CUDA, E_TIMEOUT, E_UNSUP, E_WS = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9


@pytest.fixture(scope="module")
def lib():
    return built_lib()


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) == 17, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in slope.h but not exported"
    assert sorted(names) == sorted(slope.EXPORTED)


def test_status_strings_and_version(lib):
    for code in (S_OK, E_NULL, E_DTYPE, E_SHAPE, E_STRIDE, E_LAYOUT, E_CUDA, E_TIMEOUT, E_UNSUP, E_WS):
        assert slope.status_string(code) not in ("", "unknown status")
    assert slope.status_string(12345) == "unknown status"
    assert "sm_103a" in slope.version()


def _t(shape, dtype=0, data=0x10000, stride=None):
    """Descriptor with a fake (never dereferenced) device address."""
    d = slope.SlopeTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    if stride is None:
        stride = []
        acc = 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, s in enumerate(shape):
        d.shape[i] = s
        d.stride[i] = stride[i]
    return d


def _cp(lib, q, k, v, out, lse=None, n=4, layout=1, sizes=None, ws=0x20000, ws_bytes=1 << 40, window=0):
    arr = None
    if sizes is not None:
        arr = (ctypes.c_int64 * len(sizes))(*sizes)
    return lib.slope_cp_prefill(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), n, layout,
                                ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)) if arr else None, 1, window, 0.0,
                                ctypes.byref(out), ctypes.byref(lse) if lse else None, ws, ws_bytes, None)


def test_cp_prefill_argument_errors(lib):
    S, Hq, Hkv, d = 1024, 4, 1, 64
    q, k, v = _t([S, Hq, d]), _t([S, Hkv, d]), _t([S, Hkv, d])
    out, lse = _t([S, Hq, d]), _t([Hq, S], dtype=1)
    assert lib.slope_cp_prefill(None, ctypes.byref(k), ctypes.byref(v), 4, 1, None, 1, 0, 0.0,
                                ctypes.byref(out), None, 0x20000, 1 << 40, None) == E_NULL
    assert _cp(lib, q, k, v, out, lse, ws=0) == E_WS                                  # no workspace
    assert _cp(lib, q, k, v, out, lse, ws_bytes=16) == E_WS                           # too small
    assert _cp(lib, q, k, v, out, lse, ws=0x20010) == E_WS                            # misaligned
    assert _cp(lib, _t([S, Hq, d], dtype=1), k, v, out, lse) == E_DTYPE               # fp32 q
    assert _cp(lib, q, _t([S, 3, d]), _t([S, 3, d]), out, lse) == E_SHAPE            # Hq % Hkv
    assert _cp(lib, q, k, v, out, lse, n=5) == E_LAYOUT                               # 1024 % 10
    assert _cp(lib, q, k, v, out, lse, n=3, layout=0) == E_LAYOUT                     # 1024 % 3
    assert _cp(lib, q, k, v, out, lse, n=2, layout=2, sizes=[500, 500]) == E_LAYOUT   # sizes != S
    assert _cp(lib, q, k, v, out, lse, n=2, layout=2, sizes=[1024, 0]) == E_LAYOUT    # empty chunk
    assert _cp(lib, q, k, v, out, lse, n=4, layout=7) == E_LAYOUT                     # unknown layout
    assert _cp(lib, q, k, v, out, lse, n=0) == E_LAYOUT
    assert _cp(lib, q, k, v, out, lse, n=33) == E_LAYOUT                              # > 32 ranks
    assert _cp(lib, _t([S, Hq, 96]), _t([S, Hkv, 96]), _t([S, Hkv, 96]), _t([S, Hq, 96]), lse) == E_UNSUP
    assert _cp(lib, _t([S, Hq, d], stride=[Hq * d, d, 2]), k, v, out, lse) == E_STRIDE  # inner stride
    assert _cp(lib, _t([S, Hq, d], stride=[Hq * d + 4, d, 1]), k, v, out, lse) == E_STRIDE  # 8-B row stride
    assert _cp(lib, _t([S, Hq, d], data=0x10008), k, v, out, lse) == E_STRIDE      # 8-byte aligned base
    assert _cp(lib, q, k, v, _t([S, Hq, 32]), lse) == E_SHAPE                         # out dv
    assert _cp(lib, q, k, v, out, _t([S, Hq], dtype=1)) == E_SHAPE                    # lse transposed
    assert _cp(lib, q, k, v, out, lse, window=-1) == E_SHAPE
    # Ulysses: whole KV heads per rank (Hkv % n == 0); direct bf16 output needs 8-element strides
    q8, k2, v2, out8 = _t([S, 8, d]), _t([S, 2, d]), _t([S, 2, d]), _t([S, 8, d])
    lse8 = _t([8, S], dtype=1)
    assert _cp(lib, q8, k2, v2, out8, lse8, n=4, layout=3) == E_LAYOUT                # 2 KV heads, 4 ranks
    assert _cp(lib, q8, k2, v2, out8, lse8, n=2, layout=3, ws=0) == E_WS
    assert _cp(lib, q8, k2, v2, _t([S, 8, d], stride=[8 * d + 4, d, 1]), lse8, n=2, layout=3) == E_STRIDE
    assert _cp(lib, q8, k2, v2, out8, lse8, n=33, layout=3) == E_LAYOUT
    # Ulysses x Ring: the degree (bits 8-15 of the layout word) must divide Hkv
    assert _cp(lib, q8, k2, v2, out8, lse8, n=4, layout=1 | (4 << 8)) == E_LAYOUT   # 2 KV heads, 4 groups
    assert _cp(lib, q8, k2, v2, out8, lse8, n=4, layout=3 | (2 << 8)) == E_LAYOUT   # Ulysses takes no degree


def test_attn_partial_and_merge_argument_errors(lib):
    Sq, Skv, Hq, Hkv, d = 300, 200, 8, 2, 128
    q, k, v = _t([Sq, Hq, d]), _t([Skv, Hkv, d]), _t([Skv, Hkv, 64])
    out, lse = _t([Sq, Hq, 64], dtype=1), _t([Hq, Sq], dtype=1)

    def call(q=q, k=k, v=v, out=out, lse=lse):
        return lib.slope_attn_partial(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 0, 0, 1, 0, 0.0,
                                      ctypes.byref(out) if out else None, ctypes.byref(lse) if lse else None, None)

    assert call(out=_t([Sq, Hq, 64], dtype=5)) == E_DTYPE      # unknown dtype
    assert call(out=_t([Sq, Hq, 64], dtype=0, stride=[Hq * 64 + 4, 64, 1])) == E_STRIDE  # bf16 row: 8 elements
    assert call(lse=None) == E_NULL
    assert call(v=_t([Skv, Hkv, 192])) == E_UNSUP              # (128, 192)
    assert call(k=_t([Skv + 1, Hkv, d])) == E_SHAPE
    assert call(out=_t([Sq, Hq, 64], dtype=1, stride=[Hq * 64, 66, 1])) == E_STRIDE
    o = (slope.SlopeTensor * 2)(_t([Sq, Hq, 64], dtype=1), _t([Sq, Hq, 64], dtype=1))
    l = (slope.SlopeTensor * 2)(_t([Hq, Sq], dtype=1), _t([Hq, Sq], dtype=1))
    fin = _t([Sq, Hq, 64], dtype=0)
    assert lib.slope_lse_merge(o, l, 0, ctypes.byref(fin), None, None) == E_SHAPE
    assert lib.slope_lse_merge(o, l, 33, ctypes.byref(fin), None, None) == E_SHAPE
    l_bad = (slope.SlopeTensor * 2)(_t([Hq, Sq], dtype=1), _t([Hq, Sq + 1], dtype=1))
    assert lib.slope_lse_merge(o, l_bad, 2, ctypes.byref(fin), None, None) == E_SHAPE
    o_bad = (slope.SlopeTensor * 2)(_t([Sq, Hq, 64], dtype=1), _t([Sq, Hq, 64], dtype=0))
    assert lib.slope_lse_merge(o_bad, l, 2, ctypes.byref(fin), None, None) == E_DTYPE  # mixed partial dtypes
    o_bad = (slope.SlopeTensor * 2)(_t([Sq, Hq, 64], dtype=0), _t([Sq, Hq, 64], dtype=5))
    assert lib.slope_lse_merge(o_bad, l, 2, ctypes.byref(fin), None, None) == E_DTYPE  # unknown dtype
    o_bad = (slope.SlopeTensor * 2)(_t([Sq, Hq, 64], dtype=0), _t([Sq, Hq, 64], dtype=0, data=0x10004))
    assert lib.slope_lse_merge(o_bad, l, 2, ctypes.byref(fin), None, None) == E_STRIDE  # bf16 partial: 8-B aligned


def test_cp_prefill_ex_flags(lib):
    """flags = 0 is slope_cp_prefill (same checks); unknown bits are refused before any launch;
    bf16 partials need half the plane bytes."""
    S, Hq, Hkv, d = 1024, 4, 1, 64
    q, k, v = _t([S, Hq, d]), _t([S, Hkv, d]), _t([S, Hkv, d])
    out, lse = _t([S, Hq, d]), _t([Hq, S], dtype=1)

    def call(flags, ws_bytes=1 << 40, n=4):
        return lib.slope_cp_prefill_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), n, 1, None, 1, 0, 0.0,
                                       flags, ctypes.byref(out), ctypes.byref(lse), 0x20000, ws_bytes, None)

    assert call(3) == E_UNSUP      # bf16 partials with the fused form, which keeps no partials
    assert call(4) == E_UNSUP
    assert call(1 << 31) == E_UNSUP
    assert call(1, n=5) == E_LAYOUT
    lay = ctypes.c_int(1)
    w0 = lib.slope_cp_prefill_workspace_size(S, Hq, d, 4, lay, None)
    w1 = lib.slope_cp_prefill_workspace_size_ex(S, Hq, d, 4, lay, None, 1)
    assert lib.slope_cp_prefill_workspace_size_ex(S, Hq, d, 4, lay, None, 0) == w0
    assert lib.slope_cp_prefill_workspace_size_ex(S, Hq, d, 4, lay, None, 4) == 0
    # planes: 4 x S x Hq x d x (4 | 2) bytes, then 4 fp32 lse planes (256-B rounded)
    lse_bytes = 4 * S * Hq * 4
    assert w0 == 4 * S * Hq * d * 4 + lse_bytes and w1 == 4 * S * Hq * d * 2 + lse_bytes
    assert call(1, ws_bytes=w1 - 1) == E_WS
    assert call(0, ws_bytes=w1) == E_WS  # fp32 partials need the larger workspace
    # the fused form keeps no partials: an lse plane only (used when lse is NULL)
    w2 = lib.slope_cp_prefill_workspace_size_ex(S, Hq, d, 4, lay, None, 2)
    assert w2 == S * Hq * 4
    assert lib.slope_cp_prefill_workspace_size_ex(S, Hq, d, 4, lay, None, 3) == 0
    assert call(2, ws_bytes=w2 - 1) == E_WS
    assert call(2, n=5) == E_LAYOUT


def test_attn_partial_position_bound(lib):
    """Every query and key position lies in [-2^28, 2^28]; beyond it the call is refused before any launch
    (the kernel takes position differences, less the window, in 32-bit integers)."""
    Sq, Skv, Hq, Hkv, d = 300, 200, 8, 2, 64
    q, k, v = _t([Sq, Hq, d]), _t([Skv, Hkv, d]), _t([Skv, Hkv, d])
    out, lse = _t([Sq, Hq, d], dtype=1), _t([Hq, Sq], dtype=1)

    def call(q_off, kv_off, window=0):
        return lib.slope_attn_partial(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), q_off, kv_off, 1, window,
                                      0.0, ctypes.byref(out), ctypes.byref(lse), None)

    M = 1 << 28
    assert call(1 << 30, -(1 << 30)) == E_SHAPE          # the differences would pass 2^31
    assert call(M - Sq + 1, 0) == E_SHAPE                 # last query position 2^28 + 1 - 1 = 2^28 ... + 1
    assert call(-M - 1, 0) == E_SHAPE
    assert call(0, M - Skv + 1) == E_SHAPE
    assert call(0, -M - 1) == E_SHAPE
    assert call(0, 0, window=(1 << 30) + 1) == E_SHAPE
    assert call(-(1 << 62), 0) == E_SHAPE


def test_empty_inputs_are_no_ops(lib):
    """Zero query rows (attention) or zero rows (merge) return SLOPE_OK before any launch: no GPU is
    touched here, and the descriptors may carry NULL data (strides as torch gives them for empty tensors)."""
    Hq, Hkv, d = 4, 2, 64
    q = _t([0, Hq, d], data=0)
    k, v = _t([128, Hkv, d]), _t([128, Hkv, d])
    out, lse = _t([0, Hq, d], dtype=1, data=0), _t([Hq, 0], dtype=1, data=0, stride=[1, 1])
    assert lib.slope_attn_partial(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 0, 0, 1, 0, 0.0,
                                  ctypes.byref(out), ctypes.byref(lse), None) == S_OK
    o = (slope.SlopeTensor * 2)(_t([0, Hq, d], dtype=1, data=0), _t([0, Hq, d], dtype=0, data=0))
    l = (slope.SlopeTensor * 2)(_t([Hq, 0], dtype=1, data=0, stride=[1, 1]), _t([Hq, 0], dtype=1, data=0, stride=[1, 1]))
    fin = _t([0, Hq, d], dtype=0, data=0)
    assert lib.slope_lse_merge(o, l, 2, ctypes.byref(fin), None, None) == E_DTYPE  # mixed partial dtypes
    o = (slope.SlopeTensor * 2)(_t([0, Hq, d], dtype=0, data=0), _t([0, Hq, d], dtype=0, data=0))
    assert lib.slope_lse_merge(o, l, 2, ctypes.byref(fin), None, None) == S_OK
    assert _cp(lib, _t([0, Hq, d], data=0), _t([0, Hkv, d], data=0), _t([0, Hkv, d], data=0),
               _t([0, Hq, d], data=0), _t([Hq, 0], dtype=1, data=0, stride=[1, 1])) == E_SHAPE  # a prefill needs tokens


def test_workspace_size(lib):
    # ring: N planes of fp32 [S, Hq, dv] + lse; chunked: 2 planes
    ws = slope.cp_prefill_workspace_size(1024, 4, 64, 4, "zigzag")
    assert ws >= 4 * 1024 * 4 * 65 * 4
    wc = slope.cp_prefill_workspace_size(65536, 64, 64, 6, "chunked", [12288] * 5 + [4096])
    assert wc >= 2 * 65536 * 64 * 65 * 4
    assert slope.cp_prefill_workspace_size(1000, 4, 64, 8, "zigzag") == 0
    # Ulysses keeps no partials: only an lse plane (for calls without lse)
    assert slope.cp_prefill_workspace_size(1000, 4, 64, 2, "ulysses") == (1000 * 4 * 4 + 255) // 256 * 256
    assert slope.cp_prefill_workspace_size(1024, 4, 96, 4, "zigzag") == 0


def test_cp_prefill_host_argument_errors(lib):
    """Every argument error of the host-buffer prefill returns before anything is queued (no GPU here)."""
    S, Hq, Hkv, d = 1024, 4, 1, 64
    q, k, v = _t([S, Hq, d]), _t([S, Hkv, d]), _t([S, Hkv, d])
    out, lse = _t([S, Hq, d]), _t([Hq, S], dtype=1)
    hq, hk, hv = _t([S, Hq, d], data=0x90000), _t([S, Hkv, d], data=0x90000), _t([S, Hkv, d], data=0x90000)
    hout, hlse = _t([S, Hq, d], data=0x90000), _t([Hq, S], dtype=1, data=0x90000)

    def call(hq=hq, hk=hk, hv=hv, hout=hout, hlse=hlse, q=q, k=k, v=v, out=out, lse=lse, ws=0x20000,
             ws_bytes=1 << 40, n=4):
        r = lambda t: ctypes.byref(t) if t is not None else None  # noqa: E731
        return lib.slope_cp_prefill_host(r(hq), r(hk), r(hv), r(hout), r(hlse), r(q), r(k), r(v), r(out), r(lse),
                                         n, 1, None, 1, 0, 0.0, ws, ws_bytes, None, None, None)

    assert call(hq=None) == E_NULL
    assert call(hlse=None) == E_NULL                                   # lse given, lse_host not
    assert call(hk=_t([S, Hkv + 1, d], data=0x90000)) == E_SHAPE       # host/device shapes differ
    assert call(hout=_t([S, Hq, d], dtype=1, data=0x90000)) == E_SHAPE  # host/device dtypes differ
    assert call(hv=_t([S, Hkv, d], data=0x90000, stride=[2 * Hkv * d, d, 1])) == E_STRIDE  # not dense
    assert call(q=_t([S, Hq, d], stride=[Hq * d + 8, d, 1]), hq=_t([S, Hq, d], data=0x90000,
                                                                    stride=[Hq * d + 8, d, 1])) == E_STRIDE
    assert call(ws=0) == E_WS                                          # the compute's own checks run first
    assert call(n=5) == E_LAYOUT
