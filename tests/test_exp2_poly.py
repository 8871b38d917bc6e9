"""Host-side checks of the FMA-pipe exp2 used for part of the softmax exponentials.

The kernel's softmax_pair_poly computes 2^x as 2^round(x) * p(x - round(x)) with a
cubic p fitted by ring_attention_slope_gb300/csrc/exp2_poly_fit.py.  These tests
replay that exact float32 / integer sequence in numpy with the coefficients read
from the kernel header and bound its error against exp2 in float64; the GPU
parity tests then check the kernel's attention results against the oracle.
"""
import importlib.util
import pathlib
import re

import numpy as np

CSRC = pathlib.Path(__file__).resolve().parents[1] / "ring_attention_slope_gb300" / "csrc"


def header_consts():
    txt = (CSRC / "sm103_ptx.cuh").read_text()
    out = {}
    for name in ("C0", "C1", "C2", "C3", "Magic"):
        m = re.search(r"constexpr uint32_t kExp2Poly%s = 0x([0-9A-Fa-f]{8})u;" % name, txt)
        assert m, name
        out[name] = np.uint32(int(m.group(1), 16)).view(np.float32)
    return out


def fma32(a, b, c):
    # float32 product is exact in float64; one rounding of the sum to float32 (the
    # double rounding through float64 can differ from a true FMA by one ulp at most)
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def poly_exp2(x):
    """The kernel's sequence: clamp, Cody-Waite reduction, Horner cubic, exponent add."""
    k = header_consts()
    x = np.fmax(x.astype(np.float32), np.float32(-125.0))  # max.f32 returns the non-NaN operand
    magic = np.float32(k["Magic"])
    t = (x + magic).astype(np.float32)
    j = (t - magic).astype(np.float32)
    f = (x - j).astype(np.float32)
    q = fma32(np.full_like(f, k["C3"]), f, np.full_like(f, k["C2"]))
    q = fma32(q, f, np.full_like(f, k["C1"]))
    q = fma32(q, f, np.full_like(f, k["C0"]))
    bits = q.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def test_header_coefficients_come_from_the_fit():
    spec = importlib.util.spec_from_file_location("exp2_poly_fit", CSRC / "exp2_poly_fit.py")
    fitmod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fitmod)
    c = fitmod.fit().astype(np.float32)
    k = header_consts()
    got = np.array([k["C0"], k["C1"], k["C2"], k["C3"]], dtype=np.float32)
    assert got[0] == 1.0
    ulps = np.abs(got.view(np.int32).astype(np.int64) - c.view(np.int32).astype(np.int64))
    assert np.all(ulps <= 2), (got, c)
    assert k["Magic"] == 1.5 * 2**23


def test_relative_error_bound_over_the_softmax_range():
    # x = s * scale * log2(e) - m: at most 8 above the running max (lazy rescale) and
    # unbounded below; the float32 grid covers [-125, 8] densely plus every integer
    x = np.concatenate([np.linspace(-125.0, 8.0, 4_000_001), np.arange(-125, 9)]).astype(np.float32)
    got = poly_exp2(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    assert rel.max() < 1.05e-4, rel.max()
    # a result of this size is far below bf16's 2^-9 relative rounding of P
    assert rel.max() < 2.0**-9 / 16


def test_integers_are_exact_powers_of_two():
    n = np.arange(-125, 9).astype(np.float32)
    np.testing.assert_array_equal(poly_exp2(n), np.exp2(n.astype(np.float64)).astype(np.float32))
    assert poly_exp2(np.array([0.0], np.float32))[0] == 1.0


def test_clamp_below_minus_125_and_masked_scores():
    x = np.array([-125.0, -126.0, -200.0, -1e30, -np.inf, np.nan], dtype=np.float32)
    got = poly_exp2(x).astype(np.float64)
    np.testing.assert_array_equal(got, np.full(6, 2.0**-125))
    assert np.all(np.isfinite(got)) and np.all(got > 0)


def test_half_integer_ties_and_sign():
    # f = +-1/2 at the reduction's rounding ties; both sides of a tie stay accurate
    x = np.array([-0.5, 0.5, -1.5, 1.5, -124.5, 7.5], dtype=np.float32)
    rel = np.abs(poly_exp2(x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.05e-4
    assert np.all(poly_exp2(x) > 0)
